// Cluster-variant instantiations of the tensor-core decode kernel, every mode (small work:
// one thread-block cluster per (b, h) row, the partials merged through
// distributed shared memory, no merge launch), a translation unit of their own
// so that they compile in parallel with the other variants.
#include "tq_decode_dispatch.cuh"

namespace tq {

namespace {

template <int G, int KB>
tq_status cluster_vb(const DecodeParams& p, int vb, cudaStream_t s) {
  switch (vb) {
    case 2: return launch_mma_cluster<G, KB, 2>(p, s);
    case 3: return launch_mma_cluster<G, KB, 3>(p, s);
    default: return launch_mma_cluster<G, KB, 4>(p, s);
  }
}

template <int G>
tq_status cluster_kb(const DecodeParams& p, int kb, int vb, cudaStream_t s) {
  switch (kb) {
    case 2: return cluster_vb<G, 2>(p, vb, s);
    case 3: return cluster_vb<G, 3>(p, vb, s);
    case 4: return cluster_vb<G, 4>(p, vb, s);
    case 8: return launch_mma_cluster<G, 8, 8>(p, s);  // int8 mode
    default: return cluster_vb<G, 16>(p, vb, s);      // fp16 K
  }
}

}  // namespace

tq_status dispatch_cluster(const DecodeParams& p, int g, int kb, int vb, cudaStream_t s) {
  switch (g) {
    case 1: return cluster_kb<1>(p, kb, vb, s);
    case 2: return cluster_kb<2>(p, kb, vb, s);
    default: return cluster_kb<4>(p, kb, vb, s);
  }
}

}  // namespace tq
