// Cluster-variant instantiations of the tensor-core decode kernel (small work:
// one thread-block cluster per (b, h) row, the partials merged through
// distributed shared memory, no merge launch), a translation unit of their own
// so that they compile in parallel with the other variants.
#include "tq_decode_dispatch.cuh"

namespace tq {

tq_status dispatch_cluster(const DecodeParams& p, int g, int kb, cudaStream_t s) {
  switch (g) {
    case 1:
      return kb == 2 ? launch_mma_cluster<1, 2>(p, s) : kb == 3 ? launch_mma_cluster<1, 3>(p, s) : launch_mma_cluster<1, 4>(p, s);
    case 2:
      return kb == 2 ? launch_mma_cluster<2, 2>(p, s) : kb == 3 ? launch_mma_cluster<2, 3>(p, s) : launch_mma_cluster<2, 4>(p, s);
    default:
      return kb == 2 ? launch_mma_cluster<4, 2>(p, s) : kb == 3 ? launch_mma_cluster<4, 3>(p, s) : launch_mma_cluster<4, 4>(p, s);
  }
}

}  // namespace tq
