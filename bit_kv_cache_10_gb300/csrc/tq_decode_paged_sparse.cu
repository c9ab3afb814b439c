// Paged-layout (block table) instantiations of the split-K decode kernel with
// sparse V; a translation unit of their own so that the variants compile in
// parallel.
#include "tq_decode_dispatch.cuh"

namespace tq {

tq_status dispatch_split_paged_sparse(const DecodeParams& p, int g, int kb, int vb, cudaStream_t s) {
  return dispatch_split_variant<true, true>(p, g, kb, vb, s);
}

}  // namespace tq
