// Paged-layout (block table) instantiations of the split-K decode kernel,
// dense V; a translation unit of their own so that the variants compile in
// parallel.
#include "tq_decode_dispatch.cuh"

namespace tq {

tq_status dispatch_split_paged(const DecodeParams& p, int g, int kb, int vb, cudaStream_t s) {
  return dispatch_split_variant<false, true>(p, g, kb, vb, s);
}

}  // namespace tq
