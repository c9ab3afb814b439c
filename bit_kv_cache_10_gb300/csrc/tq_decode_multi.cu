// Instantiations of the split-K kernel for several query tokens per sequence
// (multi-query attention), contiguous layout, dense V; a translation unit of
// their own so that the variants compile in parallel.
#include "tq_decode_dispatch.cuh"

namespace tq {

tq_status dispatch_split_multi(const DecodeParams& p, int g, int kb, int vb, cudaStream_t s) {
  return dispatch_split_variant<false, false, true>(p, g, kb, vb, s);
}

}  // namespace tq
