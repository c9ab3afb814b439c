// Instantiations of the split-K kernel for several query tokens per sequence
// (multi-query attention), paged layout, dense V.
#include "tq_decode_dispatch.cuh"

namespace tq {

tq_status dispatch_split_multi_paged(const DecodeParams& p, int g, int kb, int vb, cudaStream_t s) {
  return dispatch_split_variant<false, true, true>(p, g, kb, vb, s);
}

}  // namespace tq
