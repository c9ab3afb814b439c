// Launch selection of the split-K decode kernels, included by the decode
// translation units (each instantiates one variant: dense or sparse V,
// contiguous or paged layout, one or several query tokens per sequence).
//
// Every mode runs the tensor-core kernel (tq_decode_mma.cuh): packed K of 2..4
// bits or fp16 K with packed V of 2..4 bits, and the int8 mode.  The tile list,
// staging and merge helpers it uses are in tq_decode_split.cuh.
#pragma once

#include "tq_decode_mma.cuh"
#include "tq_decode_split.cuh"

namespace tq {
namespace {

template <int G, int KB, bool SPARSE, bool PAGED, bool MQ>
tq_status dispatch_vb(const DecodeParams& p, int vb, cudaStream_t s) {
  switch (vb) {
    case 2: return launch_mma<G, KB, SPARSE, PAGED, MQ, 2>(p, s);
    case 3: return launch_mma<G, KB, SPARSE, PAGED, MQ, 3>(p, s);
    default: return launch_mma<G, KB, SPARSE, PAGED, MQ, 4>(p, s);
  }
}

template <int G, bool SPARSE, bool PAGED, bool MQ>
tq_status dispatch_kb(const DecodeParams& p, int kb, int vb, cudaStream_t s) {
  switch (kb) {
    case 8: return launch_mma<G, 8, SPARSE, PAGED, MQ>(p, s);  // int8 mode
    case 2: return dispatch_vb<G, 2, SPARSE, PAGED, MQ>(p, vb, s);
    case 3: return dispatch_vb<G, 3, SPARSE, PAGED, MQ>(p, vb, s);
    case 4: return dispatch_vb<G, 4, SPARSE, PAGED, MQ>(p, vb, s);
    default: return dispatch_vb<G, 16, SPARSE, PAGED, MQ>(p, vb, s);
  }
}

// Split kernels of one variant (dense or sparse V, contiguous or paged, one or
// several query tokens per sequence) for any group size and widths.
template <bool SPARSE, bool PAGED, bool MQ = false>
tq_status dispatch_split_variant(const DecodeParams& p, int g, int kb, int vb, cudaStream_t s) {
  switch (g) {
    case 1: return dispatch_kb<1, SPARSE, PAGED, MQ>(p, kb, vb, s);
    case 2: return dispatch_kb<2, SPARSE, PAGED, MQ>(p, kb, vb, s);
    default: return dispatch_kb<4, SPARSE, PAGED, MQ>(p, kb, vb, s);
  }
}

}  // namespace

// Split-K launches of the other variants, each in a translation unit of its own
// (the dense contiguous one is in tq_decode.cu).
tq_status dispatch_split_sparse(const DecodeParams& p, int g, int kb, int vb, cudaStream_t s);
tq_status dispatch_split_paged(const DecodeParams& p, int g, int kb, int vb, cudaStream_t s);
tq_status dispatch_split_paged_sparse(const DecodeParams& p, int g, int kb, int vb, cudaStream_t s);
tq_status dispatch_split_multi(const DecodeParams& p, int g, int kb, int vb, cudaStream_t s);
tq_status dispatch_split_multi_paged(const DecodeParams& p, int g, int kb, int vb, cudaStream_t s);
// Cluster variant (any K and V width, dense V, contiguous layout, one query
// token): TQ_ERR_UNSUPPORTED without a launch when the rows do not fit in one
// wave of clusters.
tq_status dispatch_cluster(const DecodeParams& p, int g, int kb, int vb, cudaStream_t s);

}  // namespace tq
