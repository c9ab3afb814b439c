/*
 * tq_debug.h -- verification hooks of the TurboQuant library.
 *
 * These entry points run the host build of the kernels' per-vector
 * arithmetic (the same source file, compiled for the CPU with IEEE float32
 * round-to-nearest and no contraction), so that the exact-norm rounding, the
 * rotation and the bucketed threshold lookup can be checked on a machine
 * without a GPU.  No product entry point of tq.h calls them, and they are
 * not a fallback: they only exist to test the device code path.
 */
#ifndef TQ_DEBUG_H_
#define TQ_DEBUG_H_

#include "tq.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Quantize n_rows fp16 vectors of length 128 (host memory, `rows` holds the
 * raw fp16 bit patterns, row-major) with the codebook `cb` (head_dim 128,
 * bits 2..4) and the rotation signs of (seed, layer, head).  Writes
 * n_rows * bits * 4 packed words and n_rows norms (host memory).
 */
tq_status tq_debug_quantize_rows_host(const tq_codebook *cb, uint64_t seed, int32_t layer, int32_t head,
                                      const uint16_t *rows, int32_t n_rows, uint32_t *words, float *norms);

/*
 * Decode path for tests of tq_decode_attention (process-wide, not thread
 * safe against concurrent calls): 0 selects automatically (the default), 1
 * always runs the persistent split-K kernel followed by the merge kernel, 2
 * runs the cluster variant (one thread-block cluster per (sequence, KV head)
 * row, merged in distributed shared memory) wherever the mode allows it:
 * packed K of 2..4 bits with 4-bit V, dense V, contiguous layout, and every
 * row's cluster resident on the GPU at once.  Any other value means 0.
 */
void tq_debug_set_decode_path(int32_t path);

/*
 * Split plan of the persistent decode path, computed on the host by the same
 * functions the kernels use (tq_split_plan.h): the work list has nv sequences
 * of hkv rows each, a row of sequence v being tiles_cold[v] cold 16-token tiles
 * followed by tiles_hot[v] hot ones (host arrays, each entry >= 0), and a
 * CTA's share is counted in tiles plus price_cold (price_hot) tiles for every
 * cold (hot) segment it starts, a segment being the cold or the hot tiles of
 * one row.  Writes
 * starts[0 .. grid] (host, grid + 1 entries): CTA c of the split kernel takes
 * the tiles [starts[c], starts[c + 1]) of the list.  If seg_ctas is not null
 * it receives 2 nv hkv rows of grid bytes (host): byte (2 r + part) grid + c is
 * 1 when the merge kernel reads CTA c's partial for part 0 (cold) or 1 (hot)
 * of row r, else 0.  TQ_ERR_INVALID_ARG for null arrays, nv < 1, hkv < 1,
 * grid < 1, a negative count or price, or a list of 2^40 tiles or more.
 */
tq_status tq_debug_split_plan(const int32_t *tiles_cold, const int32_t *tiles_hot, int32_t nv, int32_t hkv,
                              int32_t grid, int32_t price_cold, int32_t price_hot, int64_t *starts,
                              uint8_t *seg_ctas);

#ifdef __cplusplus
}
#endif

#endif /* TQ_DEBUG_H_ */
