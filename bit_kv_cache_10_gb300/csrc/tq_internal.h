// Internal declarations shared by the library's translation units (not part of the C ABI).
#pragma once

#include <cstddef>
#include <cstdint>

#include "tq.h"

namespace tq {

constexpr int kHeadDim = 128;     // the kernels are written for d = 128
constexpr int kMinBits = 2;       // GPU path: 2..4 bits per coordinate ([MLX-VLM CLI guide] FAQ
constexpr int kMaxBits = 4;       // "What bit widths does TurboQuant support?")
constexpr int kMaxGroup = 4;      // query heads per KV head handled by the decode kernels
constexpr int kMaxDecodeCtas = 512;   // largest split-K grid (one CTA per SM)
constexpr int kMaxDecodeBatch = 512;  // sequences per decode call (per-sequence tile prefix in shared memory)
// Programmatic dependent launch of the append, split and merge kernels (each
// kernel's parameter-only prologue overlapping the grid before it).  Off: on
// GB300 the decode step (one-token append, split kernel, merge kernel) ran
// 0.1563 ms without it and 0.1688 ms with it on all three launches, the split
// kernel's early launch costing the most.  The kernels keep their
// griddepcontrol instructions, which do nothing in a launch without it.
constexpr int kProgrammaticLaunch = 0;

// Words of one packed token vector.
inline int words_per_token(int head_dim, int bits) { return head_dim * bits / 32; }

// Host validation of a descriptor: shapes, modes and codebooks only, then
// additionally the buffer pointers (non-NULL where the mode needs them, 16-byte aligned).
tq_status validate_shape(const tq_cache_desc* d);
tq_status validate_desc(const tq_cache_desc* d);

// Decode workspace: one partial (G heads x (d accumulators + max + sum)) per
// (split-K CTA, row) pair, at slot CTA + row; rows are the cold and hot rows of
// every (sequence, query token, KV head), so kMaxDecodeCtas + 2 B nq Hkv slots
// always suffice (nq query tokens per sequence; 1 for decode).
size_t decode_workspace_slots(const tq_cache_desc* d, int nq = 1);
size_t decode_workspace_bytes(const tq_cache_desc* d, int nq = 1);

// Bucket scale of the threshold lookup table used by the quantize kernel: the
// smallest power of two A for which every bucket RN(y*A) holds at most one
// float32 threshold.  Returns 0 if none up to 4096.
int quant_lut_scale(const float* thresholds, int n_thresholds);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace tq
