// Dequantize kernel: packed token vectors back to float32,
// x_hat = n * D_h * H * c[codes] / sqrt(d) (int8 mode: x_hat = s * code).
//
// One warp per token vector: lane l owns coordinates 4l..4l+3, looks up their
// centroids, runs the two low butterfly stages in registers and the five
// high stages with xor-shuffles, then applies the scale, the signs and the
// norm and writes a float4.  Hot-window V positions and fp16 K rows are
// converted from fp16 instead.
#include <cstring>

#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {
namespace {

constexpr int kQWarps = 8;

struct DequantParams {
  int which;  // 0 = K, 1 = V
  int b, seq_len, token_start, n_tokens;
  int hkv, cap, hot;
  RowMap map;     // cache row of (b, h, t): contiguous or through the block table
  uint32_t* status;
  int bits;       // packed bits, 16 for fp16 K
  const uint32_t* words;
  const float* norms;
  const uint16_t* fp16;  // fp16 K cache or V ring
  uint64_t seed;
  int layer;
  float cent[16];
  float* out;  // [Hkv, n_tokens, D]
};

__global__ void __launch_bounds__(kQWarps * 32) dequantize_kernel(const DequantParams p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kQWarps + warp;
  const int h = blockIdx.y;
  if (t >= p.n_tokens) return;
  const int pos = p.token_start + t;
  float4* dst = reinterpret_cast<float4*>(p.out + (static_cast<int64_t>(h) * p.n_tokens + t) * D) + lane;
  const bool ring = p.which == 1 && p.hot > 0 && pos >= p.seq_len - min(p.hot, p.seq_len);
  const long long row = ring ? 0 : p.map.row(p.b, h, pos);
  if (row < 0) {  // block-table entry outside the pool
    if (lane == 0 && p.status != nullptr) atomicOr(p.status, TQ_DEV_ERR_BLOCK);
    *dst = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    return;
  }
  if (p.bits == 16 || ring) {
    const uint16_t* src = ring ? p.fp16 + ((static_cast<int64_t>(p.b) * p.hkv + h) * p.hot + pos % p.hot) * D
                               : p.fp16 + row * D;
    const uint2 w = reinterpret_cast<const uint2*>(src)[lane];
    const float2 a = half2_bits_to_float2(w.x), c = half2_bits_to_float2(w.y);
    *dst = make_float4(a.x, a.y, c.x, c.y);
    return;
  }
  if (p.bits == 8) {  // int8 mode: s * code, word l holds the codes of coordinates 4l..4l+3
    const uint32_t w = p.words[row * 32 + lane];
    const float s = p.norms[row];
    float res[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) res[k] = fmul(s, static_cast<float>(static_cast<int8_t>((w >> (8 * k)) & 0xFFu)));
    *dst = make_float4(res[0], res[1], res[2], res[3]);
    return;
  }
  // codes of coordinates 4l..4l+3: bits [4*l*bits, 4*l*bits + 4*bits) of the record
  const uint32_t* rec = p.words + row * (p.bits * 4);
  const int bit0 = 4 * lane * p.bits, w0 = bit0 >> 5, off = bit0 & 31;
  uint64_t win = rec[w0];
  if (off + 4 * p.bits > 32) win |= static_cast<uint64_t>(rec[w0 + 1]) << 32;
  win >>= off;
  const uint32_t mask = (1u << p.bits) - 1u;
  float v[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) v[k] = p.cent[(win >> (k * p.bits)) & mask];
  // H over index bits 0,1 (inside the lane) ...
  float a0 = fadd(v[0], v[1]), a1 = fsub(v[0], v[1]), a2 = fadd(v[2], v[3]), a3 = fsub(v[2], v[3]);
  v[0] = fadd(a0, a2);
  v[2] = fsub(a0, a2);
  v[1] = fadd(a1, a3);
  v[3] = fsub(a1, a3);
  // ... and bits 2..6 (across lanes: lane bit k-2)
#pragma unroll
  for (int s = 1; s < 32; s *= 2) {
    const bool upper = (lane & s) != 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float o = __shfl_xor_sync(0xffffffffu, v[k], s);
      v[k] = upper ? fsub(o, v[k]) : fadd(v[k], o);
    }
  }
  const float scale = fmul(p.norms[row], 1.0f / kSqrtD);
  float res[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float x = fmul(v[k], scale);
    res[k] = sign_negative(p.seed, p.layer, h, 4 * lane + k) ? -x : x;
  }
  *dst = make_float4(res[0], res[1], res[2], res[3]);
}

}  // namespace
}  // namespace tq

extern "C" tq_status tq_dequantize(const tq_cache_desc* d, int32_t which, int32_t b, int32_t seq_len,
                                   int32_t token_start, int32_t n_tokens, float* out, tq_stream_t stream) {
  using namespace tq;
  const tq_status vs = validate_desc(d);
  if (vs != TQ_OK) return vs;
  if ((which != 0 && which != 1) || b < 0 || b >= d->batch || token_start < 0 || n_tokens < 0 || out == nullptr ||
      !aligned16(out))
    return TQ_ERR_INVALID_ARG;
  if (static_cast<int64_t>(token_start) + n_tokens > d->capacity) return TQ_ERR_CAPACITY;
  if (which == 1 && d->hot_window > 0 && (seq_len < 0 || seq_len > d->capacity ||
                                          static_cast<int64_t>(token_start) + n_tokens > seq_len))
    return TQ_ERR_INVALID_ARG;
  if (n_tokens == 0) return TQ_OK;
  DequantParams p;
  std::memset(&p, 0, sizeof(p));
  p.which = which;
  p.b = b;
  p.seq_len = seq_len;
  p.token_start = token_start;
  p.n_tokens = n_tokens;
  p.hkv = d->num_kv_heads;
  p.cap = d->capacity;
  p.hot = which == 1 ? d->hot_window : 0;
  p.map = make_row_map(d);
  p.status = d->d_status;
  p.seed = d->seed;
  p.layer = d->layer;
  if (which == 0) {
    p.bits = d->k_mode == TQ_K_FP16 ? 16 : d->k_bits;
    p.words = static_cast<const uint32_t*>(d->k_cache);
    p.norms = d->k_norms;
    p.fp16 = static_cast<const uint16_t*>(d->k_cache);
    if (p.bits != 16 && p.bits != 8) std::memcpy(p.cent, d->k_cb.centroids, sizeof(p.cent));
  } else {
    p.bits = d->v_bits;
    p.words = static_cast<const uint32_t*>(d->v_cache);
    p.norms = d->v_norms;
    p.fp16 = static_cast<const uint16_t*>(d->v_hot);
    if (p.bits != 8) std::memcpy(p.cent, d->v_cb.centroids, sizeof(p.cent));
  }
  p.out = out;
  const dim3 grid((n_tokens + kQWarps - 1) / kQWarps, d->num_kv_heads);
  dequantize_kernel<<<grid, kQWarps * 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(p);
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}
