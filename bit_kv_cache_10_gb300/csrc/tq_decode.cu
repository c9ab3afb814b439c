// Decode attention over the packed cache: a split-K kernel and a merge kernel.
//
// Split kernel: one CTA per (chunk of context, KV head, sequence); the extra
// last chunk index is the hot fp16-V window when the cache has one.  Four
// warps take 32-token tiles of the chunk round-robin; each tile is staged in
// shared memory with cp.async (double-buffered per warp).  Inside a warp,
// 8 lanes share one token and each owns 16 coordinates; 4 tokens are in
// flight per step and 8 steps cover the tile.
//   score:  lane partial sum_i q'[h][i] c[code_i] over its 16 coordinates for
//           every query head h of the GQA group, with the two codes of a
//           coordinate pair looked up at once in a (c_a, c_b) pair table;
//           a transposing butterfly over the 8 lanes leaves lane l with the
//           full scores of token l;
//   softmax: online, per tile, in base 2 (log2 e is folded into q');
//   V:      acc[h][i] += p_h n_V c[code_i] in the rotated domain, pair table
//           again (cold chunks); the hot window adds raw fp16 V in the
//           original domain.
// All arithmetic is float32 (packed pairs where possible).
//
// Merge kernel: one CTA per (sequence, query head): log-sum-exp combination
// of the chunks, one inverse rotation D_h H / sqrt(d) of the cold sum, the
// hot sum added in the original domain, division by the softmax mass.
#include <cstring>
#include <mutex>

#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {
namespace {

constexpr int kDWarps = 4;
constexpr int kDThreads = kDWarps * 32;  // == D: one thread per coordinate in prologue/epilogue
constexpr int kTile = 32;
constexpr int kCopies = 16;              // pair-table copies (one per lane of a half-warp)

struct DecodeParams {
  const uint16_t* q;
  const int* seq_lens;
  int max_seq_len;
  int batch, hkv, hq, cap, hot;
  int chunk, n_chunks, n_slots;
  const uint32_t* k_words;
  const float* k_norms;
  const uint16_t* k_fp16;
  const uint32_t* v_words;
  const float* v_norms;
  const uint16_t* v_ring;
  uint32_t* status;
  uint64_t seed;
  int layer;
  float k_cent[16];
  float v_cent[16];
  float* ws_acc;  // [B, Hq, slots, D]
  float* ws_ml;   // [B, Hq, slots, 2]
  float* out;     // [B, Hq, D]
};

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem));
}
__device__ __forceinline__ void cp_async4(void* smem, const void* gmem) {
  const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(s), "l"(gmem));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
__device__ __forceinline__ void cp_async_wait1() { asm volatile("cp.async.wait_group 1;\n" ::); }

__device__ __forceinline__ bool seq_len_ok(const DecodeParams& p, int len) {
  return len >= 0 && len <= p.cap && len <= p.max_seq_len;
}
__device__ __forceinline__ int cold_end_of(int len, int hot) { return hot > 0 ? len - min(hot, len) : len; }

template <int KB, int VB>
struct Layout {
  static constexpr bool kFp16K = KB == 16;
  static constexpr int kKRow = kFp16K ? 256 : KB * 16;  // bytes of one K token
  static constexpr int kVRow = VB * 16;
  static constexpr int kKTile = kTile * kKRow;
  static constexpr int kVTile = kTile * kVRow;
  static constexpr int kBuf = kKTile + 128 + kVTile + 128;  // K | K norms | V | V norms
  static constexpr int kKTab = kFp16K ? 0 : (1 << (2 * KB)) * kCopies * 8;
  static constexpr int kVTab = (1 << (2 * VB)) * kCopies * 8;
  static constexpr int kWarpBytes = 2 * kBuf + kTile * 4 * 4;  // two buffers + weights (up to 4 heads)
  static constexpr int kQBytes = 4 * D * 4;
  static constexpr int kSmem = kKTab + kVTab + kDWarps * kWarpBytes + kQBytes;
  static_assert(kDWarps * kWarpBytes >= kDWarps * (4 * D + 8) * 4, "epilogue scratch must fit");
};

// Lane window of 16*BITS code bits starting at bit 16*BITS*r of a token record.
template <int BITS>
__device__ __forceinline__ uint64_t code_window(const uint8_t* rec, int r) {
  if constexpr (BITS == 4) {
    const uint2 w = *reinterpret_cast<const uint2*>(rec + 8 * r);
    return (static_cast<uint64_t>(w.y) << 32) | w.x;
  } else if constexpr (BITS == 2) {
    return *reinterpret_cast<const uint32_t*>(rec + 4 * r);
  } else {
    const uint32_t* wd = reinterpret_cast<const uint32_t*>(rec) + ((3 * r) >> 1);
    const uint64_t v = (static_cast<uint64_t>(wd[1]) << 32) | wd[0];
    return v >> ((r & 1) * 16);
  }
}

// Stage one 32-token tile: K rows, K norms, V rows, V norms.
template <int KB, int VB>
__device__ __forceinline__ void stage_tile(const DecodeParams& p, uint8_t* buf, int64_t row0, int n_valid,
                                           bool hot_slot, int lane) {
  using L = Layout<KB, VB>;
  constexpr int kChunksK = L::kKRow / 16;
  constexpr int kChunksV = L::kVRow / 16;
  const uint8_t* ksrc = L::kFp16K ? reinterpret_cast<const uint8_t*>(p.k_fp16 + row0 * D)
                                  : reinterpret_cast<const uint8_t*>(p.k_words + row0 * (KB * 4));
  for (int c = lane; c < n_valid * kChunksK; c += 32) cp_async16(buf + c * 16, ksrc + c * 16);
  if (!L::kFp16K && lane < n_valid) cp_async4(buf + L::kKTile + lane * 4, p.k_norms + row0 + lane);
  if (!hot_slot) {
    uint8_t* vb = buf + L::kKTile + 128;
    const uint8_t* vsrc = reinterpret_cast<const uint8_t*>(p.v_words + row0 * (VB * 4));
    for (int c = lane; c < n_valid * kChunksV; c += 32) cp_async16(vb + c * 16, vsrc + c * 16);
    if (lane < n_valid) cp_async4(vb + L::kVTile + lane * 4, p.v_norms + row0 + lane);
  }
}

template <int G, int KB, int VB>
__global__ void __launch_bounds__(kDThreads) decode_split_kernel(const DecodeParams p) {
  using L = Layout<KB, VB>;
  extern __shared__ __align__(16) uint8_t smem[];
  float2* ktab = reinterpret_cast<float2*>(smem);
  float2* vtab = reinterpret_cast<float2*>(smem + L::kKTab);
  uint8_t* warp_base = smem + L::kKTab + L::kVTab;
  float* qs = reinterpret_cast<float*>(warp_base + kDWarps * L::kWarpBytes);

  const int slot = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 3, r = lane & 7, copy = lane & (kCopies - 1);
  const bool hot_slot = p.hot > 0 && slot == p.n_chunks;

  int len = p.seq_lens[b];
  if (!seq_len_ok(p, len)) {
    if (tid == 0 && slot == 0 && h == 0 && p.status != nullptr) atomicOr(p.status, TQ_DEV_ERR_SEQ_LEN);
    len = 0;
  }
  const int ce = cold_end_of(len, p.hot);
  int t_begin, t_end;
  if (hot_slot) {
    t_begin = ce;
    t_end = len;
  } else {
    t_begin = slot * p.chunk;
    t_end = min(t_begin + p.chunk, ce);
  }
  const int64_t ws_row0 = (static_cast<int64_t>(b) * p.hq + h * G) * p.n_slots + slot;
  if (t_end <= t_begin) {
    if (tid < G) {
      p.ws_ml[(ws_row0 + static_cast<int64_t>(tid) * p.n_slots) * 2] = -INFINITY;
      p.ws_ml[(ws_row0 + static_cast<int64_t>(tid) * p.n_slots) * 2 + 1] = 0.0f;
    }
    return;
  }

  // ---- pair tables: entry e = code_a | code_b << bits  ->  (c[code_a], c[code_b])
  if constexpr (!L::kFp16K) {
    constexpr int n = (1 << (2 * KB)) * kCopies;
    for (int i = tid; i < n; i += kDThreads) {
      const int e = i / kCopies;
      ktab[i] = make_float2(p.k_cent[e & ((1 << KB) - 1)], p.k_cent[e >> KB]);
    }
  }
  if (!hot_slot) {
    constexpr int n = (1 << (2 * VB)) * kCopies;
    for (int i = tid; i < n; i += kDThreads) {
      const int e = i / kCopies;
      vtab[i] = make_float2(p.v_cent[e & ((1 << VB) - 1)], p.v_cent[e >> VB]);
    }
  }

  // ---- query prologue: q' = (log2 e / d) H D q for packed K, (log2 e / sqrt d) q for fp16 K
#pragma unroll
  for (int j = 0; j < G; ++j) {
    const int hq = h * G + j;
    float x = half_bits_to_float(p.q[(static_cast<int64_t>(b) * p.hq + hq) * D + tid]);
    if (!L::kFp16K && sign_negative(p.seed, p.layer, h, tid)) x = -x;
    qs[j * D + tid] = x;
  }
  __syncthreads();
  if constexpr (!L::kFp16K) {
#pragma unroll
    for (int s = 1; s < D; s *= 2) {
      if ((tid & s) == 0) {
#pragma unroll
        for (int j = 0; j < G; ++j) {
          const float a = qs[j * D + tid], c = qs[j * D + tid + s];
          qs[j * D + tid] = fadd(a, c);
          qs[j * D + tid + s] = fsub(a, c);
        }
      }
      __syncthreads();
    }
  }
  const float qscale = L::kFp16K ? kLog2e / kSqrtD : kLog2e / static_cast<float>(D);
  float2 qr[G][8];
#pragma unroll
  for (int j = 0; j < G; ++j)
#pragma unroll
    for (int k = 0; k < 8; ++k)
      qr[j][k] = make_float2(fmul(qs[j * D + 16 * r + 2 * k], qscale), fmul(qs[j * D + 16 * r + 2 * k + 1], qscale));

  // ---- per-warp streaming over tiles
  uint8_t* wbuf = warp_base + warp * L::kWarpBytes;
  float* wts = reinterpret_cast<float*>(wbuf + 2 * L::kBuf);  // [32][4] softmax weights
  const int64_t kv_row0 = (static_cast<int64_t>(b) * p.hkv + h) * p.cap;
  const int n_tiles = (t_end - t_begin + kTile - 1) / kTile;

  float m[G], lsum[G];
  float2 acc[G][8];
#pragma unroll
  for (int j = 0; j < G; ++j) {
    m[j] = -INFINITY;
    lsum[j] = 0.0f;
#pragma unroll
    for (int k = 0; k < 8; ++k) acc[j][k] = make_float2(0.0f, 0.0f);
  }

  int buf = 0;
  int tile = warp;
  if (tile < n_tiles) {
    const int t0 = t_begin + tile * kTile;
    stage_tile<KB, VB>(p, wbuf, kv_row0 + t0, min(kTile, t_end - t0), hot_slot, lane);
  }
  cp_async_commit();
  __syncthreads();  // tables and q ready
  for (; tile < n_tiles; tile += kDWarps) {
    const int tn = tile + kDWarps;
    if (tn < n_tiles) {
      const int t0n = t_begin + tn * kTile;
      stage_tile<KB, VB>(p, wbuf + (buf ^ 1) * L::kBuf, kv_row0 + t0n, min(kTile, t_end - t0n), hot_slot, lane);
    }
    cp_async_commit();
    cp_async_wait1();
    __syncwarp();

    const uint8_t* tb = wbuf + buf * L::kBuf;
    const int t0 = t_begin + tile * kTile;
    const int n_valid = min(kTile, t_end - t0);

    // scores: P[u][j] = partial over this lane's 16 coordinates of token 8g + u
    float P[8][G];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int tau = 8 * g + u;
      float2 part[G];
#pragma unroll
      for (int j = 0; j < G; ++j) part[j] = make_float2(0.0f, 0.0f);
      if constexpr (L::kFp16K) {
        const uint4* kr = reinterpret_cast<const uint4*>(tb + tau * 256) + 2 * r;
        const uint4 a0 = kr[0], a1 = kr[1];
        const uint32_t wv[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const float2 kf = half2_bits_to_float2(wv[k]);
#pragma unroll
          for (int j = 0; j < G; ++j) part[j] = fma2(qr[j][k], kf, part[j]);
        }
      } else {
        const uint64_t win = code_window<KB>(tb + tau * L::kKRow, r);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t e = static_cast<uint32_t>(win >> (2 * KB * k)) & ((1u << (2 * KB)) - 1u);
          const float2 cp = ktab[e * kCopies + copy];
#pragma unroll
          for (int j = 0; j < G; ++j) part[j] = fma2(qr[j][k], cp, part[j]);
        }
      }
#pragma unroll
      for (int j = 0; j < G; ++j) P[u][j] = fadd(part[j].x, part[j].y);
    }
    // transposing butterfly over the 8 lanes of a group: lane r ends with token 8g + r
    float v4[4][G], v2[2][G], s[G];
    {
      const bool up = (r & 4) != 0;
#pragma unroll
      for (int k = 0; k < 4; ++k)
#pragma unroll
        for (int j = 0; j < G; ++j) {
          const float send = up ? P[k][j] : P[k + 4][j];
          const float keep = up ? P[k + 4][j] : P[k][j];
          v4[k][j] = fadd(keep, __shfl_xor_sync(0xffffffffu, send, 4));
        }
    }
    {
      const bool up = (r & 2) != 0;
#pragma unroll
      for (int k = 0; k < 2; ++k)
#pragma unroll
        for (int j = 0; j < G; ++j) {
          const float send = up ? v4[k][j] : v4[k + 2][j];
          const float keep = up ? v4[k + 2][j] : v4[k][j];
          v2[k][j] = fadd(keep, __shfl_xor_sync(0xffffffffu, send, 2));
        }
    }
    {
      const bool up = (r & 1) != 0;
#pragma unroll
      for (int j = 0; j < G; ++j) {
        const float send = up ? v2[0][j] : v2[1][j];
        const float keep = up ? v2[1][j] : v2[0][j];
        s[j] = fadd(keep, __shfl_xor_sync(0xffffffffu, send, 1));
      }
    }
    // lane l now holds token l of the tile
    const bool valid = lane < n_valid;
    const float nk = L::kFp16K ? 1.0f : reinterpret_cast<const float*>(tb + L::kKTile)[lane];
    const float nv = hot_slot ? 1.0f : reinterpret_cast<const float*>(tb + L::kKTile + 128 + L::kVTile)[lane];
    float alpha[G];
    bool rescale = false;
#pragma unroll
    for (int j = 0; j < G; ++j) {
      const float sj = valid ? fmul(s[j], nk) : -INFINITY;
      float tmax = sj;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
      const float mn = fmaxf(m[j], tmax);
      alpha[j] = exp2f(m[j] - mn);
      rescale |= alpha[j] != 1.0f;
      const float pj = valid ? exp2f(sj - mn) : 0.0f;
      lsum[j] = ffma(lsum[j], alpha[j], pj);
      m[j] = mn;
      wts[lane * 4 + j] = valid ? fmul(pj, nv) : 0.0f;  // staged norms of masked rows are garbage
    }
    if (rescale) {
#pragma unroll
      for (int j = 0; j < G; ++j)
#pragma unroll
        for (int k = 0; k < 8; ++k) acc[j][k] = mul2(acc[j][k], make_float2(alpha[j], alpha[j]));
    }
    __syncwarp();

    // V accumulation for tokens 8g + u
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int tau = 8 * g + u;
      float2 w2[G];
#pragma unroll
      for (int j = 0; j < G; ++j) {
        const float wj = wts[tau * 4 + j];
        w2[j] = make_float2(wj, wj);
      }
      if (!hot_slot) {
        const uint64_t win = code_window<VB>(tb + L::kKTile + 128 + tau * L::kVRow, r);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t e = static_cast<uint32_t>(win >> (2 * VB * k)) & ((1u << (2 * VB)) - 1u);
          const float2 cp = vtab[e * kCopies + copy];
#pragma unroll
          for (int j = 0; j < G; ++j) acc[j][k] = fma2(w2[j], cp, acc[j][k]);
        }
      } else if (tau < n_valid) {
        const int pos = t0 + tau;
        const uint4* vr = reinterpret_cast<const uint4*>(
                              p.v_ring + ((static_cast<int64_t>(b) * p.hkv + h) * p.hot + pos % p.hot) * D) +
                          2 * r;
        const uint4 a0 = vr[0], a1 = vr[1];
        const uint32_t wv[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const float2 vf = half2_bits_to_float2(wv[k]);
#pragma unroll
          for (int j = 0; j < G; ++j) acc[j][k] = fma2(w2[j], vf, acc[j][k]);
        }
      }
    }
    __syncwarp();
    buf ^= 1;
  }
  asm volatile("cp.async.wait_all;\n" ::);

  // ---- combine the 4 token groups of the warp, then the warps of the CTA
#pragma unroll
  for (int j = 0; j < G; ++j) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      acc[j][k].x = fadd(acc[j][k].x, __shfl_xor_sync(0xffffffffu, acc[j][k].x, 8));
      acc[j][k].y = fadd(acc[j][k].y, __shfl_xor_sync(0xffffffffu, acc[j][k].y, 8));
      acc[j][k].x = fadd(acc[j][k].x, __shfl_xor_sync(0xffffffffu, acc[j][k].x, 16));
      acc[j][k].y = fadd(acc[j][k].y, __shfl_xor_sync(0xffffffffu, acc[j][k].y, 16));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lsum[j] = fadd(lsum[j], __shfl_xor_sync(0xffffffffu, lsum[j], o));
  }
  __syncthreads();  // staging buffers are free now
  float* red = reinterpret_cast<float*>(warp_base);  // [warp][G][D] acc, then [warp][G][2] (m, l)
  float* red_ml = red + kDWarps * G * D;
  if (g == 0) {
#pragma unroll
    for (int j = 0; j < G; ++j)
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        red[(warp * G + j) * D + 16 * r + 2 * k] = acc[j][k].x;
        red[(warp * G + j) * D + 16 * r + 2 * k + 1] = acc[j][k].y;
      }
  }
  if (lane == 0) {
#pragma unroll
    for (int j = 0; j < G; ++j) {
      red_ml[(warp * G + j) * 2] = m[j];
      red_ml[(warp * G + j) * 2 + 1] = lsum[j];
    }
  }
  __syncthreads();
#pragma unroll
  for (int j = 0; j < G; ++j) {
    float mm = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDWarps; ++w) mm = fmaxf(mm, red_ml[(w * G + j) * 2]);
    float a = 0.0f, l = 0.0f;
#pragma unroll
    for (int w = 0; w < kDWarps; ++w) {
      const float mw = red_ml[(w * G + j) * 2];
      if (mw == -INFINITY) continue;
      const float sc = exp2f(mw - mm);
      a = ffma(red[(w * G + j) * D + tid], sc, a);
      l = ffma(red_ml[(w * G + j) * 2 + 1], sc, l);
    }
    const int64_t row = ws_row0 + static_cast<int64_t>(j) * p.n_slots;
    p.ws_acc[row * D + tid] = a;
    if (tid == 0) {
      p.ws_ml[row * 2] = mm;
      p.ws_ml[row * 2 + 1] = l;
    }
  }
}

__global__ void __launch_bounds__(D) decode_merge_kernel(const DecodeParams p) {
  __shared__ float y[D];
  const int hq = blockIdx.x, b = blockIdx.y, t = threadIdx.x;
  const int g = p.hq / p.hkv, h = hq / g;
  float* out = p.out + (static_cast<int64_t>(b) * p.hq + hq) * D;
  const int len = p.seq_lens[b];
  if (!seq_len_ok(p, len) || len == 0) {
    out[t] = 0.0f;
    return;
  }
  const int64_t row0 = (static_cast<int64_t>(b) * p.hq + hq) * p.n_slots;
  float mm = -INFINITY;
  for (int s = 0; s < p.n_slots; ++s) mm = fmaxf(mm, p.ws_ml[(row0 + s) * 2]);
  float cold = 0.0f, hot = 0.0f, l = 0.0f;
  for (int s = 0; s < p.n_slots; ++s) {
    const float ms = p.ws_ml[(row0 + s) * 2];
    if (ms == -INFINITY) continue;
    const float sc = exp2f(ms - mm);
    l = ffma(p.ws_ml[(row0 + s) * 2 + 1], sc, l);
    const float a = p.ws_acc[(row0 + s) * D + t];
    if (p.hot > 0 && s == p.n_chunks) hot = fmul(a, sc);
    else cold = ffma(a, sc, cold);
  }
  // inverse rotation of the cold sum: D_h H y / sqrt(d)
  y[t] = cold;
  __syncthreads();
#pragma unroll
  for (int s = 1; s < D; s *= 2) {
    float v = 0.0f;
    if ((t & s) == 0) v = fadd(y[t], y[t + s]);
    else v = fsub(y[t - s], y[t]);
    __syncthreads();
    y[t] = v;
    __syncthreads();
  }
  float v = fmul(y[t], 1.0f / kSqrtD);
  if (sign_negative(p.seed, p.layer, h, t)) v = -v;
  out[t] = fadd(v, hot) / l;
}

template <int G, int KB, int VB>
tq_status launch_split(const DecodeParams& p, cudaStream_t stream) {
  using L = Layout<KB, VB>;
  auto kern = decode_split_kernel<G, KB, VB>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmem) != cudaSuccess)
    return TQ_ERR_CUDA;
  const dim3 grid(p.n_slots, p.hkv, p.batch);
  kern<<<grid, kDThreads, L::kSmem, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

template <int G, int KB>
tq_status dispatch_vb(const DecodeParams& p, int vb, cudaStream_t s) {
  switch (vb) {
    case 2: return launch_split<G, KB, 2>(p, s);
    case 3: return launch_split<G, KB, 3>(p, s);
    default: return launch_split<G, KB, 4>(p, s);
  }
}

template <int G>
tq_status dispatch_kb(const DecodeParams& p, int kb, int vb, cudaStream_t s) {
  switch (kb) {
    case 2: return dispatch_vb<G, 2>(p, vb, s);
    case 3: return dispatch_vb<G, 3>(p, vb, s);
    case 4: return dispatch_vb<G, 4>(p, vb, s);
    default: return dispatch_vb<G, 16>(p, vb, s);
  }
}

}  // namespace
}  // namespace tq

extern "C" size_t tq_decode_workspace_bytes(const tq_cache_desc* d, int32_t max_seq_len) {
  using namespace tq;
  if (validate_shape(d) != TQ_OK || max_seq_len < 0) return 0;
  const int len = max_seq_len < d->capacity ? max_seq_len : d->capacity;
  const size_t slots = static_cast<size_t>(decode_num_slots(d, len));
  return static_cast<size_t>(d->batch) * d->num_q_heads * slots * (D + 2) * sizeof(float);
}

extern "C" tq_status tq_decode_attention(const tq_cache_desc* d, const void* q, const int32_t* d_seq_lens,
                                         int32_t max_seq_len, float* out, void* workspace, size_t workspace_bytes,
                                         tq_stream_t stream) {
  using namespace tq;
  const tq_status vs = validate_desc(d);
  if (vs != TQ_OK) return vs;
  if (q == nullptr || d_seq_lens == nullptr || out == nullptr || max_seq_len < 0) return TQ_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(out)) return TQ_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t out_bytes = static_cast<size_t>(d->batch) * d->num_q_heads * D * sizeof(float);
  const int len = max_seq_len < d->capacity ? max_seq_len : d->capacity;
  const int slots = decode_num_slots(d, len);
  if (slots == 0) return cudaMemsetAsync(out, 0, out_bytes, s) == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
  const size_t need = tq_decode_workspace_bytes(d, max_seq_len);
  if (workspace == nullptr || !aligned16(workspace) || workspace_bytes < need) return TQ_ERR_WORKSPACE;

  DecodeParams p;
  std::memset(&p, 0, sizeof(p));
  p.q = static_cast<const uint16_t*>(q);
  p.seq_lens = d_seq_lens;
  p.max_seq_len = max_seq_len;
  p.batch = d->batch;
  p.hkv = d->num_kv_heads;
  p.hq = d->num_q_heads;
  p.cap = d->capacity;
  p.hot = d->hot_window;
  p.chunk = kDecodeChunk;
  p.n_chunks = decode_num_chunks(d, len);
  p.n_slots = slots;
  p.k_words = static_cast<const uint32_t*>(d->k_cache);
  p.k_norms = d->k_norms;
  p.k_fp16 = static_cast<const uint16_t*>(d->k_cache);
  p.v_words = static_cast<const uint32_t*>(d->v_cache);
  p.v_norms = d->v_norms;
  p.v_ring = static_cast<const uint16_t*>(d->v_hot);
  p.status = d->d_status;
  p.seed = d->seed;
  p.layer = d->layer;
  if (d->k_mode == TQ_K_PACKED) std::memcpy(p.k_cent, d->k_cb.centroids, sizeof(p.k_cent));
  std::memcpy(p.v_cent, d->v_cb.centroids, sizeof(p.v_cent));
  p.ws_acc = static_cast<float*>(workspace);
  p.ws_ml = p.ws_acc + static_cast<size_t>(d->batch) * d->num_q_heads * slots * D;
  p.out = out;

  const int g = d->num_q_heads / d->num_kv_heads;
  const int kb = d->k_mode == TQ_K_FP16 ? 16 : d->k_bits;
  tq_status st;
  switch (g) {
    case 1: st = dispatch_kb<1>(p, kb, d->v_bits, s); break;
    case 2: st = dispatch_kb<2>(p, kb, d->v_bits, s); break;
    default: st = dispatch_kb<4>(p, kb, d->v_bits, s); break;
  }
  if (st != TQ_OK) return st;
  decode_merge_kernel<<<dim3(d->num_q_heads, d->batch), D, 0, s>>>(p);
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// Decode without a caller workspace: the split-K partials live in a fixed
// device array of this file, for callers that cannot allocate device memory.
// ---------------------------------------------------------------------------
namespace {

static __device__ __align__(256) unsigned char g_no_alloc_scratch[TQ_NO_ALLOC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_address[kMaxDevices] = {};

// Device address of the scratch array on the current device.  In host code the
// array's name only stands in for the symbol, so the address is looked up once
// per device with that device current.
tq_status no_alloc_scratch(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return TQ_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return TQ_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_address[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_no_alloc_scratch) != cudaSuccess || p == nullptr) return TQ_ERR_CUDA;
    g_scratch_address[dev] = p;
  }
  *out = g_scratch_address[dev];
  return TQ_OK;
}

}  // namespace

extern "C" tq_status tq_decode_attention_no_alloc(const tq_cache_desc* d, const void* q, const int32_t* d_seq_lens,
                                                  int32_t max_seq_len, float* out, tq_stream_t stream) {
  const tq_status vs = tq::validate_desc(d);
  if (vs != TQ_OK) return vs;
  if (max_seq_len < 0) return TQ_ERR_INVALID_ARG;
  if (tq_decode_workspace_bytes(d, max_seq_len) > TQ_NO_ALLOC_WORKSPACE_BYTES) return TQ_ERR_WORKSPACE;
  void* scratch = nullptr;
  const tq_status st = no_alloc_scratch(&scratch);
  if (st != TQ_OK) return st;
  return tq_decode_attention(d, q, d_seq_lens, max_seq_len, out, scratch, TQ_NO_ALLOC_WORKSPACE_BYTES, stream);
}
