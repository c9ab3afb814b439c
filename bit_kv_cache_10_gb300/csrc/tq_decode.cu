// Decode attention over the packed cache: a persistent split-K kernel and a
// merge kernel.
//
// Work list.  Every (sequence b, KV head h) has a cold row (the packed
// positions [0, L - min(W, L))) and, with a hot window, a hot row (the newest
// min(W, L) positions, whose V is read from the fp16 ring).  Rows are cut into
// 32-token tiles and listed in (b, h, cold/hot) order; the list is split into
// one contiguous, equal range per CTA, so that every SM gets the same number
// of tiles whatever the lengths are.
//
// Split kernel: one CTA of 8 warps per SM.  The codebook pair tables are built
// once per CTA in shared memory (16 copies, one per lane of a half-warp, so the
// data-dependent lookups are bank-conflict free).  Warp w takes tiles
// t0 + w, t0 + w + 8, ... of the CTA's range and streams them through a 3-4
// stage cp.async ring that runs across row boundaries.  Inside a warp 8 lanes
// share a token and each owns 16 coordinates; 4 tokens are in flight per step
// and 8 steps cover the tile:
//   score:   partial sum_i q'[h][i] c[code_i] over the lane's 16 coordinates
//            for the G query heads of the group, with the two codes of a
//            coordinate pair looked up at once in a (c_a, c_b) table; a
//            transposing butterfly over the 8 lanes leaves lane l with the
//            full scores of token l;
//   softmax: online, per 8-token group, in base 2 (log2 e is folded into q');
//   V:       acc[h][i] += p_h n_V c[code_i] in the rotated domain (cold rows)
//            or += p_h v_i with the raw fp16 V (hot rows, original domain).
// When the CTA leaves a row it combines its 8 warps and writes one partial
// (acc, max, sum) to workspace slot (CTA index + row index): these slots are
// distinct for all (CTA, row) pairs because both indices only grow along the
// tile list.  All arithmetic is float32 (packed pairs where possible).
//
// Merge kernel: one CTA per (sequence, query head): finds the CTAs that
// covered its cold and hot rows, log-sum-exp combines their partials, rotates
// the cold sum back once (D_h H / sqrt(d)), adds the hot sum and divides by
// the softmax mass.
#include <cstring>
#include <mutex>

#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kTile = 32;
constexpr int kCopies = 16;                 // pair-table copies (one per lane of a half-warp)
constexpr int kSmemBudget = 227 * 1024;

struct DecodeParams {
  const uint16_t* q;
  const int* seq_lens;
  int max_seq_len;
  int batch, hkv, hq, cap, hot;
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
  float* ws_acc;  // [slots][G][D]
  float* ws_ml;   // [slots][G][2] (max, sum)
  int grid;       // CTAs of the split kernel
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
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

// Length of sequence b, or 0 when it is outside [0, min(cap, max_seq_len)].
__device__ __forceinline__ int seq_len(const DecodeParams& p, int b) {
  const int len = p.seq_lens[b];
  return (len >= 0 && len <= p.cap && len <= p.max_seq_len) ? len : 0;
}

struct SeqTiles {
  int len, ce, tc, th;  // length, cold end, cold tiles, hot tiles
};
__device__ __forceinline__ SeqTiles seq_tiles(const DecodeParams& p, int b) {
  SeqTiles s;
  s.len = seq_len(p, b);
  s.ce = p.hot > 0 ? s.len - min(p.hot, s.len) : s.len;
  s.tc = (s.ce + kTile - 1) / kTile;
  s.th = (s.len - s.ce + kTile - 1) / kTile;
  return s;
}

// Exclusive prefix (over sequences) of the tile counts, prefix[0..B], in
// shared memory; all threads of the block must call it.  Uses `scratch`
// (at least 33 long longs).
template <int NT>
__device__ void tile_prefix(const DecodeParams& p, long long* prefix, long long* scratch) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int kPer = (kMaxDecodeBatch + NT - 1) / NT;
  long long v[kPer];
  long long mine = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int b = tid * kPer + i;
    long long c = 0;
    if (b < p.batch) {
      const SeqTiles s = seq_tiles(p, b);
      c = static_cast<long long>(p.hkv) * (s.tc + s.th);
    }
    v[i] = c;
    mine += c;
  }
  long long incl = mine;  // inclusive scan over the warp
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) scratch[warp] = incl;
  __syncthreads();
  if (tid == 0) {
    long long run = 0;
    for (int w = 0; w < NT / 32; ++w) {
      const long long t = scratch[w];
      scratch[w] = run;
      run += t;
    }
    scratch[32] = run;
  }
  __syncthreads();
  long long base = scratch[warp] + incl - mine;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int b = tid * kPer + i;
    if (b < p.batch) prefix[b] = base;
    base += v[i];
  }
  if (tid == 0) prefix[p.batch] = scratch[32];
  __syncthreads();
}

struct TileInfo {
  int b, h, hot;          // sequence, KV head, 1 for the hot row
  int t_begin, n_valid;   // first position of the tile, valid tokens
  int row;                // (b * Hkv + h) * 2 + hot
  long long row_start, row_end;  // tile-list range of the row
};

__device__ __forceinline__ TileInfo tile_info(const DecodeParams& p, const long long* prefix, long long t) {
  int lo = 0, hi = p.batch;  // largest b with prefix[b] <= t
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] <= t) lo = mid;
    else hi = mid;
  }
  TileInfo ti;
  ti.b = lo;
  const SeqTiles s = seq_tiles(p, lo);
  const int per_h = s.tc + s.th;
  const int rem = static_cast<int>(t - prefix[lo]);  // < Hkv * per_h < 2^31 (checked on the host)
  ti.h = rem / per_h;
  const int x = rem - ti.h * per_h;
  const long long hbase = prefix[lo] + static_cast<long long>(ti.h) * per_h;
  if (x < s.tc) {
    ti.hot = 0;
    ti.t_begin = x * kTile;
    ti.n_valid = min(kTile, s.ce - ti.t_begin);
    ti.row_start = hbase;
    ti.row_end = hbase + s.tc;
  } else {
    ti.hot = 1;
    ti.t_begin = s.ce + (x - s.tc) * kTile;
    ti.n_valid = min(kTile, s.len - ti.t_begin);
    ti.row_start = hbase + s.tc;
    ti.row_end = hbase + per_h;
  }
  ti.row = (lo * p.hkv + ti.h) * 2 + ti.hot;
  return ti;
}

template <int KB, int VB>
struct Cfg {
  static constexpr bool kFp16K = KB == 16;
  static constexpr int kKRow = kFp16K ? 256 : KB * 16;  // bytes of one K token
  static constexpr int kVRow = VB * 16;
  static constexpr int kKTile = kTile * kKRow;
  static constexpr int kKNorm = kFp16K ? 0 : 128;
  static constexpr int kVTile = kTile * kVRow;
  static constexpr int kBuf = kKTile + kKNorm + kVTile + 128;  // K | K norms | V | V norms
  static constexpr int kKTab = kFp16K ? 0 : (1 << (2 * (kFp16K ? 1 : KB))) * kCopies * 8;
  static constexpr int kVTab = (1 << (2 * VB)) * kCopies * 8;
  static constexpr int kWts = 36 * 32;  // per warp: (w, w) x 4 heads per token, one pad row per 8 tokens
  static constexpr int kFixed = kKTab + kVTab + kWarps * kWts + 4 * D * 4 /* q' */ + 4 * D * 4 /* combine */ +
                                kWarps * 4 * 2 * 4 /* warp (m, l) */ + kWarps * 4 * 16 /* tile descriptors */ +
                                (kMaxDecodeBatch + 1) * 8 + 34 * 8;
  static constexpr int kStages = kFixed + kWarps * 4 * kBuf <= kSmemBudget   ? 4
                                 : kFixed + kWarps * 3 * kBuf <= kSmemBudget ? 3
                                                                             : 2;
  static constexpr int kSmem = kFixed + kWarps * kStages * kBuf;
  static_assert(kSmem <= kSmemBudget, "shared memory budget");
};

// Lane window of 16*BITS code bits starting at bit 16*BITS*r of a token
// record, as two 32-bit words (bits 0..31 and 32..63 of the window).
struct Win {
  uint32_t lo, hi;
};
template <int BITS>
__device__ __forceinline__ Win code_window(const uint8_t* rec, int r) {
  if constexpr (BITS == 4) {
    const uint2 w = *reinterpret_cast<const uint2*>(rec + 8 * r);
    return Win{w.x, w.y};
  } else if constexpr (BITS == 2) {
    return Win{*reinterpret_cast<const uint32_t*>(rec + 4 * r), 0u};
  } else {
    const uint32_t* wd = reinterpret_cast<const uint32_t*>(rec) + ((3 * r) >> 1);
    const uint32_t w0 = wd[0], w1 = wd[1];
    const uint32_t sh = (r & 1) * 16;
    return Win{__funnelshift_r(w0, w1, sh), w1 >> sh};
  }
}

// Byte offset, inside a pair table, of the entry of code pair K of a window
// (entry = two codes; 16 copies x 8 bytes per entry; this lane's copy): the
// field is shifted to bit 7 with one 32-bit (funnel) shift, then masked.
template <int BITS, int K>
__device__ __forceinline__ uint32_t pair_offset(const Win& w, uint32_t copy8) {
  constexpr int kP = 2 * BITS * K;   // first bit of the field in the window
  constexpr int kW = 2 * BITS;       // field width
  uint32_t v;
  if constexpr (kP + kW <= 32) {
    v = kP >= 7 ? (w.lo >> (kP >= 7 ? kP - 7 : 0)) : (w.lo << (kP < 7 ? 7 - kP : 0));
  } else if constexpr (kP >= 32) {
    v = kP - 32 >= 7 ? (w.hi >> (kP - 32 >= 7 ? kP - 39 : 0)) : (w.hi << (kP - 32 < 7 ? 39 - kP : 0));
  } else {
    v = __funnelshift_r(w.lo, w.hi, kP - 7);
  }
  return (v & (((1u << kW) - 1u) << 7)) | copy8;
}

template <int KB, int VB>
__device__ __forceinline__ void stage_tile(const DecodeParams& p, const TileInfo& ti, uint8_t* buf, int lane) {
  using C = Cfg<KB, VB>;
  const int64_t row0 = (static_cast<int64_t>(ti.b) * p.hkv + ti.h) * p.cap + ti.t_begin;
  constexpr int kChunksK = C::kKRow / 16;
  const uint8_t* ksrc = C::kFp16K ? reinterpret_cast<const uint8_t*>(p.k_fp16 + row0 * D)
                                  : reinterpret_cast<const uint8_t*>(p.k_words + row0 * (C::kFp16K ? 0 : KB * 4));
  for (int c = lane; c < ti.n_valid * kChunksK; c += 32) cp_async16(buf + c * 16, ksrc + c * 16);
  if (!C::kFp16K && lane < ti.n_valid) cp_async4(buf + C::kKTile + lane * 4, p.k_norms + row0 + lane);
  if (!ti.hot) {
    constexpr int kChunksV = C::kVRow / 16;
    uint8_t* vb = buf + C::kKTile + C::kKNorm;
    const uint8_t* vsrc = reinterpret_cast<const uint8_t*>(p.v_words + row0 * (VB * 4));
    for (int c = lane; c < ti.n_valid * kChunksV; c += 32) cp_async16(vb + c * 16, vsrc + c * 16);
    if (lane < ti.n_valid) cp_async4(vb + C::kVTile + lane * 4, p.v_norms + row0 + lane);
  }
}

template <int G, int KB, int VB>
__global__ void __launch_bounds__(kThreads, 1) decode_split_kernel(const DecodeParams p) {
  using C = Cfg<KB, VB>;
  constexpr int S = C::kStages;
  extern __shared__ __align__(16) uint8_t smem[];
  uint8_t* ktab = smem;                         // pair tables first: constant offsets
  uint8_t* vtab = smem + C::kKTab;
  uint8_t* stages = smem + C::kKTab + C::kVTab;
  uint8_t* wts_all = stages + kWarps * S * C::kBuf;
  float* qs = reinterpret_cast<float*>(wts_all + kWarps * C::kWts);
  float* comb = qs + 4 * D;
  float* wml = comb + 4 * D;                    // [warp][head][2]
  int4* descs_all = reinterpret_cast<int4*>(wml + kWarps * 4 * 2);  // [warp][stage] tile descriptors
  long long* prefix = reinterpret_cast<long long*>(descs_all + kWarps * 4);
  long long* scan = prefix + kMaxDecodeBatch + 1;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 3, r = lane & 7;
  const uint32_t copy8 = (lane & (kCopies - 1)) * 8u;

  if (blockIdx.x == 0 && tid == 0 && p.status != nullptr) {
    for (int b = 0; b < p.batch; ++b) {
      const int len = p.seq_lens[b];
      if (len < 0 || len > p.cap || len > p.max_seq_len) {
        atomicOr(p.status, TQ_DEV_ERR_SEQ_LEN);
        break;
      }
    }
  }
  // pair tables: entry e = code_a | code_b << bits -> (c[code_a], c[code_b]), copies interleaved
  if constexpr (!C::kFp16K) {
    constexpr int n = (1 << (2 * (C::kFp16K ? 1 : KB))) * kCopies;
    for (int i = tid; i < n; i += kThreads) {
      const int e = i / kCopies;
      reinterpret_cast<float2*>(ktab)[i] = make_float2(p.k_cent[e & ((1 << KB) - 1)], p.k_cent[e >> KB]);
    }
  }
  {
    constexpr int n = (1 << (2 * VB)) * kCopies;
    for (int i = tid; i < n; i += kThreads) {
      const int e = i / kCopies;
      reinterpret_cast<float2*>(vtab)[i] = make_float2(p.v_cent[e & ((1 << VB) - 1)], p.v_cent[e >> VB]);
    }
  }
  tile_prefix<kThreads>(p, prefix, scan);  // synchronizes
  const long long total = prefix[p.batch];
  const long long t0 = total * blockIdx.x / p.grid, t1 = total * (blockIdx.x + 1) / p.grid;
  if (t0 >= t1) return;

  uint8_t* wbuf = stages + warp * S * C::kBuf;
  uint8_t* wts = wts_all + warp * C::kWts;
  int4* descs = descs_all + warp * 4;
  const int my_n = static_cast<int>((t1 - t0 - warp + kWarps - 1) / kWarps);  // tiles t0 + warp + 8 j
  int j_issue = 0, j = 0;
  // stage tile j_issue and record its descriptor {b, h | hot << 16, t_begin, n_valid}
  auto issue = [&]() {
    if (j_issue < my_n) {
      const TileInfo ti = tile_info(p, prefix, t0 + warp + static_cast<long long>(kWarps) * j_issue);
      stage_tile<KB, VB>(p, ti, wbuf + (j_issue % S) * C::kBuf, lane);
      if (lane == 0) descs[j_issue % S] = make_int4(ti.b, ti.h | (ti.hot << 16), ti.t_begin, ti.n_valid);
    }
    cp_async_commit();
    ++j_issue;
  };
#pragma unroll
  for (int s = 0; s < S - 1; ++s) issue();

  float2 qr[G][8];
  int cur_b = -1, cur_h = -1;
  long long seg = t0;
  while (seg < t1) {
    const TileInfo si = tile_info(p, prefix, seg);
    const long long seg_end = si.row_end < t1 ? si.row_end : t1;
    if (si.b != cur_b || si.h != cur_h) {
      // rotated query of the G heads: (log2 e / d) H D q for packed K, (log2 e / sqrt d) q for fp16 K
      __syncthreads();
      if (tid < D) {
        const bool neg = !C::kFp16K && sign_negative(p.seed, p.layer, si.h, tid);
#pragma unroll
        for (int jj = 0; jj < G; ++jj) {
          float x = half_bits_to_float(p.q[(static_cast<int64_t>(si.b) * p.hq + si.h * G + jj) * D + tid]);
          qs[jj * D + tid] = neg ? -x : x;
        }
      }
      __syncthreads();
      if constexpr (!C::kFp16K) {
#pragma unroll
        for (int st = 1; st < D; st *= 2) {
          if (tid < D && (tid & st) == 0) {
#pragma unroll
            for (int jj = 0; jj < G; ++jj) {
              const float a = qs[jj * D + tid], c = qs[jj * D + tid + st];
              qs[jj * D + tid] = fadd(a, c);
              qs[jj * D + tid + st] = fsub(a, c);
            }
          }
          __syncthreads();
        }
      }
      const float qscale = C::kFp16K ? kLog2e / kSqrtD : kLog2e / static_cast<float>(D);
#pragma unroll
      for (int jj = 0; jj < G; ++jj)
#pragma unroll
        for (int k = 0; k < 8; ++k)
          qr[jj][k] = make_float2(fmul(qs[jj * D + 16 * r + 2 * k], qscale),
                                  fmul(qs[jj * D + 16 * r + 2 * k + 1], qscale));
      cur_b = si.b;
      cur_h = si.h;
    }

    // per-group online-softmax state of this row
    float m[G], lsum[G];
    float2 acc[G][8];
#pragma unroll
    for (int jj = 0; jj < G; ++jj) {
      m[jj] = -INFINITY;
      lsum[jj] = 0.0f;
#pragma unroll
      for (int k = 0; k < 8; ++k) acc[jj][k] = make_float2(0.0f, 0.0f);
    }

    while (j < my_n && t0 + warp + static_cast<long long>(kWarps) * j < seg_end) {
      issue();
      cp_async_wait<S - 1>();
      __syncwarp();

      const int4 dsc = descs[j % S];
      TileInfo ti;
      ti.b = dsc.x;
      ti.h = dsc.y & 0xFFFF;
      ti.hot = dsc.y >> 16;
      ti.t_begin = dsc.z;
      ti.n_valid = dsc.w;
      const uint8_t* tb = wbuf + (j % S) * C::kBuf;
      const bool hot = ti.hot != 0;

      // ---- scores: P[u][h] = partial over this lane's 16 coordinates of token 8g + u
      float P[8][G];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int tau = 8 * g + u;
        float2 pa[G], pb[G];
#pragma unroll
        for (int jj = 0; jj < G; ++jj) pa[jj] = pb[jj] = make_float2(0.0f, 0.0f);
        if constexpr (C::kFp16K) {
          const uint4* kr = reinterpret_cast<const uint4*>(tb + tau * 256) + 2 * r;
          const uint4 a0 = kr[0], a1 = kr[1];
          const uint32_t wv[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const float2 kf = half2_bits_to_float2(wv[k]);
#pragma unroll
            for (int jj = 0; jj < G; ++jj) {
              if (k & 1) pb[jj] = fma2(qr[jj][k], kf, pb[jj]);
              else pa[jj] = fma2(qr[jj][k], kf, pa[jj]);
            }
          }
        } else {
          constexpr int KBB = C::kFp16K ? 2 : KB;
          const Win win = code_window<KBB>(tb + tau * C::kKRow, r);
          float2 cp[8];
          cp[0] = *reinterpret_cast<const float2*>(ktab + pair_offset<KBB, 0>(win, copy8));
          cp[1] = *reinterpret_cast<const float2*>(ktab + pair_offset<KBB, 1>(win, copy8));
          cp[2] = *reinterpret_cast<const float2*>(ktab + pair_offset<KBB, 2>(win, copy8));
          cp[3] = *reinterpret_cast<const float2*>(ktab + pair_offset<KBB, 3>(win, copy8));
          cp[4] = *reinterpret_cast<const float2*>(ktab + pair_offset<KBB, 4>(win, copy8));
          cp[5] = *reinterpret_cast<const float2*>(ktab + pair_offset<KBB, 5>(win, copy8));
          cp[6] = *reinterpret_cast<const float2*>(ktab + pair_offset<KBB, 6>(win, copy8));
          cp[7] = *reinterpret_cast<const float2*>(ktab + pair_offset<KBB, 7>(win, copy8));
#pragma unroll
          for (int k = 0; k < 8; ++k)
#pragma unroll
            for (int jj = 0; jj < G; ++jj) {
              if (k & 1) pb[jj] = fma2(qr[jj][k], cp[k], pb[jj]);
              else pa[jj] = fma2(qr[jj][k], cp[k], pa[jj]);
            }
        }
#pragma unroll
        for (int jj = 0; jj < G; ++jj) {
          const float2 s2 = add2(pa[jj], pb[jj]);
          P[u][jj] = fadd(s2.x, s2.y);
        }
      }
      // ---- transposing butterfly over the 8 lanes of a group: lane r ends with token 8g + r
      float v4[4][G], v2[2][G], s[G];
      {
        const bool up = (r & 4) != 0;
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
          for (int jj = 0; jj < G; ++jj) {
            const float send = up ? P[k][jj] : P[k + 4][jj];
            const float keep = up ? P[k + 4][jj] : P[k][jj];
            v4[k][jj] = fadd(keep, __shfl_xor_sync(0xffffffffu, send, 4));
          }
      }
      {
        const bool up = (r & 2) != 0;
#pragma unroll
        for (int k = 0; k < 2; ++k)
#pragma unroll
          for (int jj = 0; jj < G; ++jj) {
            const float send = up ? v4[k][jj] : v4[k + 2][jj];
            const float keep = up ? v4[k + 2][jj] : v4[k][jj];
            v2[k][jj] = fadd(keep, __shfl_xor_sync(0xffffffffu, send, 2));
          }
      }
      {
        const bool up = (r & 1) != 0;
#pragma unroll
        for (int jj = 0; jj < G; ++jj) {
          const float send = up ? v2[0][jj] : v2[1][jj];
          const float keep = up ? v2[1][jj] : v2[0][jj];
          s[jj] = fadd(keep, __shfl_xor_sync(0xffffffffu, send, 1));
        }
      }
      // ---- online softmax per 8-token group; lane l holds token l
      const bool valid = lane < ti.n_valid;
      const float nk = C::kFp16K ? 1.0f : reinterpret_cast<const float*>(tb + C::kKTile)[lane];
      const float nv = hot ? 1.0f : reinterpret_cast<const float*>(tb + C::kKTile + C::kKNorm + C::kVTile)[lane];
      float alpha[G];
      bool rescale = false;
      float4* wrow = reinterpret_cast<float4*>(wts + (lane + g) * 32);  // padded row of token `lane`
      float wv4[G];
#pragma unroll
      for (int jj = 0; jj < G; ++jj) {
        const float sj = valid ? fmul(s[jj], nk) : -INFINITY;
        float gmax = sj;
        gmax = fmaxf(gmax, __shfl_xor_sync(0xffffffffu, gmax, 1));
        gmax = fmaxf(gmax, __shfl_xor_sync(0xffffffffu, gmax, 2));
        gmax = fmaxf(gmax, __shfl_xor_sync(0xffffffffu, gmax, 4));
        const float mn = fmaxf(m[jj], gmax);
        alpha[jj] = mn == -INFINITY ? 1.0f : exp2f(m[jj] - mn);
        rescale |= alpha[jj] != 1.0f;
        const float pj = valid ? exp2f(sj - mn) : 0.0f;
        lsum[jj] = ffma(lsum[jj], alpha[jj], pj);
        m[jj] = mn;
        wv4[jj] = valid ? fmul(pj, nv) : 0.0f;  // staged norms of masked rows are garbage
      }
      if constexpr (G == 4) {
        wrow[0] = make_float4(wv4[0], wv4[0], wv4[1], wv4[1]);
        wrow[1] = make_float4(wv4[2], wv4[2], wv4[3], wv4[3]);
      } else if constexpr (G == 2) {
        wrow[0] = make_float4(wv4[0], wv4[0], wv4[1], wv4[1]);
      } else {
        reinterpret_cast<float2*>(wrow)[0] = make_float2(wv4[0], wv4[0]);
      }
      if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
        for (int jj = 0; jj < G; ++jj)
#pragma unroll
          for (int k = 0; k < 8; ++k) acc[jj][k] = mul2(acc[jj][k], make_float2(alpha[jj], alpha[jj]));
      }
      __syncwarp();

      // ---- V accumulation for tokens 8g + u
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int tau = 8 * g + u;
        const float2* wr = reinterpret_cast<const float2*>(wts + (tau + g) * 32);
        float2 w2[G];
        if constexpr (G == 4) {
          const float4 a = reinterpret_cast<const float4*>(wr)[0], b2 = reinterpret_cast<const float4*>(wr)[1];
          w2[0] = make_float2(a.x, a.y);
          w2[1] = make_float2(a.z, a.w);
          w2[2] = make_float2(b2.x, b2.y);
          w2[3] = make_float2(b2.z, b2.w);
        } else {
#pragma unroll
          for (int jj = 0; jj < G; ++jj) w2[jj] = wr[jj];
        }
        if (!hot) {
          const Win win = code_window<VB>(tb + C::kKTile + C::kKNorm + tau * C::kVRow, r);
          float2 cv[8];
          cv[0] = *reinterpret_cast<const float2*>(vtab + pair_offset<VB, 0>(win, copy8));
          cv[1] = *reinterpret_cast<const float2*>(vtab + pair_offset<VB, 1>(win, copy8));
          cv[2] = *reinterpret_cast<const float2*>(vtab + pair_offset<VB, 2>(win, copy8));
          cv[3] = *reinterpret_cast<const float2*>(vtab + pair_offset<VB, 3>(win, copy8));
          cv[4] = *reinterpret_cast<const float2*>(vtab + pair_offset<VB, 4>(win, copy8));
          cv[5] = *reinterpret_cast<const float2*>(vtab + pair_offset<VB, 5>(win, copy8));
          cv[6] = *reinterpret_cast<const float2*>(vtab + pair_offset<VB, 6>(win, copy8));
          cv[7] = *reinterpret_cast<const float2*>(vtab + pair_offset<VB, 7>(win, copy8));
#pragma unroll
          for (int k = 0; k < 8; ++k)
#pragma unroll
            for (int jj = 0; jj < G; ++jj) acc[jj][k] = fma2(w2[jj], cv[k], acc[jj][k]);
        } else if (tau < ti.n_valid) {
          const int pos = ti.t_begin + tau;
          const uint4* vr = reinterpret_cast<const uint4*>(
                                p.v_ring + ((static_cast<int64_t>(ti.b) * p.hkv + ti.h) * p.hot + pos % p.hot) * D) +
                            2 * r;
          const uint4 a0 = vr[0], a1 = vr[1];
          const uint32_t wv[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const float2 vf = half2_bits_to_float2(wv[k]);
#pragma unroll
            for (int jj = 0; jj < G; ++jj) acc[jj][k] = fma2(w2[jj], vf, acc[jj][k]);
          }
        }
      }
      __syncwarp();
      ++j;
    }

    // ---- leave the row: groups -> warp -> CTA, one partial per (CTA, row)
    for (int i = tid; i < G * D; i += kThreads) comb[i] = 0.0f;
    float mw[G];
#pragma unroll
    for (int jj = 0; jj < G; ++jj) {
      float mx = fmaxf(m[jj], __shfl_xor_sync(0xffffffffu, m[jj], 8));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      const float sc = m[jj] == -INFINITY ? 0.0f : exp2f(m[jj] - mx);
      float l = fmul(lsum[jj], sc);
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) l = fadd(l, __shfl_xor_sync(0xffffffffu, l, o));
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        float2 a = mul2(acc[jj][k], make_float2(sc, sc));
        a.x = fadd(a.x, __shfl_xor_sync(0xffffffffu, a.x, 8));
        a.y = fadd(a.y, __shfl_xor_sync(0xffffffffu, a.y, 8));
        a.x = fadd(a.x, __shfl_xor_sync(0xffffffffu, a.x, 16));
        a.y = fadd(a.y, __shfl_xor_sync(0xffffffffu, a.y, 16));
        acc[jj][k] = a;
      }
      mw[jj] = mx;
      if (lane == 0) {
        wml[(warp * 4 + jj) * 2] = mx;
        wml[(warp * 4 + jj) * 2 + 1] = l;
      }
    }
    __syncthreads();
    if (g == 0) {
#pragma unroll
      for (int jj = 0; jj < G; ++jj) {
        if (mw[jj] == -INFINITY) continue;
        float mm = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) mm = fmaxf(mm, wml[(w * 4 + jj) * 2]);
        const float sc = exp2f(mw[jj] - mm);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          atomicAdd(&comb[jj * D + 16 * r + 2 * k], fmul(acc[jj][k].x, sc));
          atomicAdd(&comb[jj * D + 16 * r + 2 * k + 1], fmul(acc[jj][k].y, sc));
        }
      }
    }
    __syncthreads();
    const long long slot = static_cast<long long>(blockIdx.x) + si.row;
    for (int i = tid; i < G * D; i += kThreads) p.ws_acc[slot * G * D + i] = comb[i];
    if (tid < G) {
      float mm = -INFINITY, ll = 0.0f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) mm = fmaxf(mm, wml[(w * 4 + tid) * 2]);
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float mwv = wml[(w * 4 + tid) * 2];
        if (mwv != -INFINITY) ll = ffma(wml[(w * 4 + tid) * 2 + 1], exp2f(mwv - mm), ll);
      }
      p.ws_ml[(slot * G + tid) * 2] = mm;
      p.ws_ml[(slot * G + tid) * 2 + 1] = ll;
    }
    __syncthreads();
    seg = seg_end;
  }
  cp_async_wait<0>();
}

// CTA of the split kernel that processes tile t (the last one whose range starts at or before t).
__device__ __forceinline__ int cta_of(long long t, long long total, int grid) {
  return static_cast<int>(((t + 1) * grid - 1) / total);
}
__device__ __forceinline__ long long cta_start(int c, long long total, int grid) { return total * c / grid; }

__global__ void __launch_bounds__(D) decode_merge_kernel(const DecodeParams p) {
  __shared__ float y[D];
  __shared__ long long prefix[kMaxDecodeBatch + 1];
  __shared__ long long scan[34];
  const int hq = blockIdx.x, b = blockIdx.y, t = threadIdx.x;
  const int g = p.hq / p.hkv, h = hq / g, jj = hq - h * g;
  float* out = p.out + (static_cast<int64_t>(b) * p.hq + hq) * D;
  tile_prefix<D>(p, prefix, scan);
  const long long total = prefix[p.batch];
  const SeqTiles st = seq_tiles(p, b);
  if (st.len == 0) {
    out[t] = 0.0f;
    return;
  }
  const int per_h = st.tc + st.th;
  const long long hbase = prefix[b] + static_cast<long long>(h) * per_h;
  // rows of this (b, h): cold [hbase, hbase + tc), hot [hbase + tc, hbase + per_h)
  float mm = -INFINITY;
  for (int kind = 0; kind < 2; ++kind) {
    const long long rs = kind ? hbase + st.tc : hbase, re = kind ? hbase + per_h : hbase + st.tc;
    if (re <= rs) continue;
    const int row = (b * p.hkv + h) * 2 + kind;
    for (int c = cta_of(rs, total, p.grid); c <= cta_of(re - 1, total, p.grid); ++c) {
      if (cta_start(c, total, p.grid) == cta_start(c + 1, total, p.grid)) continue;  // empty CTA range
      mm = fmaxf(mm, p.ws_ml[((static_cast<long long>(c) + row) * g + jj) * 2]);
    }
  }
  float cold = 0.0f, hotv = 0.0f, l = 0.0f;
  for (int kind = 0; kind < 2; ++kind) {
    const long long rs = kind ? hbase + st.tc : hbase, re = kind ? hbase + per_h : hbase + st.tc;
    if (re <= rs) continue;
    const int row = (b * p.hkv + h) * 2 + kind;
    for (int c = cta_of(rs, total, p.grid); c <= cta_of(re - 1, total, p.grid); ++c) {
      if (cta_start(c, total, p.grid) == cta_start(c + 1, total, p.grid)) continue;
      const long long slot = static_cast<long long>(c) + row;
      const float ms = p.ws_ml[(slot * g + jj) * 2];
      if (ms == -INFINITY) continue;
      const float sc = exp2f(ms - mm);
      l = ffma(p.ws_ml[(slot * g + jj) * 2 + 1], sc, l);
      const float a = p.ws_acc[(slot * g + jj) * D + t];
      if (kind) hotv = ffma(a, sc, hotv);
      else cold = ffma(a, sc, cold);
    }
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
  out[t] = fadd(v, hotv) / l;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

template <int G, int KB, int VB>
tq_status launch_split(const DecodeParams& p, cudaStream_t stream) {
  using C = Cfg<KB, VB>;
  auto kern = decode_split_kernel<G, KB, VB>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem) != cudaSuccess)
    return TQ_ERR_CUDA;
  kern<<<p.grid, kThreads, C::kSmem, stream>>>(p);
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
  if (max_seq_len == 0) return 0;
  return decode_workspace_bytes(d);
}

extern "C" tq_status tq_decode_attention(const tq_cache_desc* d, const void* q, const int32_t* d_seq_lens,
                                         int32_t max_seq_len, float* out, void* workspace, size_t workspace_bytes,
                                         tq_stream_t stream) {
  using namespace tq;
  const tq_status vs = validate_desc(d);
  if (vs != TQ_OK) return vs;
  if (q == nullptr || d_seq_lens == nullptr || out == nullptr || max_seq_len < 0) return TQ_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(out)) return TQ_ERR_INVALID_ARG;
  if (d->batch > kMaxDecodeBatch) return TQ_ERR_UNSUPPORTED;
  if (static_cast<long long>(d->num_kv_heads) * (d->capacity / 32 + d->hot_window / 32 + 2) >= (1ll << 31))
    return TQ_ERR_UNSUPPORTED;  // tiles of one sequence must fit in 32 bits
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t out_bytes = static_cast<size_t>(d->batch) * d->num_q_heads * D * sizeof(float);
  if (max_seq_len == 0) return cudaMemsetAsync(out, 0, out_bytes, s) == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
  const size_t need = tq_decode_workspace_bytes(d, max_seq_len);
  if (workspace == nullptr || !aligned16(workspace) || workspace_bytes < need) return TQ_ERR_WORKSPACE;
  const int sms = sm_count();
  if (sms <= 0) return TQ_ERR_CUDA;

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
  const int g = d->num_q_heads / d->num_kv_heads;
  const size_t slots = decode_workspace_slots(d);
  p.ws_acc = static_cast<float*>(workspace);
  p.ws_ml = p.ws_acc + slots * g * D;
  p.grid = sms < kMaxDecodeCtas ? sms : kMaxDecodeCtas;
  p.out = out;

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
