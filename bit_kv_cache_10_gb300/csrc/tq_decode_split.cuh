// Split-K decode kernel over the packed cache, included by the decode
// translation units (dense or sparse V, contiguous or paged layout, one or
// several query tokens per sequence; each instantiates one variant).
//
// Work list.  Every (sequence b, KV head h) has a cold row (the packed
// positions [0, L - min(W, L))) and, with a hot window, a hot row (the newest
// min(W, L) positions, whose V is read from the fp16 ring).  Rows are cut into
// 16-token tiles and listed in (b, h, cold/hot) order; the list is split into
// one contiguous, equal range per CTA, so that every SM gets the same number
// of tiles whatever the lengths are.  For attention of nq query tokens per
// sequence (MQ variants) every query token is a sequence of the list of its
// own, whose length is its causal prefix; its tiles are read from the cache
// rows of the sequence it belongs to.
//
// This float32 kernel serves V of 2 or 3 bits (packed or fp16 K); packed K of
// 2..4 bits or fp16 K with 4-bit V and the int8 mode run the tensor-core kernel
// (tq_decode_mma.cuh), which shares the work list, the staging and the merge.
//
// Split kernel: one CTA of 8 warps per SM (up to 255 registers per thread).  The
// codebook pair tables are built once per CTA in shared memory (16 copies, one
// per lane of a half-warp, so the data-dependent lookups are bank-conflict
// free), at a base aligned to the table size so that a lookup address is one
// PRMT (4-bit codes) or one shift and one masked OR.  Warp w takes tiles
// t0 + w, t0 + w + 8, ... of the CTA's range and streams them through a cp.async
// ring of up to 8 tiles that runs across row boundaries.  Per tile:
//   scores:  packed K: 8 lanes share a token, each owning 16 coordinates (8 code
//            pairs, each looked up at once as (c_a, c_b)); 4 tokens per step, 4 steps.
//            fp16 K: on the tensor cores (mma m16n8k16, exact fp16 operands),
//            the softmax in the MMA fragment layout.
//            Partial sums over the lane's coordinates for the G query heads,
//            then a 3-stage transposing butterfly over the 8 lanes leaves each
//            lane with the full scores of one token for G/2 heads;
//   softmax: online over the tile in base 2 (log2 e is folded into q'); the
//            running maximum is raised lazily (only when a score exceeds it by
//            more than 2^8), so most tiles need no cross-lane maximum or rescale;
//   V:       16 lanes share a token, each owning 8 coordinates; 2 tokens per
//            step, 8 steps: acc[h][i] += p_h n_V c[code_i] in the rotated domain
//            (cold rows) or += p_h v_i with the raw fp16 V (hot rows).
// When the CTA leaves a row it combines its warps and writes one partial
// (acc, max, sum) to workspace slot (CTA index + row index): these slots are
// distinct for all (CTA, row) pairs because both indices only grow along the
// tile list.  All arithmetic is float32 (packed pairs where possible).
//
// Merge kernel: one warp per (sequence, query head): finds the CTAs that
// covered its cold and hot rows, log-sum-exp combines their partials, rotates
// the cold sum back once (D_h H / sqrt(d)), adds the hot sum and divides by
// the softmax mass.
#pragma once

#include <cstring>
#include <type_traits>

#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {

struct DecodeParams {
  const uint16_t* q;
  const int* seq_lens;
  int max_seq_len;
  int batch, hkv, hq, cap, hot;  // batch: sequences x nq query tokens (the work list's "sequences")
  int nq;         // query tokens per cache sequence (1: decode)
  const uint32_t* k_words;
  const float* k_norms;
  const uint16_t* k_fp16;
  const uint32_t* v_words;
  const float* v_norms;
  const uint16_t* v_ring;
  RowMap map;     // cache row of (b, h, t): contiguous or through the block table
  uint32_t* status;
  uint64_t seed;
  int layer;
  float k_cent[16];
  float v_cent[16];
  float* ws_acc;  // [slots][G][D]
  float* ws_ml;   // [slots][G][2] (max, sum)
  float sparse_tau;  // sparse-V threshold (0: dense)
  int rotated;    // 1: V is summed in the rotated domain (packed modes); 0: int8 mode
  int grid;       // CTAs of the split kernel
  float* out;     // [B, Hq, D]
};

namespace {

constexpr int kTile = 16;
constexpr int kCopies = 16;                 // pair-table copies (one per lane of a half-warp)
constexpr int kSmemBudget = 227 * 1024;
constexpr float kLazy = 8.0f;               // log2 headroom of the lazily raised softmax maximum



__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

// Length of cache sequence b, or 0 when it is outside [0, min(cap, max_seq_len)].
__device__ __forceinline__ int seq_len(const DecodeParams& p, int b) {
  const int len = p.seq_lens[b];
  return (len >= 0 && len <= p.cap && len <= p.max_seq_len) ? len : 0;
}

// Cache sequence of work-list sequence v (v itself for decode; MQ: kernels
// compiled for several query tokens per sequence).
template <bool MQ>
__device__ __forceinline__ int cache_seq(const DecodeParams& p, int v) { return MQ ? v / p.nq : v; }

struct SeqTiles {
  int len, ce, tc, th;  // length, cold end, cold tiles, hot tiles
};
// Work-list sequence v is query token i = v mod nq of cache sequence b = v / nq:
// with the cache holding L positions it sits at position L - nq + i and attends
// to the prefix [0, L - nq + i + 1) (causal).  The cold end is the cache
// sequence's, so that hot positions are the ones in the fp16 ring.
template <bool MQ>
__device__ __forceinline__ SeqTiles seq_tiles(const DecodeParams& p, int v) {
  SeqTiles s;
  const int b = cache_seq<MQ>(p, v);
  const int L = seq_len(p, b);
  s.len = MQ ? max(0, L - (p.nq - 1 - (v - b * p.nq))) : L;
  const int ce = p.hot > 0 ? L - min(p.hot, L) : L;
  s.ce = min(ce, s.len);
  s.tc = (s.ce + kTile - 1) / kTile;
  s.th = (s.len - s.ce + kTile - 1) / kTile;
  return s;
}

// Exclusive prefix (over sequences) of the tile counts, prefix[0..B], in
// shared memory; all threads of the block must call it.  Uses `scratch`
// (at least 33 long longs).
template <int NT, bool MQ>
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
      const SeqTiles s = seq_tiles<MQ>(p, b);
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

template <bool MQ>
__device__ __forceinline__ TileInfo tile_info(const DecodeParams& p, const long long* prefix, long long t) {
  int lo = 0, hi = p.batch;  // largest b with prefix[b] <= t
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] <= t) lo = mid;
    else hi = mid;
  }
  TileInfo ti;
  ti.b = lo;
  const SeqTiles s = seq_tiles<MQ>(p, lo);
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
  static constexpr bool kInt8 = KB == 8;               // int8 mode: K and V int8 codes with absmax scales
  static_assert(!kInt8 || VB == 8, "the int8 mode has int8 K and V");
  static constexpr int kKBits = kFp16K ? 2 : KB;       // placeholder width when K is fp16
  static constexpr int kKRow = kFp16K ? 256 : KB * 16;  // bytes of one K token
  static constexpr int kVRow = VB * 16;
  // fp16 and int8 K: scores on the tensor cores (their values are exact in fp16; the
  // int8 staging layout also serves the tensor-core kernel, which runs that mode);
  // the staged K rows are padded so that the MMA operand loads of 4 tokens by 4
  // lanes each fall in distinct banks (288 = 256 + 32, 144 = 128 + 16 bytes)
  static constexpr bool kMmaK = kFp16K || kInt8;
  // warps per CTA (one CTA per SM): 8 at up to 255 registers; the tensor-core
  // variants need about 160, so 12 warps fit (int8 0.192 -> 0.174 ms, asym 0.077 ->
  // 0.073 ms against 8 warps)
  static constexpr int kWarps = kMmaK ? 12 : 8;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kKPitch = kFp16K ? kKRow + 32 : kInt8 ? kKRow + 16 : kKRow;
  static constexpr int kKTile = kTile * kKPitch;
  static constexpr int kKNorm = kFp16K ? 0 : kTile * 4;
  static constexpr int kVTile = kTile * kVRow;
  static constexpr int kBuf = kKTile + kKNorm + kVTile + kTile * 4;  // K | K norms | V | V norms
  // Pair tables.  Packed K: 256-byte rows, V entries in bytes [0,128), K entries in
  // [128,256) of row e (16 copies x 8 bytes); fp16 K: V only, 128-byte rows.  The
  // table base is aligned to the table size so that an entry's address is
  // base | (e << row_shift) | copy * 8 (one OR instead of an add).
  // The int8 mode needs no table: a 1 KB placeholder keeps the layout code uniform.
  static constexpr int kRowShift = kFp16K ? 7 : 8;
  static constexpr int kTabBits = kInt8 ? 2 : kFp16K ? 2 * VB : 2 * (VB > kKBits ? VB : kKBits);
  static constexpr int kTab = (1 << kTabBits) << kRowShift;
  static constexpr int kWts = kTile * 32;  // per warp: up to 4 head weights per token (16 bytes used)
  static constexpr int kSmall = kWarps * kWts + 4 * D * 4 /* q' */ + 4 * D * 4 /* combine */ +
                                kWarps * 4 * 2 * 4 /* warp (m, l) */ + kWarps * 8 * 16 /* tile descriptors */ +
                                (kMaxDecodeBatch + 1) * 8 + 34 * 8;
  // the aligned table can leave a gap of up to kTab - 1024 bytes before it (shared
  // windows start at a 1 KB multiple); buffers are placed around the table
  static constexpr int kWorst(int stages) { return kTab + kSmall + (kWarps + 1) * stages * kBuf + 1024; }
  static constexpr int kStages = kWorst(8) <= kSmemBudget ? 8 : kWorst(6) <= kSmemBudget ? 6 : kWorst(4) <= kSmemBudget ? 4 : kWorst(3) <= kSmemBudget ? 3 : 2;
  // requested dynamic shared memory: the layout's bound (1 KB multiple), so that
  // a small kernel (the decode step's append) can share the SM with a CTA
  static constexpr int kSmem = (kWorst(kStages) + 1023) / 1024 * 1024;
  static_assert(kWorst(kStages) <= kSmemBudget, "shared memory budget");
};

// Bump allocator over the dynamic shared window that skips the table region.
struct SmemLayout {
  uint32_t cur, tab_lo, tab_hi;
  __device__ uint32_t take(uint32_t bytes) {
    cur = (cur + 15u) & ~15u;
    if (cur < tab_hi && cur + bytes > tab_lo) cur = tab_hi;
    const uint32_t at = cur;
    cur += bytes;
    return at;
  }
};

// ---- lane maps --------------------------------------------------------------
// K phase: lane = 8 s + rr; token slot s (0..3) and 16 coordinates per lane,
// as 8 coordinate pairs.  Packed 4- and 2-bit K: coordinates 16 rr .. 16 rr + 15
// (one aligned 64- or 32-bit load per token).  Packed 3-bit and fp16 K: two
// chunks, 8 rr .. 8 rr + 7 and 64 + 8 rr .. 64 + 8 rr + 7 (equal bit shifts in
// both chunks for 3-bit; consecutive 16-byte chunks per quarter-warp for fp16).
template <int KB>
__device__ __forceinline__ int k_pair_coord(int rr, int pr) {
  if constexpr (KB == 4 || KB == 2 || KB == 8) return 16 * rr + 2 * pr;
  else return (pr >> 2) * 64 + 8 * rr + 2 * (pr & 3);
}
// Tile token of K step u (0..3) in slot s.  For 48-byte (3-bit) records the
// four tokens of a step start 8 banks apart, so that the window loads of the
// whole warp are conflict free; other widths take four consecutive tokens.
template <int KB>
__device__ __forceinline__ constexpr int k_token(int u, int s) {
  return KB == 3 ? 8 * (u >> 1) + (u & 1) + 2 * s : 4 * u + s;
}
// Byte offset of the K-phase lane's first window word within a staged K tile.
template <int KB>
__device__ __forceinline__ uint32_t k_lane_offset(int s, int rr) {
  constexpr int kRec = KB == 16 ? 256 : KB * 16;
  const uint32_t tok = static_cast<uint32_t>(k_token<KB>(0, s) * kRec);
  if constexpr (KB == 16 || KB == 8) return tok + 16u * rr;
  else if constexpr (KB == 4) return tok + 8u * rr;
  else if constexpr (KB == 2) return tok + 4u * rr;
  else return tok + 4u * ((3 * rr) >> 2);
}
// V phase: lane = 16 g + r, coordinates 8 r .. 8 r + 7, token 2 u + g at step u.
template <int VB>
__device__ __forceinline__ uint32_t v_lane_offset(int g, int r) {
  const uint32_t tok = static_cast<uint32_t>(g * VB * 16);
  if constexpr (VB == 8) return tok + 8u * r;
  else if constexpr (VB == 4) return tok + 4u * r;
  else if constexpr (VB == 2) return tok + 4u * (r >> 1);
  else return tok + 4u * ((3 * r) >> 2);
}
template <int VB>
__device__ __forceinline__ uint32_t v_lane_shift(int r) {
  if constexpr (VB == 4 || VB == 8) return 0u;
  else if constexpr (VB == 2) return 16u * (r & 1);
  else return (24u * r) & 31u;
}

// Shared address of the table entry of code pair K (bits 2*BITS*K ..) of a
// window: basecopy = table base | (128 for K) | copy * 8.
template <int BITS, int K, int ROWSHIFT>
__device__ __forceinline__ uint32_t pair_addr(uint32_t win, uint32_t basecopy) {
  if constexpr (BITS == 4 && ROWSHIFT == 8) {
    // byte K of the window into byte 1; bytes 0, 2, 3 from basecopy
    return __byte_perm(win, basecopy, 0x7604 | (K << 4));
  } else {
    constexpr int kP = 2 * BITS * K, kW = 2 * BITS;
    const uint32_t v = kP >= ROWSHIFT ? (win >> (kP >= ROWSHIFT ? kP - ROWSHIFT : 0))
                                      : (win << (kP < ROWSHIFT ? ROWSHIFT - kP : 0));
    return (v & (((1u << kW) - 1u) << ROWSHIFT)) | basecopy;
  }
}

__device__ __forceinline__ float2 lds64(uint32_t addr) {
  float2 v;
  asm("ld.shared.v2.f32 {%0, %1}, [%2];\n" : "=f"(v.x), "=f"(v.y) : "r"(addr));
  return v;
}

// D += A B on the tensor cores, m16n8k16, f16 operands, f32 accumulators.  Only
// A rows 0..7 are used (the query heads): their fragment registers a1 and a3
// (rows 8..15) are zero.
__device__ __forceinline__ void mma_16816(float& d0, float& d1, float& d2, float& d3, uint32_t a0, uint32_t a2,
                                          uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};\n"
      : "+f"(d0), "+f"(d1), "+f"(d2), "+f"(d3)
      : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}
// Two int8 codes (bytes K and K + 1 of a biased word xw = w ^ 0x80808080) as an
// exact f16 pair: the byte u = code + 128 becomes the mantissa of 1024 + u, and
// one packed subtraction of 1152 leaves the code.
template <int K>
__device__ __forceinline__ uint32_t int8_half2(uint32_t xw) {
  const uint32_t h = __byte_perm(xw, 0x64646464u, 0x4040 | (K + 1) << 8 | K);
  const __half2 r = __hsub2(*reinterpret_cast<const __half2*>(&h), __floats2half2_rn(1152.0f, 1152.0f));
  return *reinterpret_cast<const uint32_t*>(&r);
}

// Shared loads at a register base plus a compile-time byte offset (no address arithmetic).
template <int OFF>
__device__ __forceinline__ uint32_t lds32(uint32_t base) {
  uint32_t v;
  asm("ld.shared.u32 %0, [%1+%2];\n" : "=r"(v) : "r"(base), "n"(OFF));
  return v;
}
template <int OFF>
__device__ __forceinline__ uint2 lds64u(uint32_t base) {
  uint2 v;
  asm("ld.shared.v2.u32 {%0, %1}, [%2+%3];\n" : "=r"(v.x), "=r"(v.y) : "r"(base), "n"(OFF));
  return v;
}
template <int OFF>
__device__ __forceinline__ uint4 lds128(uint32_t base) {
  uint4 v;
  asm("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4+%5];\n" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(base), "n"(OFF));
  return v;
}
template <int OFF>
__device__ __forceinline__ float4 lds128f(uint32_t base) {
  float4 v;
  asm("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4+%5];\n" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(base), "n"(OFF));
  return v;
}
template <int OFF>
__device__ __forceinline__ float2 lds64f(uint32_t base) {
  float2 v;
  asm("ld.shared.v2.f32 {%0, %1}, [%2+%3];\n" : "=f"(v.x), "=f"(v.y) : "r"(base), "n"(OFF));
  return v;
}

// Issue cursor: the tile a warp stages next, advanced by the warp stride
// without searching the tile list again.
struct Cursor {
  int b, h, x;              // work-list sequence, KV head, tile index within the (b, h) rows
  int ce, len, tc, per_h;   // cold end, length, cold tiles, tiles of one head
};
template <bool MQ>
__device__ __forceinline__ void cursor_seq(const DecodeParams& p, Cursor& c) {
  const SeqTiles s = seq_tiles<MQ>(p, c.b);
  c.ce = s.ce;
  c.len = s.len;
  c.tc = s.tc;
  c.per_h = s.tc + s.th;
}
template <bool MQ>
__device__ __forceinline__ Cursor cursor_at(const DecodeParams& p, const long long* prefix, long long t) {
  const TileInfo ti = tile_info<MQ>(p, prefix, t);
  Cursor c;
  c.b = ti.b;
  c.h = ti.h;
  cursor_seq<MQ>(p, c);
  c.x = ti.hot ? c.tc + (ti.t_begin - c.ce) / kTile : ti.t_begin / kTile;
  return c;
}
// First token and token count of the tile a cursor points at.
__device__ __forceinline__ int cursor_t_begin(const Cursor& c) {
  return c.x >= c.tc ? c.ce + (c.x - c.tc) * kTile : c.x * kTile;
}
__device__ __forceinline__ int cursor_n_valid(const Cursor& c) {
  return min(kTile, (c.x >= c.tc ? c.len : c.ce) - cursor_t_begin(c));
}
template <bool MQ>
__device__ __forceinline__ void cursor_advance(const DecodeParams& p, Cursor& c, int n) {
  c.x += n;
  while (c.x >= c.per_h) {  // per_h is 0 for empty sequences
    c.x -= c.per_h;
    if (++c.h == p.hkv) {
      c.h = 0;
      if (++c.b >= p.batch) return;  // past the tile list: never staged
      cursor_seq<MQ>(p, c);
    }
  }
}

// 2^x with the hardware approximation (flushes results below 2^-126 to zero).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

// 16-byte cp.async at a shared and a global register base plus the same
// compile-time byte offset.
template <int OFF>
__device__ __forceinline__ void cp_async16_at(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0+%2], [%1+%2], 16;\n" ::"r"(dst), "l"(src), "n"(OFF));
}
__device__ __forceinline__ void cp_async16s(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst), "l"(src));
}
__device__ __forceinline__ void cp_async4s(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(dst), "l"(src));
}
// Copies `bytes` (a multiple of 16, at most 32 * 16 * N) from src to dst with the
// 32 lanes of a warp; full 512-byte rounds are unrolled with immediate offsets.
template <int BYTES>
__device__ __forceinline__ void copy_full(uint32_t dst, const uint8_t* src, int lane) {
  constexpr int kChunks = BYTES / 16, kRounds = kChunks / 32, kRest = kChunks % 32;
  const uint32_t d = dst + 16u * lane;
  const uint8_t* sp = src + 16 * lane;
  static_assert(kRounds <= 8, "tile larger than 8 rounds");
  if constexpr (kRounds > 0) cp_async16_at<0>(d, sp);
  if constexpr (kRounds > 1) cp_async16_at<512>(d, sp);
  if constexpr (kRounds > 2) cp_async16_at<1024>(d, sp);
  if constexpr (kRounds > 3) cp_async16_at<1536>(d, sp);
  if constexpr (kRounds > 4) cp_async16_at<2048>(d, sp);
  if constexpr (kRounds > 5) cp_async16_at<2560>(d, sp);
  if constexpr (kRounds > 6) cp_async16_at<3072>(d, sp);
  if constexpr (kRounds > 7) cp_async16_at<3584>(d, sp);
  if constexpr (kRest > 0)
    if (lane < kRest) cp_async16_at<kRounds * 512>(d, sp);
}

// 16-byte cp.async with distinct compile-time offsets at the shared and the
// global side.
template <int DOFF, int SOFF>
__device__ __forceinline__ void cp_async16_at2(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0+%2], [%1+%3], 16;\n" ::"r"(dst), "l"(src), "n"(DOFF), "n"(SOFF));
}
// Copies a full K tile of 16 rows of ROW bytes from contiguous global rows into
// shared rows of PITCH bytes: round r moves 512 bytes, rows 32 r / (ROW / 16) ..
template <int ROW, int PITCH>
__device__ __forceinline__ void copy_full_pitched(uint32_t dst, const uint8_t* src, int lane) {
  if constexpr (ROW == PITCH) {
    copy_full<kTile * ROW>(dst, src, lane);
  } else {
    constexpr int kRC = ROW / 16, kRounds = kTile * ROW / 512, kRowsPerRound = 32 / kRC;
    static_assert(32 % kRC == 0 && kRounds <= 8, "pitched copy layout");
    const uint32_t d = dst + static_cast<uint32_t>((lane / kRC) * PITCH + (lane % kRC) * 16);
    const uint8_t* sp = src + 16 * lane;
    constexpr int kD = kRowsPerRound * PITCH;
    if constexpr (kRounds > 0) cp_async16_at2<0 * kD, 0>(d, sp);
    if constexpr (kRounds > 1) cp_async16_at2<1 * kD, 512>(d, sp);
    if constexpr (kRounds > 2) cp_async16_at2<2 * kD, 1024>(d, sp);
    if constexpr (kRounds > 3) cp_async16_at2<3 * kD, 1536>(d, sp);
    if constexpr (kRounds > 4) cp_async16_at2<4 * kD, 2048>(d, sp);
    if constexpr (kRounds > 5) cp_async16_at2<5 * kD, 2560>(d, sp);
    if constexpr (kRounds > 6) cp_async16_at2<6 * kD, 3072>(d, sp);
    if constexpr (kRounds > 7) cp_async16_at2<7 * kD, 3584>(d, sp);
  }
}
// Shared offset of 16-byte chunk c of a K tile (chunks numbered row-major over
// the contiguous global rows).
template <int ROW, int PITCH>
__device__ __forceinline__ uint32_t k_chunk_dst(int c) {
  return static_cast<uint32_t>((c / (ROW / 16)) * PITCH + (c % (ROW / 16)) * 16);
}

// Block-table entries of the first and the last token of a tile.  The kernel
// loads them one issue ahead, so that their latency hides behind the
// consumption of a tile instead of stalling the copies that depend on them.
struct TileBlocks {
  int first, last;
};
__device__ __forceinline__ TileBlocks load_tile_blocks(const DecodeParams& p, int b, int t_begin, int n_valid) {
  const int32_t* row = p.map.table + static_cast<long long>(b) * p.map.max_blocks;
  TileBlocks tb;
  tb.first = __ldg(row + (t_begin >> p.map.shift));
  tb.last = __ldg(row + ((t_begin + n_valid - 1) >> p.map.shift));
  return tb;
}

// Paged staging of tile [t_begin, t_begin + n_valid) of (b, h) whose block-table
// entries are tb; returns the number of tokens the consumer may read (0 when
// the table maps the tile outside the pool, after flagging TQ_DEV_ERR_BLOCK).
// Cold tiles start at a multiple of the tile size and never straddle a block
// (blocks hold at least one tile); a hot tile (K only) that straddles a block
// boundary is copied token by token.  The common case (a full tile inside one
// valid block) takes one branch; the others share the second.
template <int KB, int VB, int VPITCH, int KPITCH>
__device__ __forceinline__ int stage_tile_paged(const DecodeParams& p, int h, bool hot, int t_begin, int n_valid,
                                             TileBlocks tb, uint32_t buf, int lane) {
  using C = Cfg<KB, VB>;
  constexpr int kVTileP = kTile * VPITCH;
  constexpr int kKP = KPITCH ? KPITCH : C::kKPitch, kKTileP = kTile * kKP;
  const int sh = p.map.shift;
  const unsigned nb = static_cast<unsigned>(p.map.num_blocks);
  const bool in_pool = static_cast<unsigned>(tb.first) < nb && static_cast<unsigned>(tb.last) < nb;
  const bool one_block = tb.first == tb.last && ((t_begin + n_valid - 1) >> sh) == (t_begin >> sh);
  const long long row0 = ((static_cast<long long>(tb.first) * p.map.hkv + h) << sh) + (t_begin & ((1 << sh) - 1));
  const uint8_t* kbase = C::kFp16K ? reinterpret_cast<const uint8_t*>(p.k_fp16)
                                   : reinterpret_cast<const uint8_t*>(p.k_words);
  const uint32_t vbuf = buf + kKTileP + C::kKNorm;
  long long rn = row0 + (lane & 15);  // norm row of the lane's token
  if (in_pool && one_block && n_valid == kTile) {
    copy_full_pitched<C::kKRow, kKP>(buf, kbase + row0 * C::kKRow, lane);
    if (!hot) copy_full_pitched<VB * 16, VPITCH>(vbuf, reinterpret_cast<const uint8_t*>(p.v_words) + row0 * (VB * 16), lane);
  } else {
    if (!in_pool) {  // outside the pool: nothing is staged, the tile is read as empty
      if (lane == 0 && p.status != nullptr) atomicOr(p.status, TQ_DEV_ERR_BLOCK);
      return 0;
    }
    const int blk0 = t_begin >> sh;
    constexpr int kPer = C::kKRow / 16;
    for (int c = lane; c < n_valid * kPer; c += 32) {  // K token by token (a partial or a straddling tile)
      const int t = t_begin + c / kPer;
      const long long r = p.map.in_block((t >> sh) == blk0 ? tb.first : tb.last, h, t);
      cp_async16s(buf + k_chunk_dst<C::kKRow, kKP>(c), kbase + r * C::kKRow + (c % kPer) * 16);
    }
    if (!hot) {  // cold tiles never straddle
      const uint8_t* vsrc = reinterpret_cast<const uint8_t*>(p.v_words) + row0 * (VB * 16);
      for (int c = lane; c < n_valid * (C::kVRow / 16); c += 32)
        cp_async16s(vbuf + k_chunk_dst<VB * 16, VPITCH>(c), vsrc + 16 * c);
    }
    const int tn = t_begin + min(lane & 15, n_valid - 1);
    rn = p.map.in_block((tn >> sh) == blk0 ? tb.first : tb.last, h, tn);
  }
  const int nl = lane & 15;
  const bool is_k = lane < 16;
  const bool want = nl < n_valid && (is_k ? !C::kFp16K : !hot);
  const float* nsrc = (is_k ? p.k_norms : p.v_norms) + rn;
  const uint32_t ndst = (is_k ? buf + kKTileP : vbuf + kVTileP) + 4u * nl;
  if (want) cp_async4s(ndst, nsrc);
  return n_valid;
}

// Stages tile [t_begin, t_begin + n_valid) of (b, h) into buf; returns the
// number of tokens the consumer may read.
// V rows are VPITCH bytes apart in the staged tile (VB * 16: contiguous).
// KPITCH: pitch of the staged K rows (0: the split kernel's Cfg::kKPitch).
template <int KB, int VB, bool PAGED, int VPITCH = VB * 16, int KPITCH = 0>
__device__ __forceinline__ int stage_tile(const DecodeParams& p, int b, int h, bool hot, int t_begin, int n_valid,
                                          TileBlocks tb, uint32_t buf, int lane) {
  using C = Cfg<KB, VB>;
  constexpr int kVTileP = kTile * VPITCH;
  constexpr int kKP = KPITCH ? KPITCH : C::kKPitch, kKTileP = kTile * kKP;
  if constexpr (PAGED) return stage_tile_paged<KB, VB, VPITCH, KPITCH>(p, h, hot, t_begin, n_valid, tb, buf, lane);
  const int64_t row0 = (static_cast<int64_t>(b) * p.hkv + h) * p.cap + t_begin;
  const uint8_t* ksrc = C::kFp16K ? reinterpret_cast<const uint8_t*>(p.k_fp16 + row0 * D)
                                  : reinterpret_cast<const uint8_t*>(p.k_words + row0 * (C::kKBits * 4));
  const uint8_t* vsrc = reinterpret_cast<const uint8_t*>(p.v_words + row0 * (VB * 4));
  const uint32_t vbuf = buf + kKTileP + C::kKNorm;
  if (n_valid == kTile) {
    copy_full_pitched<C::kKRow, kKP>(buf, ksrc, lane);
    if (!hot) copy_full_pitched<VB * 16, VPITCH>(vbuf, vsrc, lane);
  } else {
    for (int c = lane; c < n_valid * (C::kKRow / 16); c += 32)
      cp_async16s(buf + k_chunk_dst<C::kKRow, kKP>(c), ksrc + 16 * c);
    if (!hot)
      for (int c = lane; c < n_valid * (C::kVRow / 16); c += 32)
        cp_async16s(vbuf + k_chunk_dst<VB * 16, VPITCH>(c), vsrc + 16 * c);
  }
  // norms: lanes 0..15 the K norms, lanes 16..31 the V norms of the tile's tokens
  const int nl = lane & 15;
  const bool is_k = lane < 16;
  const bool want = nl < n_valid && (is_k ? !C::kFp16K : !hot);
  const float* nsrc = (is_k ? p.k_norms : p.v_norms) + row0 + nl;
  const uint32_t ndst = (is_k ? buf + kKTileP : vbuf + kVTileP) + 4u * nl;
  if (want) cp_async4s(ndst, nsrc);
  return n_valid;
}

// Split kernel.
template <int G, int KB, int VB, bool SPARSE, bool PAGED, bool MQ>
__global__ void __launch_bounds__(Cfg<KB, VB>::kThreads, 1) decode_split_kernel(const DecodeParams p) {
  using C = Cfg<KB, VB>;
  static_assert(!C::kInt8, "the int8 mode runs the tensor-core kernel");
  constexpr int S = C::kStages;
  constexpr int kRS = C::kRowShift;
  constexpr int GH = G >= 2 ? G / 2 : 1;  // heads whose scores a K-phase lane owns after the butterfly
  extern __shared__ __align__(16) uint8_t smem[];
  const uint32_t s0 = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  SmemLayout lay;
  lay.tab_lo = (s0 + C::kTab - 1) & ~static_cast<uint32_t>(C::kTab - 1);
  lay.tab_hi = lay.tab_lo + C::kTab;
  lay.cur = s0;
  auto ptr = [&](uint32_t addr) { return smem + (addr - s0); };
  const uint32_t tab = lay.tab_lo;
  float* qs = reinterpret_cast<float*>(ptr(lay.take(4 * D * 4)));
  float* comb = reinterpret_cast<float*>(ptr(lay.take(4 * D * 4)));
  float* wml = reinterpret_cast<float*>(ptr(lay.take(C::kWarps * 4 * 2 * 4)));
  int4* descs_all = reinterpret_cast<int4*>(ptr(lay.take(C::kWarps * 8 * 16)));
  long long* prefix = reinterpret_cast<long long*>(ptr(lay.take((kMaxDecodeBatch + 1) * 8)));
  long long* scan = reinterpret_cast<long long*>(ptr(lay.take(34 * 8)));
  uint8_t* wts_all = ptr(lay.take(C::kWarps * C::kWts));

  // the merge grid may be launched now; it waits for this grid's completion
  asm volatile("griddepcontrol.launch_dependents;\n");
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int s = lane >> 3, rr = lane & 7;   // K phase
  const int g = lane >> 4, r = lane & 15;   // V phase
  const uint32_t copy8 = static_cast<uint32_t>(r) * 8u;
  const uint32_t vbase = tab | copy8;
  const uint32_t kbase = tab | 128u | copy8;

  // pair tables: entry e = code_a | code_b << bits -> (c[code_a], c[code_b]), 16 copies per row
  if constexpr (!C::kFp16K && !C::kInt8) {
    constexpr int n = (1 << (2 * C::kKBits)) * kCopies;
    for (int i = tid; i < n; i += C::kThreads) {
      const int e = i / kCopies, c = i % kCopies;
      *reinterpret_cast<float2*>(ptr(tab + (e << kRS) + 128 + c * 8)) =
          make_float2(p.k_cent[e & ((1 << C::kKBits) - 1)], p.k_cent[e >> C::kKBits]);
    }
  }
  if constexpr (!C::kInt8) {
    constexpr int n = (1 << (2 * VB)) * kCopies;
    for (int i = tid; i < n; i += C::kThreads) {
      const int e = i / kCopies, c = i % kCopies;
      *reinterpret_cast<float2*>(ptr(tab + (e << kRS) + c * 8)) =
          make_float2(p.v_cent[e & ((1 << VB) - 1)], p.v_cent[e >> VB]);
    }
  }
  // launched as a programmatic dependent grid: the tables above use only the
  // parameters; the lengths and the cache may come from the preceding grids
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  if (blockIdx.x == 0 && tid == 0 && p.status != nullptr) {
    for (int b = 0; b < p.batch / p.nq; ++b) {
      const int len = p.seq_lens[b];
      if (len < 0 || len > p.cap || len > p.max_seq_len) {
        atomicOr(p.status, TQ_DEV_ERR_SEQ_LEN);
        break;
      }
    }
  }
  tile_prefix<C::kThreads, MQ>(p, prefix, scan);  // synchronizes
  const long long total = prefix[p.batch];
  const long long t0 = total * blockIdx.x / p.grid, t1 = total * (blockIdx.x + 1) / p.grid;
  if (t0 >= t1) return;

  // per-warp staging rings of S buffers, allocated around the table in warp order
  uint32_t ring = 0;
  for (int w = 0; w < C::kWarps; ++w) {
    const uint32_t a = lay.take(S * C::kBuf);
    if (w == warp) ring = a;
  }
  if (lay.cur > s0 + static_cast<uint32_t>(C::kSmem)) {  // cannot happen within the static budget
    if (tid == 0 && p.status != nullptr) atomicOr(p.status, TQ_DEV_ERR_LAYOUT);
    return;
  }
  uint8_t* const wring = ptr(ring);
  uint8_t* wts = wts_all + warp * C::kWts;
  int4* descs = descs_all + warp * 8;
  const int my_n = static_cast<int>((t1 - t0 - warp + C::kWarps - 1) / C::kWarps);  // tiles t0 + warp + C::kWarps j
  int j_issue = 0, j = 0;
  Cursor cur;
  TileBlocks tb{0, 0};  // paged: block-table entries of the tile the cursor points at
  if (my_n > 0) {
    cur = cursor_at<MQ>(p, prefix, t0 + warp);
    if constexpr (PAGED) tb = load_tile_blocks(p, cache_seq<MQ>(p, cur.b), cursor_t_begin(cur), cursor_n_valid(cur));
  }
  auto issue = [&]() {
    if (j_issue < my_n) {
      const bool hot = cur.x >= cur.tc;
      const int t_begin = cursor_t_begin(cur);
      const int n_valid = cursor_n_valid(cur);
      const int cb = cache_seq<MQ>(p, cur.b);
      const int staged = stage_tile<KB, VB, PAGED>(p, cb, cur.h, hot, t_begin, n_valid, tb,
                                                   ring + static_cast<uint32_t>((j_issue % S) * C::kBuf), lane);
      if (lane == 0) descs[j_issue % S] = make_int4(cb, cur.h | (hot << 16), t_begin, staged);
      cursor_advance<MQ>(p, cur, C::kWarps);
      if constexpr (PAGED)
        if (j_issue + 1 < my_n) tb = load_tile_blocks(p, cache_seq<MQ>(p, cur.b), cursor_t_begin(cur), cursor_n_valid(cur));
    }
    cp_async_commit();
    ++j_issue;
  };
#pragma unroll
  for (int st = 0; st < S - 1; ++st) issue();

  // The butterfly is free of selects: bit 2 of rr picks which of a step pair a lane
  // keeps, bit 1 which pair, bit 0 which heads (the lane's q' is stored in head order
  // jj ^ h0), so every lane computes its steps in (keep, send) order from its own bases.
  const int b2 = (rr >> 2) & 1, b1 = (rr >> 1) & 1;
  auto step_off = [&](int u) {
    return static_cast<uint32_t>((k_token<KB>(u, 0) - k_token<KB>(0, 0)) * C::kKRow);
  };
  const uint32_t k_off = k_lane_offset<KB>(s, rr);
  const uint32_t k_off_kk = k_off + step_off(2 * b1 + b2), k_off_ks = k_off + step_off(2 * b1 + 1 - b2);
  const uint32_t k_off_sk = k_off + step_off(2 * (1 - b1) + b2), k_off_ss = k_off + step_off(2 * (1 - b1) + 1 - b2);
  const uint32_t k_sh = KB == 3 ? (24u * rr) & 31u : 0u;
  const uint32_t v_off = v_lane_offset<VB>(g, r);
  const uint32_t v_sh = v_lane_shift<VB>(r);
  const uint32_t wts_s = static_cast<uint32_t>(__cvta_generic_to_shared(wts));
  // after the butterfly a K-phase lane holds token u_own of slot s, heads h0 .. h0 + GH - 1
  const int u_own = 2 * ((rr >> 1) & 1) + ((rr >> 2) & 1);
  const int tau_own = k_token<KB>(u_own, s);
  const int h0 = G >= 2 ? GH * (rr & 1) : 0;
  const bool owner = G >= 2 || (rr & 1) == 0;  // for G = 1 lanes rr and rr ^ 1 hold the same score
  constexpr bool sparse = SPARSE;
  float2 qr[G][8];
  uint32_t qa[8][2];  // MMA variants: the A fragments (fp16 query) of the 8 coordinate chunks
  const int gq = lane >> 2, tq = lane & 3;  // MMA: group (query head, token) and thread in the group
  int cur_b = -1, cur_h = -1;
  long long seg = t0;
  while (seg < t1) {
    const TileInfo si = tile_info<MQ>(p, prefix, seg);
    const long long seg_end = si.row_end < t1 ? si.row_end : t1;
    if (C::kMmaK && (si.b != cur_b || si.h != cur_h)) {
      // fp16 or int8 K: the raw fp16 query of head gq (exact) as MMA A fragments; chunk c
      // holds coordinates 16 c + 4 tq .. + 3, the order the B fragments read K in
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint2 v = make_uint2(0u, 0u);
        if (gq < G)
          v = *reinterpret_cast<const uint2*>(p.q + (static_cast<int64_t>(si.b) * p.hq + si.h * G + gq) * D +
                                              16 * c + 4 * tq);
        qa[c][0] = v.x;
        qa[c][1] = v.y;
      }
      cur_b = si.b;
      cur_h = si.h;
    }
    if (!C::kMmaK && (si.b != cur_b || si.h != cur_h)) {
      // rotated query of the G heads: (log2 e / d) H D q (packed K)
      constexpr bool kRotQ = true;
      __syncthreads();
      if (tid < D) {
        const bool neg = kRotQ && sign_negative(p.seed, p.layer, si.h, tid);
#pragma unroll
        for (int jj = 0; jj < G; ++jj) {
          const float x = half_bits_to_float(p.q[(static_cast<int64_t>(si.b) * p.hq + si.h * G + jj) * D + tid]);
          qs[jj * D + tid] = neg ? -x : x;
        }
      }
      __syncthreads();
      if constexpr (kRotQ) {
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
      const float qscale = kRotQ ? kLog2e / static_cast<float>(D) : kLog2e / kSqrtD;
#pragma unroll
      for (int jj = 0; jj < G; ++jj)
#pragma unroll
        for (int pr = 0; pr < 8; ++pr) {
          const int c = k_pair_coord<KB>(rr, pr), hh = jj ^ h0;
          qr[jj][pr] = make_float2(fmul(qs[hh * D + c], qscale), fmul(qs[hh * D + c + 1], qscale));
        }
      cur_b = si.b;
      cur_h = si.h;
    }

    // online-softmax state of this row: maxima of the lane's own heads (equal on
    // all lanes of the same parity), mass of the lane's own (token, head) pairs
    float m_own[GH], lsum[GH];
    float2 acc[G][4];
#pragma unroll
    for (int i = 0; i < GH; ++i) {
      m_own[i] = -INFINITY;
      lsum[i] = 0.0f;
    }
#pragma unroll
    for (int jj = 0; jj < G; ++jj)
#pragma unroll
      for (int k = 0; k < 4; ++k) acc[jj][k] = make_float2(0.0f, 0.0f);

    while (j < my_n && t0 + warp + static_cast<long long>(C::kWarps) * j < seg_end) {
      issue();
      cp_async_wait<S - 1>();
      __syncwarp();
      const int4 dsc = descs[j % S];
      const int tb_b = dsc.x, tb_h = dsc.y & 0xFFFF, n_valid = dsc.w, t_begin = dsc.z;  // tb_b: cache sequence
      const bool hot = (dsc.y >> 16) != 0;
      const uint8_t* tb = wring + (j % S) * C::kBuf;
      const uint32_t tbs = ring + static_cast<uint32_t>((j % S) * C::kBuf);  // shared address of the tile

      uint32_t stepmask = 0xFFu;  // V steps (2 tokens each) that carry a nonzero weight, warp-uniform
      if constexpr (C::kMmaK) {
        // ---- scores on the tensor cores: S = Q K^T, Q the G fp16 query heads (A rows,
        // zero above G), K the tile's 16 tokens (B columns, two blocks of 8); the
        // operands are exact in fp16 (fp16 K, or int8 codes) and the products are
        // summed in float32.  Lane (gq, tq) then holds head gq's raw scores of tokens
        // 2 tq, 2 tq + 1, 8 + 2 tq, 9 + 2 tq.
        float sraw[4];
        const uint32_t kb = tbs + static_cast<uint32_t>(gq * C::kKPitch + (C::kFp16K ? 8 : 4) * tq);
#pragma unroll
        for (int nb = 0; nb < 2; ++nb) {
          float d0 = 0.0f, d1 = 0.0f, d2 = 0.0f, d3 = 0.0f;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            uint32_t b0, b1;
            if constexpr (C::kFp16K) {
              const uint2 w = lds64u<0>(kb + static_cast<uint32_t>(nb * 8 * C::kKPitch + 32 * c));
              b0 = w.x;
              b1 = w.y;
            } else {
              const uint32_t w = lds32<0>(kb + static_cast<uint32_t>(nb * 8 * C::kKPitch + 16 * c)) ^ 0x80808080u;
              b0 = int8_half2<0>(w);
              b1 = int8_half2<2>(w);
            }
            mma_16816(d0, d1, d2, d3, qa[c][0], qa[c][1], b0, b1);
          }
          sraw[2 * nb] = d0;
          sraw[2 * nb + 1] = d1;
        }
        // ---- online softmax in that layout (base 2, lazily raised maximum)
        const bool head_ok = gq < G;
        const float* vnorm = reinterpret_cast<const float*>(tb + C::kKTile + C::kKNorm + C::kVTile);
        const int tk[4] = {2 * tq, 2 * tq + 1, 8 + 2 * tq, 9 + 2 * tq};
        constexpr float kQs = kLog2e / kSqrtD;
        float sj[4];
        bool bump = false;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float s = sraw[i];
          s = fmul(s, kQs);
          sj[i] = head_ok && tk[i] < n_valid ? s : -INFINITY;  // staged data of masked rows is stale
          bump |= sj[i] > fadd(m_own[0], kLazy);
        }
        if (__any_sync(0xffffffffu, bump)) {
          float tm = fmaxf(fmaxf(sj[0], sj[1]), fmaxf(sj[2], sj[3]));
          tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 1));
          tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 2));
          const float mn = fmaxf(m_own[0], tm);
          const float al = mn == -INFINITY ? 1.0f : ex2_approx(fsub(m_own[0], mn));  // 0 for the row's first tile
          lsum[0] = fmul(lsum[0], al);
          m_own[0] = mn;
#pragma unroll
          for (int jj = 0; jj < G; ++jj) {
            const float aj = __shfl_sync(0xffffffffu, al, 4 * jj);
#pragma unroll
            for (int k = 0; k < 4; ++k) acc[jj][k] = mul2(acc[jj][k], make_float2(aj, aj));
          }
        }
        float w4[4];
        uint32_t bits = 0u;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const bool live = sj[i] != -INFINITY;
          float pj = ex2_approx(fsub(sj[i], m_own[0]));
          pj = live ? pj : 0.0f;  // masked rows (also before any valid token)
          lsum[0] = fadd(lsum[0], pj);
          float w = fmul(pj, hot ? 1.0f : vnorm[tk[i]]);
          w = live ? w : 0.0f;  // the staged norm of a masked row is stale (possibly not a number)
          if (sparse && pj < p.sparse_tau) w = 0.0f;  // sparse V, as in the other layout
          w4[i] = w;
          bits |= (w != 0.0f ? 1u : 0u) << (tk[i] >> 1);
        }
        if (head_ok) {  // weights of token tk, head gq: row tk of 4 G bytes
          float* wf = reinterpret_cast<float*>(wts);
#pragma unroll
          for (int i = 0; i < 4; ++i) wf[tk[i] * G + gq] = w4[i];
        }
        if (sparse) stepmask = __reduce_or_sync(0xffffffffu, head_ok ? bits : 0u);
      } else {
        // ---- K phase: partial scores over the lane's 16 coordinates, 4 tokens per step
        float Ak[G], As[G];  // after butterfly stage A: the kept step pair and the sent one
        {
          auto k_step = [&](uint32_t kw, float* P) {
            constexpr int OFF = 0;
            float2 c[8];
            // packed K only: the fp16 and int8 modes take their scores on the tensor cores
            if constexpr (KB == 4) {
              const uint2 wv = lds64u<OFF>(kw);
              c[0] = lds64(pair_addr<4, 0, kRS>(wv.x, kbase));
              c[1] = lds64(pair_addr<4, 1, kRS>(wv.x, kbase));
              c[2] = lds64(pair_addr<4, 2, kRS>(wv.x, kbase));
              c[3] = lds64(pair_addr<4, 3, kRS>(wv.x, kbase));
              c[4] = lds64(pair_addr<4, 0, kRS>(wv.y, kbase));
              c[5] = lds64(pair_addr<4, 1, kRS>(wv.y, kbase));
              c[6] = lds64(pair_addr<4, 2, kRS>(wv.y, kbase));
              c[7] = lds64(pair_addr<4, 3, kRS>(wv.y, kbase));
            } else if constexpr (KB == 3) {
              const uint32_t wa = __funnelshift_r(lds32<OFF>(kw), lds32<OFF + 4>(kw), k_sh);
              const uint32_t wb = __funnelshift_r(lds32<OFF + 24>(kw), lds32<OFF + 28>(kw), k_sh);
              c[0] = lds64(pair_addr<3, 0, kRS>(wa, kbase));
              c[1] = lds64(pair_addr<3, 1, kRS>(wa, kbase));
              c[2] = lds64(pair_addr<3, 2, kRS>(wa, kbase));
              c[3] = lds64(pair_addr<3, 3, kRS>(wa, kbase));
              c[4] = lds64(pair_addr<3, 0, kRS>(wb, kbase));
              c[5] = lds64(pair_addr<3, 1, kRS>(wb, kbase));
              c[6] = lds64(pair_addr<3, 2, kRS>(wb, kbase));
              c[7] = lds64(pair_addr<3, 3, kRS>(wb, kbase));
            } else {
              const uint32_t wv = lds32<OFF>(kw);
              c[0] = lds64(pair_addr<2, 0, kRS>(wv, kbase));
              c[1] = lds64(pair_addr<2, 1, kRS>(wv, kbase));
              c[2] = lds64(pair_addr<2, 2, kRS>(wv, kbase));
              c[3] = lds64(pair_addr<2, 3, kRS>(wv, kbase));
              c[4] = lds64(pair_addr<2, 4, kRS>(wv, kbase));
              c[5] = lds64(pair_addr<2, 5, kRS>(wv, kbase));
              c[6] = lds64(pair_addr<2, 6, kRS>(wv, kbase));
              c[7] = lds64(pair_addr<2, 7, kRS>(wv, kbase));
            }
            // heads interleaved: consecutive packed FMAs are independent
            float2 pa[G];
#pragma unroll
            for (int jj = 0; jj < G; ++jj) pa[jj] = mul2(qr[jj][0], c[0]);
#pragma unroll
            for (int pr = 1; pr < 8; ++pr)
#pragma unroll
              for (int jj = 0; jj < G; ++jj) pa[jj] = fma2(qr[jj][pr], c[pr], pa[jj]);
#pragma unroll
            for (int jj = 0; jj < G; ++jj) P[jj] = fadd(pa[jj].x, pa[jj].y);
          };
          // stage A of the butterfly: the partner (rr ^ 4) sends what this lane keeps
          auto stage_a = [&](const float* Pk, const float* Ps, float* A) {
#pragma unroll
            for (int jj = 0; jj < G; ++jj) A[jj] = fadd(Pk[jj], __shfl_xor_sync(0xffffffffu, Ps[jj], 4));
          };
          {
            float Pk[G], Ps[G];
            k_step(tbs + k_off_kk, Pk);
            k_step(tbs + k_off_ks, Ps);
            stage_a(Pk, Ps, Ak);
          }
          {
            float Pk[G], Ps[G];
            k_step(tbs + k_off_sk, Pk);
            k_step(tbs + k_off_ss, Ps);
            stage_a(Pk, Ps, As);
          }
        }
        // ---- stages B (rr ^ 2, step pairs) and C (rr ^ 1, head pairs) of the butterfly
        float sc[GH];
        {
          float B[G];
#pragma unroll
          for (int jj = 0; jj < G; ++jj) B[jj] = fadd(Ak[jj], __shfl_xor_sync(0xffffffffu, As[jj], 2));
          if constexpr (G >= 2) {
#pragma unroll
            for (int i = 0; i < GH; ++i) sc[i] = fadd(B[i], __shfl_xor_sync(0xffffffffu, B[GH + i], 1));
          } else {
            sc[0] = fadd(B[0], __shfl_xor_sync(0xffffffffu, B[0], 1));
          }
        }
        // ---- online softmax over the tile (base 2; log2 e is folded into q').  The
        // running maximum of a head is raised only when a score exceeds it by more
        // than kLazy, so most tiles need neither the cross-lane maximum nor a rescale
        // (weights stay below 2^kLazy).
        const float nk = C::kFp16K ? 1.0f : reinterpret_cast<const float*>(tb + C::kKTile)[tau_own];
        const float nv = hot ? 1.0f : reinterpret_cast<const float*>(tb + C::kKTile + C::kKNorm + C::kVTile)[tau_own];
        const bool full = n_valid == kTile;  // warp-uniform
        const bool valid = tau_own < n_valid;
        float sj[GH];
        bool bump = false;
#pragma unroll
        for (int i = 0; i < GH; ++i) {
          sj[i] = fmul(sc[i], nk);
          if (!full) sj[i] = valid ? sj[i] : -INFINITY;  // staged data of masked rows is stale
          bump |= sj[i] > fadd(m_own[i], kLazy);
        }
        if (__any_sync(0xffffffffu, bump)) {
          float alpha[G];
#pragma unroll
          for (int i = 0; i < GH; ++i) {
            float tm = sj[i];
            tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 2));
            tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 4));
            tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 8));
            tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 16));
            const float mn = fmaxf(m_own[i], tm);  // finite: every staged tile has a valid token
            const float al = ex2_approx(fsub(m_own[i], mn));  // 0 for the first tile of the row
            lsum[i] = fmul(lsum[i], al);
            m_own[i] = mn;
            if constexpr (G >= 2) {
              const float oa = __shfl_xor_sync(0xffffffffu, al, 1);  // head (h0 + i) ^ GH
              const bool hi = (rr & 1) != 0;
              alpha[i] = hi ? oa : al;
              alpha[GH + i] = hi ? al : oa;
            } else {
              alpha[0] = al;
            }
          }
#pragma unroll
          for (int jj = 0; jj < G; ++jj)
#pragma unroll
            for (int k = 0; k < 4; ++k) acc[jj][k] = mul2(acc[jj][k], make_float2(alpha[jj], alpha[jj]));
        }
        float w_own[GH];
#pragma unroll
        for (int i = 0; i < GH; ++i) {
          float pj = ex2_approx(fsub(sj[i], m_own[i]));
          if (!full) pj = valid ? pj : 0.0f;  // masked rows (also before any valid token: -inf - -inf)
          lsum[i] = fadd(lsum[i], (G >= 2 || owner) ? pj : 0.0f);
          w_own[i] = fmul(pj, nv);
          if (!full) w_own[i] = valid ? w_own[i] : 0.0f;
          // sparse V: a weight below tau relative to the (lazily raised) running
          // maximum, hence below tau after normalization, contributes no V
          if (sparse && pj < p.sparse_tau) w_own[i] = 0.0f;
        }
        // V steps (2 tokens each) that carry a nonzero weight, warp-uniform
        if (sparse) {
          bool keep = false;
#pragma unroll
          for (int i = 0; i < GH; ++i) keep |= w_own[i] != 0.0f;
          stepmask = __reduce_or_sync(0xffffffffu, keep ? 1u << (tau_own >> 1) : 0u);
        }
        // weights of token tau_own, heads h0.. : row tau_own of 4 G bytes
        if constexpr (G == 4) {
          *reinterpret_cast<float2*>(wts + tau_own * 16 + h0 * 4) = make_float2(w_own[0], w_own[1]);
        } else if constexpr (G == 2) {
          *reinterpret_cast<float*>(wts + tau_own * 8 + h0 * 4) = w_own[0];
        } else {
          if (owner) *reinterpret_cast<float*>(wts + tau_own * 4) = w_own[0];
        }
      }
      __syncwarp();

      // ---- V phase: tokens 2u + g, 8 coordinates per lane
      const uint32_t wsb = wts_s + static_cast<uint32_t>(g * 4 * G);
      const uint32_t vw = tbs + static_cast<uint32_t>(C::kKTile + C::kKNorm) + v_off;
      auto load_w = [&](auto U_, float2* w2) {
        constexpr int U = decltype(U_)::value;
        if constexpr (G == 4) {  // one 16-byte broadcast per step, the (w, w) pairs built in registers
          const float4 a = lds128f<U * 32>(wsb);
          w2[0] = make_float2(a.x, a.x);
          w2[1] = make_float2(a.y, a.y);
          w2[2] = make_float2(a.z, a.z);
          w2[3] = make_float2(a.w, a.w);
        } else if constexpr (G == 2) {
          const float2 a = lds64f<U * 16>(wsb);
          w2[0] = make_float2(a.x, a.x);
          w2[G - 1] = make_float2(a.y, a.y);
        } else {
          const float a = __uint_as_float(lds32<U * 8>(wsb));
          w2[0] = make_float2(a, a);
        }
      };
      auto v_cold = [&](auto U_) {
        constexpr int U = decltype(U_)::value;
        constexpr int kVRec = VB * 16;
        float2 w2[G];
        load_w(U_, w2);
        {  // packed codes: one pair-table lookup per two coordinates
          uint32_t win;
          if constexpr (VB == 4) win = lds32<U * 2 * kVRec>(vw);
          else if constexpr (VB == 2) win = lds32<U * 2 * kVRec>(vw) >> v_sh;
          else win = __funnelshift_r(lds32<U * 2 * kVRec>(vw), lds32<U * 2 * kVRec + 4>(vw), v_sh);
          const float2 c0 = lds64(pair_addr<VB, 0, kRS>(win, vbase));
          const float2 c1 = lds64(pair_addr<VB, 1, kRS>(win, vbase));
          const float2 c2 = lds64(pair_addr<VB, 2, kRS>(win, vbase));
          const float2 c3 = lds64(pair_addr<VB, 3, kRS>(win, vbase));
#pragma unroll
          for (int jj = 0; jj < G; ++jj) {
            acc[jj][0] = fma2(w2[jj], c0, acc[jj][0]);
            acc[jj][1] = fma2(w2[jj], c1, acc[jj][1]);
            acc[jj][2] = fma2(w2[jj], c2, acc[jj][2]);
            acc[jj][3] = fma2(w2[jj], c3, acc[jj][3]);
          }
        }
      };
      auto v_hot = [&](auto U_) {
        constexpr int U = decltype(U_)::value;
        const int tau = 2 * U + g;
        float2 w2[G];
        load_w(U_, w2);
        if (tau < n_valid) {
          const int pos = t_begin + tau;
          const uint4 a0 = reinterpret_cast<const uint4*>(
              p.v_ring + ((static_cast<int64_t>(tb_b) * p.hkv + tb_h) * p.hot + pos % p.hot) * D)[r];
          const uint32_t wv[4] = {a0.x, a0.y, a0.z, a0.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float2 vf = half2_bits_to_float2(wv[k]);
#pragma unroll
            for (int jj = 0; jj < G; ++jj) acc[jj][k] = fma2(w2[jj], vf, acc[jj][k]);
          }
        }
      };
      if (!hot && stepmask == 0xFFu) {
        v_cold(std::integral_constant<int, 0>{});
        v_cold(std::integral_constant<int, 1>{});
        v_cold(std::integral_constant<int, 2>{});
        v_cold(std::integral_constant<int, 3>{});
        v_cold(std::integral_constant<int, 4>{});
        v_cold(std::integral_constant<int, 5>{});
        v_cold(std::integral_constant<int, 6>{});
        v_cold(std::integral_constant<int, 7>{});
      } else if (!hot) {  // sparse V: only the steps with a nonzero weight
        if (stepmask & 0x01u) v_cold(std::integral_constant<int, 0>{});
        if (stepmask & 0x02u) v_cold(std::integral_constant<int, 1>{});
        if (stepmask & 0x04u) v_cold(std::integral_constant<int, 2>{});
        if (stepmask & 0x08u) v_cold(std::integral_constant<int, 3>{});
        if (stepmask & 0x10u) v_cold(std::integral_constant<int, 4>{});
        if (stepmask & 0x20u) v_cold(std::integral_constant<int, 5>{});
        if (stepmask & 0x40u) v_cold(std::integral_constant<int, 6>{});
        if (stepmask & 0x80u) v_cold(std::integral_constant<int, 7>{});
      } else {
        v_hot(std::integral_constant<int, 0>{});
        v_hot(std::integral_constant<int, 1>{});
        v_hot(std::integral_constant<int, 2>{});
        v_hot(std::integral_constant<int, 3>{});
        v_hot(std::integral_constant<int, 4>{});
        v_hot(std::integral_constant<int, 5>{});
        v_hot(std::integral_constant<int, 6>{});
        v_hot(std::integral_constant<int, 7>{});
      }
      __syncwarp();
      ++j;
    }

    // ---- leave the row: lanes -> warp -> CTA, one partial per (CTA, row)
    for (int i = tid; i < G * D; i += C::kThreads) comb[i] = 0.0f;
    float mw[G];  // warp maxima of all heads
    if constexpr (C::kMmaK) {  // head jj's maximum is on lanes 4 jj .. 4 jj + 3
#pragma unroll
      for (int jj = 0; jj < G; ++jj) mw[jj] = __shfl_sync(0xffffffffu, m_own[0], 4 * jj);
    } else if constexpr (G >= 2) {
      const bool hi = (rr & 1) != 0;
#pragma unroll
      for (int i = 0; i < GH; ++i) {
        const float om = __shfl_xor_sync(0xffffffffu, m_own[i], 1);
        mw[i] = hi ? om : m_own[i];
        mw[GH + i] = hi ? m_own[i] : om;
      }
    } else {
      mw[0] = m_own[0];
    }
#pragma unroll
    for (int jj = 0; jj < G; ++jj)
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float2 a = acc[jj][k];
        a.x = fadd(a.x, __shfl_xor_sync(0xffffffffu, a.x, 16));
        a.y = fadd(a.y, __shfl_xor_sync(0xffffffffu, a.y, 16));
        acc[jj][k] = a;
      }
    {
      float lw[G];
      if constexpr (C::kMmaK) {  // head jj's mass: the sum over its 4 lanes
        float l4 = fadd(lsum[0], __shfl_xor_sync(0xffffffffu, lsum[0], 1));
        l4 = fadd(l4, __shfl_xor_sync(0xffffffffu, l4, 2));
#pragma unroll
        for (int jj = 0; jj < G; ++jj) lw[jj] = __shfl_sync(0xffffffffu, l4, 4 * jj);
      } else {
#pragma unroll
        for (int jj = 0; jj < G; ++jj) lw[jj] = 0.0f;
#pragma unroll
        for (int i = 0; i < GH; ++i)
#pragma unroll
          for (int jj = 0; jj < G; ++jj)
            if (jj == h0 + i) lw[jj] = lsum[i];
#pragma unroll
        for (int jj = 0; jj < G; ++jj)
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) lw[jj] = fadd(lw[jj], __shfl_xor_sync(0xffffffffu, lw[jj], o));
      }
#pragma unroll
      for (int jj = 0; jj < G; ++jj) {
        if (lane == 0) {
          wml[(warp * 4 + jj) * 2] = mw[jj];
          wml[(warp * 4 + jj) * 2 + 1] = lw[jj];
        }
      }
    }
    __syncthreads();
    // warps add into comb one after another in warp order, so that the result
    // does not depend on timing (decode is bit-reproducible)
    float sc2[G];
#pragma unroll
    for (int jj = 0; jj < G; ++jj) {
      float mm = -INFINITY;
#pragma unroll
      for (int w = 0; w < C::kWarps; ++w) mm = fmaxf(mm, wml[(w * 4 + jj) * 2]);
      sc2[jj] = mw[jj] == -INFINITY ? 0.0f : exp2f(mw[jj] - mm);
    }
    for (int w = 0; w < C::kWarps; ++w) {
      if (warp == w && g == 0) {
#pragma unroll
        for (int jj = 0; jj < G; ++jj) {
          if (mw[jj] == -INFINITY) continue;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            float* c2 = comb + jj * D + 8 * r + 2 * k;
            c2[0] = fadd(c2[0], fmul(acc[jj][k].x, sc2[jj]));
            c2[1] = fadd(c2[1], fmul(acc[jj][k].y, sc2[jj]));
          }
        }
      }
      __syncthreads();
    }
    const long long slot = static_cast<long long>(blockIdx.x) + si.row;
    for (int i = tid; i < G * D; i += C::kThreads) p.ws_acc[slot * G * D + i] = comb[i];
    if (tid < G) {
      float mm = -INFINITY, ll = 0.0f;
#pragma unroll
      for (int w = 0; w < C::kWarps; ++w) mm = fmaxf(mm, wml[(w * 4 + tid) * 2]);
#pragma unroll
      for (int w = 0; w < C::kWarps; ++w) {
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

// Output of one (b, query head) row from its merged sums, by a full warp (lane
// l holds coordinates 4 l .. 4 l + 3): the cold sum y is rotated back, D_h H y /
// sqrt(d) (sign flips neg4, a Hadamard transform over index bits 0..1 in
// registers and 2..6 across lanes; not in the int8 mode, whose V is summed
// unrotated), the hot sum hv is added and the softmax mass l divided out (a row
// that read no token gives zeros).
__device__ __forceinline__ void merge_finish(float (&y)[4], const float (&hv)[4], float l, unsigned neg4, bool rotated,
                                             float* out_row, int lane) {
  float4* out = reinterpret_cast<float4*>(out_row);
  if (!rotated) {
#pragma unroll
    for (int i = 0; i < 4; ++i) y[i] = l > 0.0f ? fadd(y[i], hv[i]) / l : 0.0f;
    out[lane] = make_float4(y[0], y[1], y[2], y[3]);
    return;
  }
  {
    float a0 = fadd(y[0], y[1]), a1 = fsub(y[0], y[1]), a2 = fadd(y[2], y[3]), a3 = fsub(y[2], y[3]);  // bit 0
    y[0] = fadd(a0, a2);  // bit 1
    y[2] = fsub(a0, a2);
    y[1] = fadd(a1, a3);
    y[3] = fsub(a1, a3);
  }
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {  // bits 2..6
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float o = __shfl_xor_sync(0xffffffffu, y[i], m);
      y[i] = upper ? fsub(o, y[i]) : fadd(y[i], o);
    }
  }
  float r[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float v = fmul(y[i], 1.0f / kSqrtD);
    if ((neg4 >> i) & 1u) v = -v;
    r[i] = l > 0.0f ? fadd(v, hv[i]) / l : 0.0f;
  }
  out[lane] = make_float4(r[0], r[1], r[2], r[3]);
}

// CTA of the split kernel that processes tile t (the last one whose range starts
// at or before t): floor(((t + 1) grid - 1) / total), a value below grid.  A float
// estimate of the quotient is off by at most one (its relative error is a few
// 2^-24 and the quotient is below 2^10); exact 64-bit products correct it, so no
// 64-bit division is needed.
__device__ __forceinline__ int cta_of(long long t, long long total, int grid) {
  const long long num = (t + 1) * grid - 1;
  int c = static_cast<int>(static_cast<float>(num) * (1.0f / static_cast<float>(total)));
  c = c < 0 ? 0 : (c > grid - 1 ? grid - 1 : c);
  if (static_cast<long long>(c) * total > num) --c;
  if (static_cast<long long>(c + 1) * total <= num) ++c;
  return c;
}
// Whether CTA c of the split kernel has a non-empty range: always when there are
// at least as many tiles as CTAs (then total / grid >= 1 separates the starts).
__device__ __forceinline__ bool cta_live(int c, long long total, int grid) {
  if (total >= grid) return true;
  const int t32 = static_cast<int>(total);
  return t32 * c / grid != t32 * (c + 1) / grid;
}

template <int G, int KB, int VB, bool SPARSE, bool PAGED, bool MQ>
tq_status launch_split(const DecodeParams& p, cudaStream_t stream) {
  using C = Cfg<KB, VB>;
  auto kern = decode_split_kernel<G, KB, VB, SPARSE, PAGED, MQ>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem) != cudaSuccess)
    return TQ_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.grid);
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see griddepcontrol.wait
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, p) != cudaSuccess) return TQ_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

}  // namespace
}  // namespace tq
