// Split-K decode over the packed cache: the pieces the decode kernel
// (tq_decode_mma.cuh) and the merge kernel (tq_decode.cu) share — parameters,
// work list, tile staging and the output of a merged row.
//
// Work list.  Every (sequence b, KV head h) has a cold row (the packed
// positions [0, L - min(W, L))) and, with a hot window, a hot row (the newest
// min(W, L) positions, whose V is read from the fp16 ring).  Rows are cut into
// 16-token tiles and listed in (b, h, cold/hot) order; the list is split into
// one contiguous range per CTA, equal in tiles plus a price for every row part
// a CTA starts (tq_split_plan.h), so that every SM gets the same work whatever
// the lengths are.  For attention of nq query tokens per
// sequence (MQ variants) every query token is a sequence of the list of its
// own, whose length is its causal prefix; its tiles are read from the cache
// rows of the sequence it belongs to.
//
// Partials.  When a CTA leaves a row it combines its warps and writes one
// partial (acc, max, sum) to workspace slot (CTA index + row index): these
// slots are distinct for all (CTA, row) pairs because both indices only grow
// along the tile list.
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
#include "tq_split_plan.h"

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
  SplitPrice price;  // segment start prices of the weighted split (tq_split_plan.h)
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

// Staging layout of one 16-token tile: K | K norms | V | V norms (the pitches
// of the tensor-core kernel may override the K and V row pitches).
template <int KB, int VB>
struct Cfg {
  static constexpr bool kFp16K = KB == 16;
  static constexpr bool kInt8 = KB == 8;               // int8 mode: K and V int8 codes with absmax scales
  static_assert(!kInt8 || VB == 8, "the int8 mode has int8 K and V");
  static constexpr int kKBits = kFp16K ? 2 : KB;       // placeholder width when K is fp16
  static constexpr int kKRow = kFp16K ? 256 : KB * 16;  // bytes of one K token
  static constexpr int kVRow = VB * 16;
  // int8 K rows padded (144 = 128 + 16 bytes) so that the loads of 8 tokens by 4
  // lanes fall in distinct banks
  static constexpr int kKPitch = kFp16K ? kKRow + 32 : kInt8 ? kKRow + 16 : kKRow;
  static constexpr int kKTile = kTile * kKPitch;
  static constexpr int kKNorm = kFp16K ? 0 : kTile * 4;
  static constexpr int kVTile = kTile * kVRow;
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
  } else if constexpr (32 % (ROW / 16) != 0) {  // e.g. 48-byte rows: chunk by chunk
    for (int c = lane; c < kTile * (ROW / 16); c += 32)
      cp_async16s(dst + static_cast<uint32_t>((c / (ROW / 16)) * PITCH + (c % (ROW / 16)) * 16), src + 16 * c);
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
// KPITCH: pitch of the staged K rows (0: Cfg::kKPitch).
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

}  // namespace
}  // namespace tq
