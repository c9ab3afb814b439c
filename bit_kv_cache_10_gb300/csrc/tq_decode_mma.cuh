// Split-K decode kernel with the scores and the V sums on the tensor cores, for
// every mode: packed K of 2, 3 or 4 bits or fp16 K, with packed V of 2, 3 or 4
// bits (narrower codes spread to nibbles), and the int8 mode.  The work list,
// the tile staging, the partial slots and the merge output are in
// tq_decode_split.cuh; the persistent variant covers one contiguous tile range
// per CTA (the weighted split of tq_split_plan.h), the cluster variant (CL) one
// (b, h) row per 8-CTA cluster.
//
// Exact operands from lookups.  A float32 centroid c is the sum of two fp16
// numbers, hi = RN16(c) and lo = RN16(c - hi), which together carry 22
// significant bits; the same holds for the rotated query and for the softmax
// weights.  Products of fp16 numbers are exact in float32, so
//   sum_i q_i c_i = sum_i (q_hi + q_lo)_i (c_hi + c_lo)_i
// is computed by mma.sync (f16 operands, float32 accumulation) to about 2^-21
// relative, against the 2^-11 of a plain fp16 operand.  Centroids are
// tabulated times 2^10 so that both halves are normal fp16 numbers.
//
// Tables.  Row e (256 bytes) of a shared table holds, for the code pair
// e = code_a | code_b << bits, the pair (hi_a, hi_b) of fp16 halves 32 times
// over in bytes [0, 128) and (lo_a, lo_b) 32 times over in bytes [128, 256):
// lane l reads copy l, so the data-dependent 32-bit loads of a warp fall in 32
// distinct banks, and the lo half is the same address plus 128.  Each load
// returns one A-fragment register, so the fragments need no register moves.
// The V table (256 rows) and the K table (2^(2 bits) rows) start at 64 KB
// boundaries, so that an entry address is (e << 8) | (table + 4 l) (K: (e << 7) | ...).
//
// Scores (tokens as M, coordinates as K, 8 columns as N = the G query heads'
// rotated query in hi and in lo halves).  An MMA covers 8 tokens: row g holds
// the hi halves of token g's centroids and row g + 8 the lo halves, so that one
// 64-bit load of a K entry (hi pair, lo pair) fills an aligned register pair of
// the A fragment; row g plus row g + 8 is the token's dot product.  Lane (g, t)
// holds coordinates 32 t .. 32 t + 31; chunk c of the MMA K dimension takes
// coordinates 32 t + 4 c .. + 3 of every lane t.  Column h plus column h + 4
// is head h.  The K table keeps (hi pair, lo pair) entries 16 times over (one
// copy per lane of a half-warp, rows of 128 bytes).
//
// Softmax.  Lane (g, t) then owns token g + 8 (t >> 1) for heads 2 (t & 1) and
// 2 (t & 1) + 1.  The V weight of a token is w = 2^(s - m) n_V; the running
// maximum m of a head is raised lazily (only when a score exceeds it by 2^8) against
// s + e_V + 1, e_V the binary exponent of n_V, so every weight stays below 2^8
// and its fp16 hi and lo halves are exact.  The mass sums 2^(s - m) alone.
//
// V (coordinates as M, tokens as K, N = the weights in hi and lo halves).  Lane
// (g, t) holds coordinates 16 g .. 16 g + 15 (M block b: rows 16 g + 2 b and
// 16 g + 2 b + 1) and tokens 2 t, 2 t + 1, 2 t + 8, 2 t + 9; an A register
// pairs the codes of two tokens at one coordinate, built from two code words
// by nibble interleaving.  Hot rows read the fp16 ring (exact in fp16: one MMA
// per block).  The cold sum is tabulated times 2^10, removed at the row exit.
#pragma once

#include <cuda_fp16.h>

#include "tq_decode_split.cuh"
#include "tq_launch.cuh"

namespace tq {
namespace {

constexpr float kCentScale = 1024.0f;       // centroids are tabulated times 2^10
constexpr float kCentUnscale = 1.0f / 1024.0f;

constexpr int kClusterCtas = 8;  // CTAs of a (b, h) row in the cluster variant (the portable cluster size)

template <int KB, bool CL = false, int VB = 4>
struct MmaCfg {
  static constexpr bool kF16K = KB == 16;    // fp16 K (asym): K tiles read with ldmatrix, no K table
  static constexpr bool kI8 = KB == 8;       // int8 mode: int8 K and V codes, exact in fp16, no tables
  static constexpr int kVB = kI8 ? 8 : VB;  // V of 2 or 3 bits: codes expanded to nibbles, 4-bit path
  using Stage = Cfg<KB, kVB>;                // K | K norms | V | V norms, with V rows padded:
  // fp16 K rows 256 + 16 bytes apart (the 8 rows of an ldmatrix phase hit distinct banks)
  static constexpr int kKPitch = kF16K ? 272 : Stage::kKPitch;
  static constexpr int kKTile = kTile * kKPitch;
  static constexpr int kKNorm = Stage::kKNorm;
  // 64-byte records 80 bytes apart (conflict-free V code loads; 32- and 48-byte records
  // use the same pitch); int8: 128-byte records 144 apart
  static constexpr int kVPitch = kI8 ? 144 : 80;
  static constexpr int kVTile = kTile * kVPitch;
  static constexpr int kBuf = kKTile + kKNorm + kVTile + kTile * 4;
  // fp16 K tiles are 2.7 times larger: 10 warps keep two stages each within the budget
  static constexpr int kWarps = kF16K ? 10 : 12;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kTabAlign = kI8 ? 1024 : 65536;
  static constexpr int kKTabRows = (kF16K || kI8) ? 0 : 1 << (2 * ((kF16K || kI8) ? 2 : KB));
  static constexpr int kVTabRows = kI8 ? 0 : 256;
  // V table (256-byte rows) | K table (128-byte rows); int8: a 1 KB placeholder
  static constexpr int kTab = (kI8 ? 1024 : 65536) + kKTabRows * 128;
  static constexpr int kW16 = 2 * 4 * kTile * 2;  // per warp: fp16 weights [hi/lo][head][token]
  // cluster variant: the CTA's cold and hot partials, acc [part][4][D] then (m, l) [part][4]
  static constexpr int kPart = CL ? 2 * 4 * (D + 2) * 4 : 0;
  static constexpr int kSmall = kWarps * kW16 + 4 * 132 * 4 /* rotated query */ + kWarps * 4 * 136 * 4 /* combine */ +
                                kWarps * 4 * 2 * 4 /* warp (m, l) */ + kWarps * 8 * 16 /* tile descriptors */ +
                                (kMaxDecodeBatch + 1) * 8 + 34 * 8 + kPart;
  static constexpr int kWorst(int stages) { return kTab + kSmall + (kWarps + 1) * stages * kBuf + 1024; }
  // the aligned table can leave a gap of up to kTabAlign - 1024 bytes before it, filled by the other buffers
  static constexpr int kStages = kWorst(6) <= kSmemBudget ? 6 : kWorst(4) <= kSmemBudget ? 4 : kWorst(3) <= kSmemBudget ? 3 : 2;
  static constexpr int kSmem = (kWorst(kStages) + 1023) / 1024 * 1024;
  static_assert(kWorst(kStages) <= kSmemBudget, "shared memory budget");
};

// D += A B, m16n8k16, f16 operands, float32 accumulators (all four A registers).
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
               "{%0, %1, %2, %3};\n"
               : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
               : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// fp16 hi and lo halves of x (x = hi + lo to 22 significant bits).
__device__ __forceinline__ void split_f16(float x, uint16_t& hi, uint16_t& lo) {
  const __half h = __float2half_rn(x);
  hi = __half_as_ushort(h);
  lo = __half_as_ushort(__float2half_rn(fsub(x, __half2float(h))));
}
// Pair of fp16 halves as one register (a in the low half).
__device__ __forceinline__ uint32_t pack16(uint16_t a, uint16_t b) {
  return static_cast<uint32_t>(a) | (static_cast<uint32_t>(b) << 16);
}
// Table entry of a code pair: (hi_a, hi_b) in .x, (lo_a, lo_b) in .y (stored 128 bytes apart).
__device__ __forceinline__ uint2 pair_entry(float ca, float cb) {
  uint16_t ha, la, hb, lb;
  split_f16(fmul(ca, kCentScale), ha, la);
  split_f16(fmul(cb, kCentScale), hb, lb);
  return make_uint2(pack16(ha, hb), pack16(la, lb));
}

// Four 8x8 fp16 matrices from shared memory in the mma.sync A-fragment layout.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& a0, uint32_t& a1, uint32_t& a2, uint32_t& a3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];\n"
               : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
               : "r"(addr));
}

__device__ __forceinline__ uint2 lds64a(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];\n" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

// hi half (.x) and lo half (.y) of the table entry at addr.
__device__ __forceinline__ uint2 lds_entry(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.u32 %0, [%1];\n" : "=r"(v.x) : "r"(addr));
  asm volatile("ld.shared.u32 %0, [%1+128];\n" : "=r"(v.y) : "r"(addr));
  return v;
}

// Shared address of the K table entry of code pair J (bits 2 KB J .. of the
// lane's window of 32 coordinates); kbase = K table + 8 (lane mod 16), rows of 128 bytes.
template <int KB, int J>
__device__ __forceinline__ uint32_t k_pair_addr(const uint32_t* win, uint32_t kbase) {
  if constexpr (KB == 4) {
    return (__byte_perm(win[J / 4], 0u, 0x4440 | (J % 4)) << 7) | kbase;  // byte J of the window
  } else {
    constexpr int kOff = 2 * KB * J, kW = kOff / 32, kBit = kOff % 32;
    uint32_t x;
    if constexpr (kBit + 2 * KB > 32) x = __funnelshift_r(win[kW], win[kW + 1], kBit - 7);
    else if constexpr (kBit >= 7) x = win[kW] >> (kBit - 7);
    else x = win[kW] << (7 - kBit);
    return (x & (((1u << (2 * KB)) - 1u) << 7)) | kbase;
  }
}

// Address of the V table entry whose index is byte K of x; vbase = V table + 4 lane.
template <int K>
__device__ __forceinline__ uint32_t v_pair_addr(uint32_t x, uint32_t vbase) {
  return __byte_perm(x, vbase, 0x7604 | (K << 4));
}

// Codes of 8 coordinates (3 or 2 bits each, LSB-first) spread to one nibble each.
__device__ __forceinline__ uint32_t spread3(uint32_t v) {  // 24 bits -> 8 nibbles
  v = (v & 0x00000FFFu) | ((v & 0x00FFF000u) << 4);       // 12-bit groups at bits 0, 16
  v = (v & 0x003F003Fu) | ((v & 0x0FC00FC0u) << 2);       // 6-bit groups at bytes 0..3
  return (v & 0x07070707u) | ((v & 0x38383838u) << 1);    // 3-bit codes at nibbles
}
__device__ __forceinline__ uint32_t spread2(uint32_t v) {  // 16 bits -> 8 nibbles
  v = (v & 0x000000FFu) | ((v & 0x0000FF00u) << 8);       // bytes at bits 0, 16
  v = (v & 0x000F000Fu) | ((v & 0x00F000F0u) << 4);       // nibbles at bytes 0..3
  return (v & 0x03030303u) | ((v & 0x0C0C0C0Cu) << 2);    // 2-bit codes at nibbles
}
// The lane's 16 V codes of one token (coordinates 16 g .. 16 g + 15, at shared
// address `addr`) as two words of nibbles, codes 0..7 and 8..15: the 4-bit record
// as it is, narrower codes spread.  A 3-bit window (6 bytes at 6 g) starts on a
// 4-byte boundary or 2 bytes after one.
template <int VB>
__device__ __forceinline__ uint2 v_nibbles(uint32_t addr) {
  if constexpr (VB == 4) {
    uint2 v;
    asm("ld.shared.v2.u32 {%0, %1}, [%2];\n" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
  } else if constexpr (VB == 2) {
    uint32_t w;
    asm("ld.shared.u32 %0, [%1];\n" : "=r"(w) : "r"(addr));
    return make_uint2(spread2(w & 0xFFFFu), spread2(w >> 16));
  } else {
    const uint32_t base = addr & ~3u, sh = (addr & 3u) * 8u;
    uint32_t w0, w1;
    asm("ld.shared.u32 %0, [%1];\n" : "=r"(w0) : "r"(base));
    asm("ld.shared.u32 %0, [%1+4];\n" : "=r"(w1) : "r"(base));
    const uint32_t x = __funnelshift_r(w0, w1, sh), y = w1 >> sh;  // window bits 0..31 and 32..47
    return make_uint2(spread3(x & 0x00FFFFFFu), spread3((x >> 24) | (y << 8)));
  }
}

// Nibble interleave of two code words of tokens a and b: byte k of lo_pairs is
// code_a | code_b << 4 of the even coordinate of byte k, hi_pairs the odd one.
__device__ __forceinline__ void interleave(uint32_t wa, uint32_t wb, uint32_t& lo_pairs, uint32_t& hi_pairs) {
  lo_pairs = (wa & 0x0F0F0F0Fu) | ((wb << 4) & 0xF0F0F0F0u);
  hi_pairs = ((wa >> 4) & 0x0F0F0F0Fu) | (wb & 0xF0F0F0F0u);
}

// Padded shared layouts: the rotated query with one word after every 32
// coordinates (the lanes' 32-coordinate windows of the four heads fall in
// distinct banks), the row combine with one word after every 16 coordinates.
__device__ __forceinline__ int qs_at(int h, int i) { return h * 132 + i + (i >> 5); }

// Thread-block cluster: barrier of every thread of the cluster (release /
// acquire: shared-memory writes before it are seen by the cluster's reads after
// it), the address of the same shared variable in CTA `rank`, and loads from it.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}
__device__ __forceinline__ uint32_t map_cluster(uint32_t addr, int rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ float2 ld_cluster_f2(uint32_t addr) {
  float2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];\n" : "=f"(v.x), "=f"(v.y) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ float4 ld_cluster_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];\n"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ int comb_at(int h, int i) { return h * 136 + i + (i >> 4); }

template <int G, int KB, bool SPARSE, bool PAGED, bool MQ, bool CL = false, int VB = 4>
__global__ void __launch_bounds__(MmaCfg<KB, CL, VB>::kThreads, 1) decode_mma_kernel(const DecodeParams p) {
  using M = MmaCfg<KB, CL, VB>;
  using C = Cfg<KB, M::kVB>;
  constexpr int S = M::kStages;
  constexpr int NW = M::kWarps;
  extern __shared__ __align__(16) uint8_t smem[];
  const uint32_t s0 = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  SmemLayout lay;
  lay.tab_lo = (s0 + M::kTabAlign - 1) & ~static_cast<uint32_t>(M::kTabAlign - 1);
  lay.tab_hi = lay.tab_lo + M::kTab;
  lay.cur = s0;
  auto ptr = [&](uint32_t addr) { return smem + (addr - s0); };
  const uint32_t tab = lay.tab_lo;
  float* qs = reinterpret_cast<float*>(ptr(lay.take(4 * 132 * 4)));
  float* comb = reinterpret_cast<float*>(ptr(lay.take(NW * 4 * 136 * 4)));  // one row sum per warp
  float* wml = reinterpret_cast<float*>(ptr(lay.take(NW * 4 * 2 * 4)));
  int4* descs_all = reinterpret_cast<int4*>(ptr(lay.take(NW * 8 * 16)));
  long long* prefix = reinterpret_cast<long long*>(ptr(lay.take((kMaxDecodeBatch + 1) * 8)));
  long long* scan = reinterpret_cast<long long*>(ptr(lay.take(34 * 8)));
  const uint32_t w16_all = lay.take(NW * M::kW16);
  float* cpart = nullptr;
  if constexpr (CL) cpart = reinterpret_cast<float*>(ptr(lay.take(M::kPart)));

  asm volatile("griddepcontrol.launch_dependents;\n");
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const uint32_t vbase = tab + 4u * lane;
  const uint32_t kbase = tab + 65536u + 8u * (lane & 15);

  // tables (from the parameters only): each lane computes one distinct entry
  // and writes its copies in an order rotated by the lane, so that the 32 stores
  // of a warp fall in 32 distinct banks
  {
    constexpr int kK = M::kKTabRows, kV = M::kVTabRows;
    for (int e = tid; e < kV + kK; e += M::kThreads) {
      if (e < kV) {
        const uint2 v = pair_entry(p.v_cent[e & 15], p.v_cent[e >> 4]);
        if constexpr (CL) {  // latency first: 16-byte stores, the 8 lanes of a store phase in 8 distinct chunks
          uint4* row = reinterpret_cast<uint4*>(ptr(tab + (e << 8)));
          const uint4 hi4 = make_uint4(v.x, v.x, v.x, v.x), lo4 = make_uint4(v.y, v.y, v.y, v.y);
#pragma unroll
          for (int c0 = 0; c0 < 8; ++c0) {
            row[(c0 + lane) & 7] = hi4;
            row[8 + ((c0 + lane) & 7)] = lo4;
          }
        } else {
          uint32_t* row = reinterpret_cast<uint32_t*>(ptr(tab + (e << 8)));
          for (int c0 = 0; c0 < 32; ++c0) {
            const int c = (c0 + lane) & 31;
            row[c] = v.x;
            row[32 + c] = v.y;
          }
        }
      } else {
        const int ek = e - kV;
        constexpr int kb = M::kF16K ? 2 : KB;  // (no K table for fp16 K)
        const uint2 v = pair_entry(p.k_cent[ek & ((1 << kb) - 1)], p.k_cent[ek >> kb]);
        if constexpr (CL) {
          uint4* row = reinterpret_cast<uint4*>(ptr(tab + 65536 + (ek << 7)));
          const uint4 v4 = make_uint4(v.x, v.y, v.x, v.y);
#pragma unroll
          for (int c0 = 0; c0 < kCopies / 2; ++c0) row[(c0 + lane) & (kCopies / 2 - 1)] = v4;
        } else {
          uint2* row = reinterpret_cast<uint2*>(ptr(tab + 65536 + (ek << 7)));
          for (int c0 = 0; c0 < kCopies; ++c0) row[(c0 + lane) & (kCopies - 1)] = v;
        }
      }
    }
  }
  // cluster variant: the CTA's row is known from its index, so the rotation
  // signs of the query (parameters only) are computed before the wait and the
  // query itself is loaded right after it, alongside the sequence lengths
  unsigned cl_neg = 0u;
  uint2 cl_q = make_uint2(0u, 0u);
  if constexpr (CL) {
    const int crow = blockIdx.x / kClusterCtas;
    if (warp < G)
#pragma unroll
      for (int i = 0; i < 4; ++i) cl_neg |= sign_negative(p.seed, p.layer, crow % p.hkv, 4 * lane + i) ? 1u << i : 0u;
  }
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  if constexpr (CL) {
    const int crow = blockIdx.x / kClusterCtas;
    if (warp < G)
      cl_q = *reinterpret_cast<const uint2*>(p.q + (static_cast<int64_t>(crow / p.hkv) * p.hq + (crow % p.hkv) * G + warp) * D +
                                             4 * lane);
  }
  if (blockIdx.x == 0 && tid == 0 && p.status != nullptr) {
    for (int b = 0; b < p.batch / p.nq; ++b) {
      const int len = p.seq_lens[b];
      if (len < 0 || len > p.cap || len > p.max_seq_len) {
        atomicOr(p.status, TQ_DEV_ERR_SEQ_LEN);
        break;
      }
    }
  }
  tile_prefix<M::kThreads, MQ>(p, prefix, scan);  // synchronizes (the tables too)
  const long long total = prefix[p.batch];

  uint32_t ring = 0;
  for (int w = 0; w < NW; ++w) {
    const uint32_t a = lay.take(S * M::kBuf);
    if (w == warp) ring = a;
  }
  if (lay.cur > s0 + static_cast<uint32_t>(M::kSmem)) {  // cannot happen within the static budget
    if (tid == 0 && p.status != nullptr) atomicOr(p.status, TQ_DEV_ERR_LAYOUT);
    return;
  }
  uint8_t* const wring = ptr(ring);
  const uint32_t w16 = w16_all + static_cast<uint32_t>(warp * M::kW16);
  int4* descs = descs_all + warp * 8;

  // softmax role of the lane: token tau, heads h0 and h0 + 1
  const int tau = g + 8 * (t >> 1);
  const int h0 = 2 * (t & 1);
  // K-phase window offset of the lane within a token record, V-phase record offset
  constexpr int kKRec = KB * 16;
  const uint32_t k_win = static_cast<uint32_t>(4 * KB * t);  // bytes: 32 coordinates of KB bits
  const uint32_t v_win = static_cast<uint32_t>(2 * M::kVB * g);  // byte offset of coordinates 16 g .. 16 g + 15
  uint32_t qb[16];   // B fragments of the scores: [q hi | q lo] of the lane's (head, half), 8 chunks
  float sc[2];       // log2-domain score scale of heads h0, h0 + 1 (rotation, centroid and query scales)
  int cur_b = -1, cur_h = -1;

  long long t0, t1;
  if constexpr (CL) {
    // one cluster of kClusterCtas CTAs per (b, h) row, CTA rank r taking the r-th
    // equal part of the row's tiles (cold, then hot); a CTA with no tile still
    // takes part in the cluster barriers of the merge
    const int crow = blockIdx.x / kClusterCtas, rank = blockIdx.x % kClusterCtas;
    const int rb = crow / p.hkv, rh = crow % p.hkv;
    const SeqTiles sq = seq_tiles<MQ>(p, rb);
    const long long per_h = sq.tc + sq.th;
    const long long hb = prefix[rb] + rh * per_h;
    t0 = hb + per_h * rank / kClusterCtas;
    t1 = hb + per_h * (rank + 1) / kClusterCtas;
    if (tid < 2 * 4) {  // no partial yet: (m, l) = (-inf, 0) for both parts of every head slot
      cpart[2 * 4 * D + 2 * tid] = -INFINITY;
      cpart[2 * 4 * D + 2 * tid + 1] = 0.0f;
    }
  } else {
    // the CTA's range of the weighted split (tq_split_plan.h): tiles plus a
    // price for every segment start, in equal shares
    const long long cost_all = split_total_cost(total, static_cast<long long>(p.batch) * p.hkv, p.price);
    auto start_of = [&](int c) -> long long {
      if (c >= p.grid) return total;
      const long long tau = split_cost_at(cost_all, p.grid, c);
      const int v = split_find_seq(prefix, p.batch, p.hkv, p.price, tau);
      return v < 0 ? 0 : split_tile_in_seq(prefix, v, p.hkv, seq_tiles<MQ>(p, v).tc, p.price, tau);
    };
    t0 = start_of(blockIdx.x);
    t1 = start_of(blockIdx.x + 1);
    if (t0 >= t1) return;
  }
  const int my_n = static_cast<int>((t1 - t0 - warp + NW - 1) / NW);
  int j_issue = 0, j = 0;
  Cursor cur;
  TileBlocks tb{0, 0};
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
      const int staged = stage_tile<KB, M::kVB, PAGED, M::kVPitch, M::kKPitch>(p, cb, cur.h, hot, t_begin, n_valid, tb,
                                                              ring + static_cast<uint32_t>((j_issue % S) * M::kBuf), lane);
      if (hot && (lane >> 1) < n_valid) {  // the fp16 ring rows of a hot tile into L1: 128 bytes per lane
        const int pos = t_begin + (lane >> 1);
        const uint16_t* row = p.v_ring + ((static_cast<int64_t>(cb) * p.hkv + cur.h) * p.hot + pos % p.hot) * D;
        asm volatile("prefetch.global.L1 [%0];\n" ::"l"(row + 64 * (lane & 1)));
      }
      if (lane == 0) descs[j_issue % S] = make_int4(cb, cur.h | (hot << 16), t_begin, staged);
      cursor_advance<MQ>(p, cur, NW);
      if constexpr (PAGED)
        if (j_issue + 1 < my_n) tb = load_tile_blocks(p, cache_seq<MQ>(p, cur.b), cursor_t_begin(cur), cursor_n_valid(cur));
    }
    cp_async_commit();
    ++j_issue;
  };
  if constexpr (CL) {
#pragma unroll 1
    for (int st = 0; st < S - 1; ++st) issue();  // one copy of the code: it runs once per CTA here
  } else {
#pragma unroll
    for (int st = 0; st < S - 1; ++st) issue();
  }

  long long seg = t0;
  while (seg < t1) {
    const TileInfo si = tile_info<MQ>(p, prefix, seg);
    const long long seg_end = si.row_end < t1 ? si.row_end : t1;
    if (si.b != cur_b || si.h != cur_h) {
      if constexpr (M::kF16K || M::kI8) {
        // fp16 K and the int8 mode: the scores are q . k / sqrt(d) (times the K
        // scale in the int8 mode) with the raw fp16 query, exact operands.  Lane
        // (g, t) holds column g (query head g of the group, zero for g >= G) of
        // every chunk's B fragment: for fp16 K coordinates 16 c + 2 t, + 1 and
        // 16 c + 2 t + 8, + 9; for int8 K, whose chunk rows are permuted so that a
        // lane's four codes are one word, coordinates 16 c + 4 t .. 16 c + 4 t + 3.
        const uint32_t* q32 =
            reinterpret_cast<const uint32_t*>(p.q + (static_cast<int64_t>(si.b) * p.hq + si.h * G + (g < G ? g : 0)) * D);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          qb[2 * c] = g < G ? q32[M::kI8 ? 8 * c + 2 * t : 8 * c + t] : 0u;
          qb[2 * c + 1] = g < G ? q32[M::kI8 ? 8 * c + 2 * t + 1 : 8 * c + t + 4] : 0u;
        }
        sc[0] = sc[1] = kLog2e / kSqrtD;
      } else {
      // rotated query of the G heads, H D q (unnormalized), in qs: warp jj
      // transforms head jj, lane l holding coordinates 4 l .. 4 l + 3 (index bits
      // 0 and 1 in registers, bits 2..6 across lanes, in ascending order)
      __syncthreads();
      if (warp < G) {
        uint2 raw;
        if constexpr (CL) raw = cl_q;  // the cluster variant's one row, loaded after the wait
        else raw = *reinterpret_cast<const uint2*>(p.q + (static_cast<int64_t>(si.b) * p.hq + si.h * G + warp) * D + 4 * lane);
        float x[4];
        const float2 x01 = half2_bits_to_float2(raw.x), x23 = half2_bits_to_float2(raw.y);
        x[0] = x01.x;
        x[1] = x01.y;
        x[2] = x23.x;
        x[3] = x23.y;
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (CL ? ((cl_neg >> i) & 1u) != 0 : sign_negative(p.seed, p.layer, si.h, 4 * lane + i)) x[i] = -x[i];
        float a0 = fadd(x[0], x[1]), a1 = fsub(x[0], x[1]), a2 = fadd(x[2], x[3]), a3 = fsub(x[2], x[3]);  // bit 0
        x[0] = fadd(a0, a2);  // bit 1
        x[2] = fsub(a0, a2);
        x[1] = fadd(a1, a3);
        x[3] = fsub(a1, a3);
#pragma unroll
        for (int m = 1; m < 32; m <<= 1) {  // bits 2..6
          const bool upper = (lane & m) != 0;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float o = __shfl_xor_sync(0xffffffffu, x[i], m);
            x[i] = upper ? fsub(o, x[i]) : fadd(x[i], o);
          }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) qs[qs_at(warp, 4 * lane + i)] = x[i];
      }
      __syncthreads();
      // lane (g, t): head g & 3, half g >> 2, coordinates 32 t .. 32 t + 31, scaled by a
      // power of two that puts the head's largest |value| in [2^13, 2^14).  Warp 0
      // computes the fragments and publishes them (the row-combine buffer is free
      // here); every warp then loads its lanes' copies.
      uint32_t* qb_s = reinterpret_cast<uint32_t*>(comb);         // [32 lanes][16]
      float* qsc_s = comb + 32 * 16;                              // [32 lanes]
      if (warp == 0) {
        const int hh = g & 3;
        float amax = 0.0f;
        if (hh < G) {
          float am[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};  // independent partial maxima
#pragma unroll
          for (int i = 0; i < 32; ++i) am[i & 7] = fmaxf(am[i & 7], fabsf(qs[qs_at(hh, 32 * t + i)]));
          amax = fmaxf(fmaxf(fmaxf(am[0], am[1]), fmaxf(am[2], am[3])), fmaxf(fmaxf(am[4], am[5]), fmaxf(am[6], am[7])));
        }
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        const int ex = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu);  // biased exponent, 0 for zero
        const float qscale = ex == 0 ? 1.0f : __uint_as_float(static_cast<uint32_t>(127 + 13 + 127 - ex) << 23);
        uint32_t frag[16];
#pragma unroll
        for (int c = 0; c < 8; ++c)
#pragma unroll
          for (int jp = 0; jp < 2; ++jp) {
            uint32_t v = 0u;
            if (hh < G) {
              const float x0 = fmul(qs[qs_at(hh, 32 * t + 4 * c + 2 * jp)], qscale);
              const float x1 = fmul(qs[qs_at(hh, 32 * t + 4 * c + 2 * jp + 1)], qscale);
              uint16_t a0, l0, a1, l1;
              split_f16(x0, a0, l0);
              split_f16(x1, a1, l1);
              v = (g >> 2) == 0 ? pack16(a0, a1) : pack16(l0, l1);
            }
            frag[2 * c + jp] = v;
          }
        uint4* dst = reinterpret_cast<uint4*>(qb_s + 16 * lane);
#pragma unroll
        for (int k = 0; k < 4; ++k) dst[k] = make_uint4(frag[4 * k], frag[4 * k + 1], frag[4 * k + 2], frag[4 * k + 3]);
        qsc_s[lane] = qscale;
      }
      __syncthreads();
      {
        const uint4* src = reinterpret_cast<const uint4*>(qb_s + 16 * lane);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint4 v = src[k];
          qb[4 * k] = v.x;
          qb[4 * k + 1] = v.y;
          qb[4 * k + 2] = v.z;
          qb[4 * k + 3] = v.w;
        }
        // the scale of head h was computed by lane 4 h (half 0, t = 0)
#pragma unroll
        for (int i = 0; i < 2; ++i) sc[i] = kLog2e / static_cast<float>(D) * kCentUnscale / qsc_s[4 * ((h0 + i) & 3)];
      }
      }
      cur_b = si.b;
      cur_h = si.h;
    }

    float m_own[2] = {-INFINITY, -INFINITY}, lsum[2] = {0.0f, 0.0f};
    float ms_own[2] = {-INFINITY, -INFINITY};  // sparse V: running maximum of the scores alone
    float acc[8][4];
#pragma unroll
    for (int mb = 0; mb < 8; ++mb)
#pragma unroll
      for (int k = 0; k < 4; ++k) acc[mb][k] = 0.0f;

    while (j < my_n && t0 + warp + static_cast<long long>(NW) * j < seg_end) {
      issue();
      cp_async_wait<S - 1>();
      __syncwarp();
      const int4 dsc = descs[j % S];
      const int tb_b = dsc.x, tb_h = dsc.y & 0xFFFF, n_valid = dsc.w, t_begin = dsc.z;
      const bool hot = (dsc.y >> 16) != 0;
      const uint8_t* tbp = wring + (j % S) * M::kBuf;
      const uint32_t tbs = ring + static_cast<uint32_t>((j % S) * M::kBuf);

      // ---- scores on the tensor cores: tokens 0..7 and 8..15 in two MMA chains,
      // A row g = hi and row g + 8 = lo halves of the token's centroids
      float sacc[4];
      if constexpr (M::kI8) {
        // int8 K: tokens as M (rows g and g + 8), chunk c as K with k = 2 t, 2 t + 1 ->
        // coordinates 16 c + 4 t, + 1 and k = 2 t + 8, 2 t + 9 -> 16 c + 4 t + 2, + 3:
        // one 32-bit load per token and chunk, its codes made exact fp16 pairs
        float dk[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        const uint32_t ka = tbs + static_cast<uint32_t>(g * M::kKPitch + 4 * t);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint32_t wg = lds32<0>(ka + 16u * c) ^ 0x80808080u;
          const uint32_t wh = lds32<0>(ka + static_cast<uint32_t>(8 * M::kKPitch) + 16u * c) ^ 0x80808080u;
          mma_f16(dk, int8_half2<0>(wg), int8_half2<0>(wh), int8_half2<2>(wg), int8_half2<2>(wh), qb[2 * c],
                  qb[2 * c + 1]);
        }
        sacc[0] = dk[0];
        sacc[1] = dk[1];
        sacc[2] = dk[2];
        sacc[3] = dk[3];
      } else if constexpr (M::kF16K) {
        // tokens as M (rows g and g + 8 of an MMA are tokens g and g + 8), chunk c =
        // coordinates 16 c .. 16 c + 15 as K, the query heads as N; ldmatrix reads
        // the A fragment from the staged fp16 rows (lane l addresses row l mod 16,
        // coordinate half l / 16)
        float dk[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        const uint32_t arow = tbs + static_cast<uint32_t>((lane & 15) * M::kKPitch + (lane >> 4) * 16);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint32_t a0, a1, a2, a3;
          ldsm_x4(arow + 32u * c, a0, a1, a2, a3);
          mma_f16(dk, a0, a1, a2, a3, qb[2 * c], qb[2 * c + 1]);
        }
        // columns 2 t, 2 t + 1 of tokens g and g + 8 (columns >= 4 are zero), laid out
        // as the hi / lo sums below so that the same exchange gives every lane its dot
        sacc[0] = dk[0];
        sacc[1] = dk[1];
        sacc[2] = dk[2];
        sacc[3] = dk[3];
      } else {
      float dh[2][4] = {{0.0f, 0.0f, 0.0f, 0.0f}, {0.0f, 0.0f, 0.0f, 0.0f}};
      {
        constexpr int kWords = KB;  // 32 coordinates x KB bits
        uint32_t wg[kWords + 1], wh[kWords + 1];
        const uint32_t ag = tbs + static_cast<uint32_t>(g * kKRec) + k_win;
        const uint32_t ah = ag + static_cast<uint32_t>(8 * kKRec);
        if constexpr (KB == 4) {  // vector loads sized to the window keep the warp's loads conflict free
          const uint4 a = lds128<0>(ag), b = lds128<0>(ah);
          wg[0] = a.x; wg[1] = a.y; wg[2] = a.z; wg[3] = a.w;
          wh[0] = b.x; wh[1] = b.y; wh[2] = b.z; wh[3] = b.w;
        } else if constexpr (KB == 2) {
          const uint2 a = lds64u<0>(ag), b = lds64u<0>(ah);
          wg[0] = a.x; wg[1] = a.y;
          wh[0] = b.x; wh[1] = b.y;
        } else {
#pragma unroll
          for (int i = 0; i < kWords; ++i) {
            wg[i] = lds32<0>(ag + 4u * i);
            wh[i] = lds32<0>(ah + 4u * i);
          }
        }
        wg[kWords] = 0u;
        wh[kWords] = 0u;
        auto chunk = [&](auto C_) {
          constexpr int c = decltype(C_)::value;
          const uint2 e0 = lds64a(k_pair_addr<KB, 2 * c>(wg, kbase));      // token g: (a0, a1)
          const uint2 e2 = lds64a(k_pair_addr<KB, 2 * c + 1>(wg, kbase));  // token g: (a2, a3)
          const uint2 e1 = lds64a(k_pair_addr<KB, 2 * c>(wh, kbase));      // token g + 8
          const uint2 e3 = lds64a(k_pair_addr<KB, 2 * c + 1>(wh, kbase));
          mma_f16(dh[0], e0.x, e0.y, e2.x, e2.y, qb[2 * c], qb[2 * c + 1]);
          mma_f16(dh[1], e1.x, e1.y, e3.x, e3.y, qb[2 * c], qb[2 * c + 1]);
        };
        chunk(std::integral_constant<int, 0>{});
        chunk(std::integral_constant<int, 1>{});
        chunk(std::integral_constant<int, 2>{});
        chunk(std::integral_constant<int, 3>{});
        chunk(std::integral_constant<int, 4>{});
        chunk(std::integral_constant<int, 5>{});
        chunk(std::integral_constant<int, 6>{});
        chunk(std::integral_constant<int, 7>{});
      }
      // rows g (hi) + g + 8 (lo): columns 2 t, 2 t + 1 of token g (dh[0]) and g + 8 (dh[1])
      sacc[0] = fadd(dh[0][0], dh[0][2]);
      sacc[1] = fadd(dh[0][1], dh[0][3]);
      sacc[2] = fadd(dh[1][0], dh[1][2]);
      sacc[3] = fadd(dh[1][1], dh[1][3]);
      }
      // hi and lo columns of the lane's token: lanes t < 2 hold the hi columns of
      // token g, lanes t >= 2 the lo columns of token g + 8; exchange with t ^ 2
      float dot[2];
      {
        const bool lo_lane = (t >> 1) != 0;
        const float s0v = lo_lane ? sacc[0] : sacc[2], s1v = lo_lane ? sacc[1] : sacc[3];
        const float r0 = __shfl_xor_sync(0xffffffffu, s0v, 2), r1 = __shfl_xor_sync(0xffffffffu, s1v, 2);
        dot[0] = fadd(lo_lane ? sacc[2] : sacc[0], r0);
        dot[1] = fadd(lo_lane ? sacc[3] : sacc[1], r1);
      }

      // ---- online softmax (base 2); weights below 2^8 (see the header)
      const float* knorm = reinterpret_cast<const float*>(tbp + M::kKTile);
      const float* vnorm = reinterpret_cast<const float*>(tbp + M::kKTile + M::kKNorm + M::kVTile);
      const bool tok_ok = tau < n_valid;
      const float nk = M::kF16K ? 1.0f : knorm[tau];  // fp16 K: the dot product is the score
      const float nv = hot ? 1.0f : vnorm[tau];
      int ev = static_cast<int>((__float_as_uint(nv) >> 23) & 0xFFu) - 127;
      ev = ev < -64 ? -64 : ev;
      const float evf = static_cast<float>(ev + 1);
      float sj[2];
      bool ok[2];
      bool bump = false;
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        ok[i] = tok_ok && h0 + i < G;
        sj[i] = ok[i] ? fmul(fmul(dot[i], sc[i]), nk) : -INFINITY;  // staged data of masked rows is stale
        bump |= ok[i] && fadd(sj[i], evf) > fadd(m_own[i], kLazy);
      }
      if (__any_sync(0xffffffffu, bump)) {
        float alpha[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          float tm = ok[i] ? fadd(sj[i], evf) : -INFINITY;
          tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 2));
          tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 4));
          tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 8));
          tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 16));
          const float mn = fmaxf(m_own[i], tm);
          alpha[i] = mn == -INFINITY ? 1.0f : ex2_approx(fsub(m_own[i], mn));  // 0 for the row's first tile
          lsum[i] = fmul(lsum[i], alpha[i]);
          m_own[i] = mn;
        }
        // accumulator columns 2 t, 2 t + 1 are heads h0, h0 + 1 (hi or lo half)
#pragma unroll
        for (int mb = 0; mb < 8; ++mb) {
          acc[mb][0] = fmul(acc[mb][0], alpha[0]);
          acc[mb][1] = fmul(acc[mb][1], alpha[1]);
          acc[mb][2] = fmul(acc[mb][2], alpha[0]);
          acc[mb][3] = fmul(acc[mb][3], alpha[1]);
        }
      }
      if constexpr (SPARSE) {
        // a token whose weight relative to the running score maximum is below tau has a
        // normalized weight below tau: its V is skipped (its weight still counts in the mass)
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          float tm = sj[i];
          tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 2));
          tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 4));
          tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 8));
          tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 16));
          ms_own[i] = fmaxf(ms_own[i], tm);
        }
      }
      bool any_w = false;
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        float pj = ok[i] ? ex2_approx(fsub(sj[i], m_own[i])) : 0.0f;
        lsum[i] = fadd(lsum[i], pj);
        float w = ok[i] ? fmul(pj, nv) : 0.0f;  // the staged norm of a masked row is stale
        if (SPARSE && ok[i] && ex2_approx(fsub(sj[i], ms_own[i])) < p.sparse_tau) w = 0.0f;
        any_w |= w != 0.0f;
        uint16_t wh16, wl16;
        split_f16(w, wh16, wl16);
        const uint32_t o = static_cast<uint32_t>(((h0 + i) * kTile + tau) * 2);
        asm volatile("st.shared.u16 [%0], %1;\n" ::"r"(w16 + o), "h"(wh16));
        asm volatile("st.shared.u16 [%0], %1;\n" ::"r"(w16 + 4u * kTile * 2u + o), "h"(wl16));
      }
      const bool do_v = SPARSE ? __any_sync(0xffffffffu, any_w) : true;
      __syncwarp();

      // ---- V on the tensor cores: B = the weights of column g (head g & 3, half g >> 2)
      if (do_v) {
        const uint32_t wb = w16 + static_cast<uint32_t>(((g >> 2) * 4 + (g & 3)) * kTile * 2);
        const uint32_t b0 = lds32<0>(wb + 4u * t), b1 = lds32<0>(wb + 4u * t + 16u);
        if (M::kI8 && !hot) {
          // int8 V codes (exact fp16) in the layout of the hot rows: lane (g, t) holds
          // coordinates 16 g .. 16 g + 15 of tokens 2 t, 2 t + 1, 2 t + 8, 2 t + 9 (one
          // 16-byte load each); M block b pairs the bytes of coordinates 16 g + 2 b, + 1
          const uint32_t vt = tbs + static_cast<uint32_t>(M::kKTile + M::kKNorm + 16 * g);
          constexpr int P = M::kVPitch;
          const uint4 xa = lds128<0>(vt + static_cast<uint32_t>((2 * t) * P));
          const uint4 xb = lds128<0>(vt + static_cast<uint32_t>((2 * t + 1) * P));
          const uint4 xc = lds128<0>(vt + static_cast<uint32_t>((2 * t + 8) * P));
          const uint4 xd = lds128<0>(vt + static_cast<uint32_t>((2 * t + 9) * P));
          auto w4 = [](const uint4& v, int i) { return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w; };
#pragma unroll
          for (int mb = 0; mb < 8; ++mb) {
            const int wi = mb >> 1, c0 = 2 * (mb & 1);
            const uint32_t sel = static_cast<uint32_t>(c0 | (4 + c0) << 4 | (c0 + 1) << 8 | (5 + c0) << 12);
            // bytes (a, b) of coordinate 16 g + 2 mb, then of + 1, biased to code + 128
            const uint32_t ab = __byte_perm(w4(xa, wi), w4(xb, wi), sel) ^ 0x80808080u;
            const uint32_t cd = __byte_perm(w4(xc, wi), w4(xd, wi), sel) ^ 0x80808080u;
            mma_f16(acc[mb], int8_half2<0>(ab), int8_half2<2>(ab), int8_half2<0>(cd), int8_half2<2>(cd), b0, b1);
          }
        } else if (!hot) {
          const uint32_t vt = tbs + static_cast<uint32_t>(M::kKTile + M::kKNorm) + v_win;
          constexpr int P = M::kVPitch;
          const uint2 wa = v_nibbles<M::kVB>(vt + static_cast<uint32_t>((2 * t) * P));
          const uint2 wbw = v_nibbles<M::kVB>(vt + static_cast<uint32_t>((2 * t + 1) * P));
          const uint2 wc = v_nibbles<M::kVB>(vt + static_cast<uint32_t>((2 * t + 8) * P));
          const uint2 wd = v_nibbles<M::kVB>(vt + static_cast<uint32_t>((2 * t + 9) * P));
          uint32_t ab_lo[2], ab_hi[2], cd_lo[2], cd_hi[2];
          interleave(wa.x, wbw.x, ab_lo[0], ab_hi[0]);
          interleave(wa.y, wbw.y, ab_lo[1], ab_hi[1]);
          interleave(wc.x, wd.x, cd_lo[0], cd_hi[0]);
          interleave(wc.y, wd.y, cd_lo[1], cd_hi[1]);
          auto vblock = [&](auto B_) {
            constexpr int mb = decltype(B_)::value, w = mb >> 2, k = mb & 3;
            const uint2 e0 = lds_entry(v_pair_addr<k>(ab_lo[w], vbase));
            const uint2 e1 = lds_entry(v_pair_addr<k>(ab_hi[w], vbase));
            const uint2 e2 = lds_entry(v_pair_addr<k>(cd_lo[w], vbase));
            const uint2 e3 = lds_entry(v_pair_addr<k>(cd_hi[w], vbase));
            mma_f16(acc[mb], e0.x, e1.x, e2.x, e3.x, b0, b1);
            mma_f16(acc[mb], e0.y, e1.y, e2.y, e3.y, b0, b1);
          };
          vblock(std::integral_constant<int, 0>{});
          vblock(std::integral_constant<int, 1>{});
          vblock(std::integral_constant<int, 2>{});
          vblock(std::integral_constant<int, 3>{});
          vblock(std::integral_constant<int, 4>{});
          vblock(std::integral_constant<int, 5>{});
          vblock(std::integral_constant<int, 6>{});
          vblock(std::integral_constant<int, 7>{});
        } else {
          // hot row: the fp16 ring (exact operands), coordinates 16 g .. 16 g + 15 of
          // tokens 2 t, 2 t + 1, 2 t + 8, 2 t + 9 (zeros past the tile's tokens)
          uint4 x[4][2];
          const int tk[4] = {2 * t, 2 * t + 1, 2 * t + 8, 2 * t + 9};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            x[u][0] = make_uint4(0u, 0u, 0u, 0u);
            x[u][1] = make_uint4(0u, 0u, 0u, 0u);
            if (tk[u] < n_valid) {
              const int pos = t_begin + tk[u];
              const uint4* src = reinterpret_cast<const uint4*>(
                  p.v_ring + ((static_cast<int64_t>(tb_b) * p.hkv + tb_h) * p.hot + pos % p.hot) * D + 16 * g);
              x[u][0] = src[0];
              x[u][1] = src[1];
            }
          }
          auto word = [&](int u, int i) {
            const uint4& q4 = x[u][i >> 2];
            return (i & 3) == 0 ? q4.x : (i & 3) == 1 ? q4.y : (i & 3) == 2 ? q4.z : q4.w;
          };
#pragma unroll
          for (int mb = 0; mb < 8; ++mb) {
            const uint32_t a0 = __byte_perm(word(0, mb), word(1, mb), 0x5410);
            const uint32_t a1 = __byte_perm(word(0, mb), word(1, mb), 0x7632);
            const uint32_t a2 = __byte_perm(word(2, mb), word(3, mb), 0x5410);
            const uint32_t a3 = __byte_perm(word(2, mb), word(3, mb), 0x7632);
            mma_f16(acc[mb], a0, a1, a2, a3, b0, b1);
          }
        }
      }
      __syncwarp();
      ++j;
    }

    // ---- leave the row: hi + lo halves, lanes -> warp -> CTA, one partial per (CTA, row).
    // Each warp writes its sum, scaled to the CTA's maximum, to a slot of its own;
    // the slots are then added in warp order (the result does not depend on timing)
    // lanes t < 2 keep head 2 t + (k & 1) at coordinate 16 g + 2 mb + (k >> 1)
#pragma unroll
    for (int mb = 0; mb < 8; ++mb)
#pragma unroll
      for (int k = 0; k < 4; ++k) acc[mb][k] = fadd(acc[mb][k], __shfl_xor_sync(0xffffffffu, acc[mb][k], 2));
    float lw[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      float l = lsum[i];
      l = fadd(l, __shfl_xor_sync(0xffffffffu, l, 2));
      l = fadd(l, __shfl_xor_sync(0xffffffffu, l, 4));
      l = fadd(l, __shfl_xor_sync(0xffffffffu, l, 8));
      l = fadd(l, __shfl_xor_sync(0xffffffffu, l, 16));
      lw[i] = l;
    }
    if (lane < 2) {  // lane t (g = 0) holds heads 2 t, 2 t + 1
#pragma unroll
      for (int i = 0; i < 2; ++i)
        if (h0 + i < G) {
          wml[(warp * 4 + h0 + i) * 2] = m_own[i];
          wml[(warp * 4 + h0 + i) * 2 + 1] = lw[i];
        }
    }
    __syncthreads();
    if (t < 2) {
      float* slot_w = comb + warp * 4 * 136;
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int hd = h0 + i;
        if (hd >= G) continue;
        float mm = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w) mm = fmaxf(mm, wml[(w * 4 + hd) * 2]);
        const float sc2 = m_own[i] == -INFINITY ? 0.0f : exp2f(m_own[i] - mm);  // 0: no token of the head
        float* c2 = slot_w + comb_at(hd, 16 * g);  // coordinates 16 g .. 16 g + 15 are contiguous
#pragma unroll
        for (int mb = 0; mb < 8; ++mb) {
          c2[2 * mb] = fmul(acc[mb][i], sc2);
          c2[2 * mb + 1] = fmul(acc[mb][2 + i], sc2);
        }
      }
    }
    __syncthreads();
    const float unscale = (si.hot || M::kI8) ? 1.0f : kCentUnscale;  // cold packed sums carry the table scale
    if constexpr (CL) {
      // the partial stays in this CTA's shared memory, part 0 cold and part 1 hot
      float* pa = cpart + si.hot * 4 * D;
      for (int i = tid; i < G * D; i += M::kThreads) {
        const int at = comb_at(i / D, i % D);
        float sum = 0.0f;
#pragma unroll
        for (int w = 0; w < NW; ++w) sum = fadd(sum, comb[w * 4 * 136 + at]);
        pa[i] = fmul(sum, unscale);
      }
      if (tid < G) {
        float mm = -INFINITY, ll = 0.0f;
#pragma unroll
        for (int w = 0; w < NW; ++w) mm = fmaxf(mm, wml[(w * 4 + tid) * 2]);
#pragma unroll
        for (int w = 0; w < NW; ++w) {
          const float mwv = wml[(w * 4 + tid) * 2];
          if (mwv != -INFINITY) ll = ffma(wml[(w * 4 + tid) * 2 + 1], exp2f(mwv - mm), ll);
        }
        cpart[2 * 4 * D + (si.hot * 4 + tid) * 2] = mm;
        cpart[2 * 4 * D + (si.hot * 4 + tid) * 2 + 1] = ll;
      }
    } else {
      const long long slot = static_cast<long long>(blockIdx.x) + si.row;
      for (int i = tid; i < G * D; i += M::kThreads) {
        const int at = comb_at(i / D, i % D);
        float sum = 0.0f;
#pragma unroll
        for (int w = 0; w < NW; ++w) sum = fadd(sum, comb[w * 4 * 136 + at]);
        p.ws_acc[slot * G * D + i] = fmul(sum, unscale);
      }
      if (tid < G) {
        float mm = -INFINITY, ll = 0.0f;
#pragma unroll
        for (int w = 0; w < NW; ++w) mm = fmaxf(mm, wml[(w * 4 + tid) * 2]);
#pragma unroll
        for (int w = 0; w < NW; ++w) {
          const float mwv = wml[(w * 4 + tid) * 2];
          if (mwv != -INFINITY) ll = ffma(wml[(w * 4 + tid) * 2 + 1], exp2f(mwv - mm), ll);
        }
        p.ws_ml[(slot * G + tid) * 2] = mm;
        p.ws_ml[(slot * G + tid) * 2 + 1] = ll;
      }
    }
    __syncthreads();
    seg = seg_end;
  }
  cp_async_wait<0>();
  if constexpr (CL) {
    // merge of the row's partials through distributed shared memory: CTA rank
    // hd < G combines query head hd of every CTA of the cluster (one warp, lane l
    // holding coordinates 4 l .. 4 l + 3) and writes the output; the second
    // barrier keeps every CTA's shared memory alive until the reads are done
    cluster_sync_all();
    const int rank = blockIdx.x % kClusterCtas, crow = blockIdx.x / kClusterCtas;
    if (rank < G && warp == 0) {
      const int hd = rank, rb = crow / p.hkv, rh = crow % p.hkv;
      const uint32_t base = static_cast<uint32_t>(__cvta_generic_to_shared(cpart));
      float2 ml[2 * kClusterCtas];
      float4 av[2 * kClusterCtas];
#pragma unroll
      for (int r = 0; r < kClusterCtas; ++r) {
        const uint32_t rbase = map_cluster(base, r);
#pragma unroll
        for (int part = 0; part < 2; ++part) {
          ml[2 * r + part] = ld_cluster_f2(rbase + 4u * (2 * 4 * D + (part * 4 + hd) * 2));
          av[2 * r + part] = ld_cluster_f4(rbase + 4u * ((part * 4 + hd) * D + 4 * lane));
        }
      }
      float mm = -INFINITY;
#pragma unroll
      for (int i = 0; i < 2 * kClusterCtas; ++i) mm = fmaxf(mm, ml[i].x);
      float l = 0.0f, y[4] = {0.0f, 0.0f, 0.0f, 0.0f}, hv[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
      for (int i = 0; i < 2 * kClusterCtas; ++i) {
        if (ml[i].x == -INFINITY) continue;  // a CTA without tiles of this part
        const float sc = exp2f(ml[i].x - mm);
        l = ffma(ml[i].y, sc, l);
        const float a[4] = {av[i].x, av[i].y, av[i].z, av[i].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          if (i & 1) hv[k] = ffma(a[k], sc, hv[k]);
          else y[k] = ffma(a[k], sc, y[k]);
        }
      }
      unsigned neg4 = 0u;
#pragma unroll
      for (int i = 0; i < 4; ++i) neg4 |= sign_negative(p.seed, p.layer, rh, 4 * lane + i) ? 1u << i : 0u;
      merge_finish(y, hv, l, neg4, !M::kI8, p.out + (static_cast<int64_t>(rb) * p.hq + rh * G + hd) * D, lane);
    }
    cluster_sync_all();
  }
}

template <int G, int KB, bool SPARSE, bool PAGED, bool MQ, int VB = 4>
tq_status launch_mma(const DecodeParams& p, cudaStream_t stream) {
  using M = MmaCfg<KB, false, VB>;
  auto kern = decode_mma_kernel<G, KB, SPARSE, PAGED, MQ, false, VB>;
  static KernelMemo memo;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.grid);
  cfg.blockDim = dim3(M::kThreads);
  cfg.dynamicSmemBytes = M::kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = kProgrammaticLaunch;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (launch_with_limit(kern, M::kSmem, memo, current_device(), cfg, p) != cudaSuccess) return TQ_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

// Cluster variant (one cluster of kClusterCtas CTAs per (b, h) row, partials
// merged through distributed shared memory, no merge launch).  Returns
// TQ_ERR_UNSUPPORTED without launching when the rows do not fit in one wave of
// clusters on this GPU (the caller then runs the persistent kernel).
template <int G, int KB, int VB>
tq_status launch_mma_cluster(const DecodeParams& p, cudaStream_t stream) {
  using M = MmaCfg<KB, true, VB>;
  auto kern = decode_mma_kernel<G, KB, false, false, false, true, VB>;
  static KernelMemo memo;
  const int dev = current_device();
  if (!ensure_smem_limit(kern, M::kSmem, memo, dev)) return TQ_ERR_CUDA;
  const long long rows = static_cast<long long>(p.batch) * p.hkv;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(rows * kClusterCtas));
  cfg.blockDim = dim3(M::kThreads);
  cfg.dynamicSmemBytes = M::kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kClusterCtas;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = kProgrammaticLaunch;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const int fit = cluster_fit(kern, cfg, memo, dev);  // clusters resident at once (device and kernel)
  if (fit < 0) return TQ_ERR_CUDA;
  if (rows > fit) return TQ_ERR_UNSUPPORTED;
  if (launch_with_limit(kern, M::kSmem, memo, dev, cfg, p) != cudaSuccess) return TQ_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

}  // namespace
}  // namespace tq
