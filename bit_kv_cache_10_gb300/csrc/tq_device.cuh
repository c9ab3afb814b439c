// Device building blocks of the quantize and dequantize kernels.
//
// Every function here is __host__ __device__: the device build is what the
// kernels run; the host build of the same source (IEEE float32 with
// round-to-nearest, no contraction) backs a verification hook that lets the
// per-vector arithmetic be checked on a CPU-only machine.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>

#include "tq.h"
#include "tq_signs.h"

namespace tq {

// Cache row of token t of (sequence b, KV head h): the contiguous layout
// [B, Hkv, cap] or, with a block table, row (block * Hkv + h) * bs + t % bs of
// block table[b][t / bs] (bs = 2^shift).  -1 for a table entry outside the pool.
struct RowMap {
  int hkv, cap;
  const int32_t* table;  // nullptr: contiguous
  int max_blocks, shift, num_blocks;
#ifdef __CUDACC__
  // Pool row of position t of head h inside pool block blk; -1 outside the pool.
  __device__ __forceinline__ long long in_block(int blk, int h, int t) const {
    if (blk < 0 || blk >= num_blocks) return -1;
    return ((static_cast<long long>(blk) * hkv + h) << shift) | (t & ((1 << shift) - 1));
  }
  __device__ __forceinline__ long long row(int b, int h, int t) const {
    if (table == nullptr) return (static_cast<long long>(b) * hkv + h) * cap + t;
    return in_block(table[b * max_blocks + (t >> shift)], h, t);
  }
#endif
};

inline RowMap make_row_map(const tq_cache_desc* d) {
  RowMap m{d->num_kv_heads, d->capacity, nullptr, 0, 0, 0};
  if (d->block_size > 0) {
    m.table = d->block_table;
    m.max_blocks = d->max_blocks_per_seq;
    int sh = 0;
    while ((1 << sh) < d->block_size) ++sh;
    m.shift = sh;
    m.num_blocks = d->num_blocks;
  }
  return m;
}

constexpr int D = 128;               // head_dim of the kernels
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kSqrtD = 11.313708498984761f;   // sqrt(128), float32 rounding
constexpr float kMagic = 12582912.0f;           // 1.5 * 2^23: FMA with it rounds to an integer

// ---------------------------------------------------------------------------
// Rounding-explicit float helpers (identical results on host and device)
// ---------------------------------------------------------------------------

TQ_HD float fadd(float a, float b) {
#ifdef __CUDA_ARCH__
  return __fadd_rn(a, b);
#else
  volatile float r = a + b;
  return r;
#endif
}
TQ_HD float fsub(float a, float b) {
#ifdef __CUDA_ARCH__
  return __fsub_rn(a, b);
#else
  volatile float r = a - b;
  return r;
#endif
}
TQ_HD float fmul(float a, float b) {
#ifdef __CUDA_ARCH__
  return __fmul_rn(a, b);
#else
  volatile float r = a * b;
  return r;
#endif
}
TQ_HD float ffma(float a, float b, float c) {
#ifdef __CUDA_ARCH__
  return __fmaf_rn(a, b, c);
#else
  return std::fma(a, b, c);
#endif
}
TQ_HD float fsqrt(float a) {
#ifdef __CUDA_ARCH__
  return __fsqrt_rn(a);
#else
  return std::sqrt(a);
#endif
}
TQ_HD float frcp(float a) {
#ifdef __CUDA_ARCH__
  return __frcp_rn(a);
#else
  volatile float r = 1.0f / a;
  return r;
#endif
}
TQ_HD uint32_t fbits(float f) {
#ifdef __CUDA_ARCH__
  return __float_as_uint(f);
#else
  uint32_t u;
  std::memcpy(&u, &f, 4);
  return u;
#endif
}
TQ_HD float bitsf(uint32_t u) {
#ifdef __CUDA_ARCH__
  return __uint_as_float(u);
#else
  float f;
  std::memcpy(&f, &u, 4);
  return f;
#endif
}

// Packed float32 pairs: one sm_100+ instruction for two round-to-nearest ops.
TQ_HD float2 add2(float2 a, float2 b) {
#ifdef __CUDA_ARCH__
  return __fadd2_rn(a, b);
#else
  return make_float2(fadd(a.x, b.x), fadd(a.y, b.y));
#endif
}
TQ_HD float2 sub2(float2 a, float2 b) {  // a - b as b * (-1) + a: exact product, one rounding
#ifdef __CUDA_ARCH__
  return __ffma2_rn(b, make_float2(-1.0f, -1.0f), a);
#else
  return make_float2(fsub(a.x, b.x), fsub(a.y, b.y));
#endif
}
TQ_HD float2 mul2(float2 a, float2 b) {
#ifdef __CUDA_ARCH__
  return __fmul2_rn(a, b);
#else
  return make_float2(fmul(a.x, b.x), fmul(a.y, b.y));
#endif
}
TQ_HD float2 fma2(float2 a, float2 b, float2 c) {
#ifdef __CUDA_ARCH__
  return __ffma2_rn(a, b, c);
#else
  return make_float2(ffma(a.x, b.x, c.x), ffma(a.y, b.y, c.y));
#endif
}

// fp16 bits -> float32 (exact).
TQ_HD float half_bits_to_float(uint32_t h) {
#ifdef __CUDA_ARCH__
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h)));
#else
  const uint32_t sign = (h & 0x8000u) << 16, e = (h >> 10) & 31u, m = h & 1023u;
  if (e == 0) {
    const float v = static_cast<float>(m) * 5.9604644775390625e-08f;  // m * 2^-24, exact
    return sign ? -v : v;
  }
  if (e == 31) return bitsf(sign | 0x7F800000u | (m << 13));
  return bitsf(sign | ((e + 112u) << 23) | (m << 13));
#endif
}

TQ_HD float2 half2_bits_to_float2(uint32_t w) {
  return make_float2(half_bits_to_float(w & 0xFFFFu), half_bits_to_float(w >> 16));
}

// ---------------------------------------------------------------------------
// Exact float32 norm of 128 fp16 values
// ---------------------------------------------------------------------------

// Sum of x^2 in units of 2^-48 (every fp16 square is a multiple of it): exact.
TQ_HD unsigned __int128 exact_sum_squares(const uint32_t* w) {
  unsigned __int128 s = 0;
#pragma unroll 1
  for (int j = 0; j < 2 * 64; ++j) {
    const uint32_t h = (j & 1) ? (w[j >> 1] >> 16) : (w[j >> 1] & 0xFFFFu);
    const uint32_t e = (h >> 10) & 31u, m = h & 1023u;
    // |x| * 2^24 = mant << (e - 1) for normal numbers, mant for subnormals
    const uint64_t mant = e ? (m | 1024u) : m;
    const int sh = e ? static_cast<int>(e) - 1 : 0;
    const unsigned __int128 sq = static_cast<unsigned __int128>(mant * mant) << (2 * sh);
    s += sq;
  }
  return s;
}

// Compare the exact sum (units 2^-48) with m^2, m > 0 a double holding at most
// 25 significant bits.  Returns -1, 0, +1 for S < m^2, S == m^2, S > m^2.
TQ_HD int compare_square(unsigned __int128 s, double m) {
  int e = 0;
  const double f = std::frexp(m, &e);               // m = f * 2^e, f in [0.5, 1)
  const uint64_t mm = static_cast<uint64_t>(std::ldexp(f, 25));  // exact: <= 25 bits
  const int sh = 2 * (e - 25) + 48;                 // m^2 = mm^2 * 2^(2(e-25)), S = s * 2^-48
  const unsigned __int128 mm2 = static_cast<unsigned __int128>(mm) * mm;
  if (sh >= 0) {
    if (sh > 77) return -1;                         // m^2 >= 2^127 units exceeds any sum of 128 fp16 squares
    const unsigned __int128 rhs = mm2 << sh;
    return s < rhs ? -1 : (s > rhs ? 1 : 0);
  }
  const int r = -sh;
  if (r >= 100) return 1;                           // m^2 below 2^-148: any nonzero S is larger
  if ((s >> (127 - r)) != 0) return 1;              // s << r would overflow: S is far larger
  const unsigned __int128 lhs = s << r;
  return lhs < mm2 ? -1 : (lhs > mm2 ? 1 : 0);
}

// Sum of squares of 2N fp16 values (N packed pairs) as an unevaluated pair
// h + l: the squares are exact in float32 and are added with TwoSum in two
// interleaved lanes, then the lanes are merged with one more TwoSum.
template <int N>
TQ_HD void norm_partial(const float2* xs, float& h_out, float& l_out) {
  float2 hi = make_float2(0.0f, 0.0f), lo = make_float2(0.0f, 0.0f);
#pragma unroll
  for (int j = 0; j < N; ++j) {
    const float2 x = xs[j];  // fp16 values (or their negatives: only squares are used)
    const float2 t = mul2(x, x);       // exact: 11-bit significands
    const float2 s = add2(hi, t);      // TwoSum(hi, t)
    const float2 bb = sub2(s, hi);
    const float2 e = add2(sub2(hi, sub2(s, bb)), sub2(t, bb));
    lo = add2(lo, e);
    hi = s;
  }
  const float h = fadd(hi.x, hi.y);
  const float hb = fsub(h, hi.x);
  const float he = fadd(fsub(hi.x, fsub(h, hb)), fsub(hi.y, hb));
  h_out = h;
  l_out = fadd(fadd(lo.x, lo.y), he);
}

// (h, l) += (h2, l2), the high parts with TwoSum.
TQ_HD void twosum_merge(float& h, float& l, float h2, float l2) {
  const float s = fadd(h, h2);
  const float bb = fsub(s, h);
  const float e = fadd(fsub(h, fsub(s, bb)), fsub(h2, bb));
  l = fadd(fadd(l, l2), e);
  h = s;
}

// Correctly rounded float32 of sqrt(h + l), h + l the sum of squares of the
// 128 fp16 values of `row` (64 packed pairs, read only in the rare exact path).
//
// n = sqrt(RN(h + l)) is within one ulp of the answer; the residual
// r = (h + l) - n^2 (n^2 split exactly with an FMA) decides between n and its
// neighbours by comparison with the rounding midpoints.  When r is within
// 2^-37 S of a midpoint the exact integer sum decides (ties to even).
//
// Why 2^-37 S suffices (u = 2^-24, every square exact in float32, all terms
// positive).  One TwoSum accumulator of 16 squares of total T: each step's
// error term e_j is exact and |e_j| <= u T, the float sum of the e_j adds at
// most u |lo_j| <= j u^2 T per step, 136 u^2 T in all.  The two accumulators of
// a lane merged (one TwoSum, two roundings of the low parts): 32 u^2 T more;
// each of the two merges across lanes: at most 80 u^2 S.  So h + l = S + E with
// |E| <= 328 u^2 S < 2^-39.6 S.  In r, h - p is exact (Sterbenz: p = RN(n^2) is
// within a factor 2 of h), l - pe and the final addition round at most 2 u^2 S
// and 2^-46 S, and t_up, t_dn round at most 2^-47 S: the float decision is
// wrong only if the exact r is within 2^-39.4 S of a midpoint, a quarter of the
// margin.  (A margin of 2^-30 S sent 3 % of the vectors to the exact sum.)
// Rare path of norm_from_sum (the float residual cannot tell n from a
// neighbour): compare the exact integer sum of squares with the squared
// midpoints.  Its loop is not unrolled and it runs after the vector's
// arithmetic (see norm_decided), so that it costs the per-token code nothing.
TQ_HD float norm_near_midpoint(float n, const uint32_t* row) {
  const float n_up = bitsf(fbits(n) + 1u), n_dn = bitsf(fbits(n) - 1u);
  const float u_up = fsub(n_up, n), u_dn = fsub(n, n_dn);
  const unsigned __int128 se = exact_sum_squares(row);
  const int cu = compare_square(se, static_cast<double>(n) + 0.5 * static_cast<double>(u_up));
  if (cu > 0 || (cu == 0 && (fbits(n_up) & 1u) == 0)) return n_up;
  const int cd = compare_square(se, static_cast<double>(n) - 0.5 * static_cast<double>(u_dn));
  if (cd < 0 || (cd == 0 && (fbits(n_dn) & 1u) == 0)) return n_dn;
  return n;
}

// The float32 norm as far as the float residual decides it: the correctly
// rounded result, or, when r lies within the margin of a rounding midpoint, the
// candidate n with `exact` set — the caller then takes norm_near_midpoint(n,
// row).  The quantizers use the candidate for the codes (it is within one ulp
// of the norm, so a code can differ only for a coordinate within a few ulps of
// a threshold) and settle the stored norm after the vector's arithmetic, where
// the integer path's registers meet no live vector registers.
TQ_HD float norm_decided(float h, float l, bool& exact) {
  exact = false;
  const float s_approx = fadd(h, l);
  if (!(s_approx > 0.0f)) return 0.0f;  // all zero (squares are >= 0)
  const float n = fsqrt(s_approx);
  const float p = fmul(n, n);
  const float pe = ffma(n, n, -p);      // n*n = p + pe exactly
  const float r = fadd(fsub(h, p), fsub(l, pe));
  const float n_up = bitsf(fbits(n) + 1u), n_dn = bitsf(fbits(n) - 1u);
  const float u_up = fsub(n_up, n), u_dn = fsub(n, n_dn);
  const float t_up = ffma(n, u_up, fmul(fmul(u_up, u_up), 0.25f));   // (n + u/2)^2 - n^2
  const float t_dn = ffma(n, u_dn, -fmul(fmul(u_dn, u_dn), 0.25f));  // n^2 - (n - u/2)^2
  const float margin = fmul(s_approx, 7.275957614183426e-12f);       // 2^-37 S
  const bool near_up = fabsf(fsub(r, t_up)) <= margin;
  const bool near_dn = fabsf(fadd(r, t_dn)) <= margin;
  if (!near_up && !near_dn) {
    if (r > t_up) return n_up;
    if (r < -t_dn) return n_dn;
    return n;
  }
  exact = true;
  return n;
}

TQ_HD float norm_from_sum(float h, float l, const uint32_t* row) {
  bool exact;
  const float n = norm_decided(h, l, exact);
  return exact ? norm_near_midpoint(n, row) : n;
}

// ---------------------------------------------------------------------------
// Threshold lookup: code = #{k : t_k <= y} through buckets RN(y * A)
// ---------------------------------------------------------------------------

struct LutEntry {
  float thr;      // the threshold inside this bucket, or +inf
  uint32_t base;  // number of thresholds in lower buckets
};

TQ_HD int lut_size(int a) { return 2 * a + 3; }

// Entry j covers bucket value j - (A + 1).  Buckets are RN(y * A), computed as
// fma(y, A, 1.5*2^23) whose bits sit 2^23 + 2^22 + bucket above those of the magic.
TQ_HD LutEntry lut_entry(const float* thr, int n_thr, int a, int j) {
  const int bucket = j - (a + 1);
  LutEntry e{INFINITY, 0u};
  for (int k = 0; k < n_thr; ++k) {
    const int bk = static_cast<int>(fbits(ffma(thr[k], static_cast<float>(a), kMagic)) - fbits(kMagic));
    if (bk < bucket) e.base += 1;
    if (bk == bucket) e.thr = thr[k];
  }
  return e;
}

// Walsh-Hadamard butterflies over index bits 0..4 of 32 values held as 16
// float2 (value 2m in .x, 2m+1 in .y): bit 0 inside each pair, bits 1..4
// between pairs with packed operations.
TQ_HD void fwht32(float2* v) {
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const float a = v[j].x, b = v[j].y;
    v[j] = make_float2(fadd(a, b), fsub(a, b));
  }
#pragma unroll
  for (int hb = 1; hb < 16; hb *= 2) {
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      if (j & hb) continue;
      const float2 a = v[j], b = v[j + hb];
      v[j] = add2(a, b);
      v[j + hb] = sub2(a, b);
    }
  }
}

// One butterfly stage between two holders of 32 values: the lower holder keeps
// own + other, the upper one other - own, as one fused multiply-add by
// sgn = (+1, +1) or (-1, -1): RN(own * (+-1) + other) is exactly the rounded
// sum or difference.
TQ_HD float2 butterfly_pair(float2 own, float2 other, float2 sgn) {
  return fma2(own, sgn, other);
}

// Codes of 32 rotated coordinates z (y = z * inv) packed LSB-first into BITS
// words.  code = base + (y >= thr) of the bucket RN(y * A) of a lookup table
// whose buckets hold at most one threshold (entries at lut[j * stride]).  Every
// finite coordinate has |y| <= 1 + 1/A, inside the table; the table index is
// clamped (unsigned) to the last entry so that any other input, even NaN, still
// reads inside the table.
template <int BITS>
TQ_HD void pack_codes32(const float2* z, float inv, const LutEntry* lut, int stride, int lut_a, uint32_t* words) {
  const float fa = static_cast<float>(lut_a);
  const uint32_t last = static_cast<uint32_t>(lut_size(lut_a) - 1);
  const uint32_t bias = fbits(kMagic) - static_cast<uint32_t>(lut_a + 1);
  uint32_t acc[BITS];
#pragma unroll
  for (int k = 0; k < BITS; ++k) acc[k] = 0u;
  float2 y2 = make_float2(0.0f, 0.0f), b2 = y2;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    if ((i & 1) == 0) {  // a pair of coordinates: scaled and bucketed with packed operations
      y2 = mul2(z[i >> 1], make_float2(inv, inv));
      b2 = fma2(y2, make_float2(fa, fa), make_float2(kMagic, kMagic));
    }
    const float y = (i & 1) ? y2.y : y2.x;
    const uint32_t raw = fbits((i & 1) ? b2.y : b2.x) - bias;
    const uint32_t idx = raw < last ? raw : last;
    const LutEntry e = lut[idx * stride];
    const uint32_t code = e.base + (y >= e.thr ? 1u : 0u);
    const int bit = i * BITS, word = bit >> 5, off = bit & 31;
    acc[word] += code * (1u << off);  // disjoint bit fields: one multiply-add inserts the code
    if (off + BITS > 32) acc[word + 1] += code >> (32 - off);
  }
#pragma unroll
  for (int k = 0; k < BITS; ++k) words[k] = acc[k];
}

// Sign masks of one KV head for 64 fp16 pairs: bit 15 for element 2j, bit 31 for 2j+1.
TQ_HD uint32_t sign_mask_pair(uint64_t seed, int layer, int head, int j) {
  return (sign_negative(seed, layer, head, 2 * j) ? 0x8000u : 0u) |
         (sign_negative(seed, layer, head, 2 * j + 1) ? 0x80000000u : 0u);
}

}  // namespace tq
