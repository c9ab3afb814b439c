// Weighted split of the decode tile list over the CTAs of the split-K kernel,
// shared by the split kernel (each CTA's tile range), the merge kernel (the CTAs
// whose partials a row combines) and a host verification hook.
//
// The tile list holds the rows r = v Hkv + h in order (v the work-list
// sequence, h the KV head); row r is tc(v) cold tiles followed by th(v) hot
// ones, starting at tile T_r.  A CTA pays for every segment (the cold or the hot
// tiles of one row) it starts: the row prologue (query rotation and fragments),
// the row exit (combine across warps, partial written) and a last round of tiles
// that not every warp gets.  On the long-context 3.5-bit decode that is a few us
// per segment against about 0.11 us per tile of a CTA, so an equal count of
// tiles per CTA left the CTAs that crossed a row end (two segment starts more)
// 7 % behind the rest.  Tiles are therefore priced, with the start prices kc of
// a cold and kh of a hot segment (in tiles),
//     cost(t) = t + kc (r + 1) + kh r        for a cold tile of row r,
//     cost(t) = t + kc (r + 1) + kh (r + 1)  for a hot tile of row r,
// a strictly increasing function of t with cost(total - 1) < C = total +
// (kc + kh) R (R rows), and CTA c of `grid` takes the tiles t with
// floor(cost(t) grid / C) = c: a contiguous range, the ranges in CTA order.
// With kc = kh = 0 the split is the plain equal count of tiles.
#pragma once

#include <cstdint>

#include "tq_signs.h"  // TQ_HD

namespace tq {

struct SplitPrice {
  long long cold, hot;  // start price of a cold and of a hot segment, in tiles (>= 0)
};

// C: one past the largest cost of a list of `total` tiles in `rows` rows.
TQ_HD long long split_total_cost(long long total, long long rows, SplitPrice k) {
  return total + (k.cold + k.hot) * rows;
}

// Least integer cost x with x grid >= c C: the first cost CTA c may take.
TQ_HD long long split_cost_at(long long C, int grid, int c) {
  return (static_cast<long long>(c) * C + grid - 1) / grid;
}

// Largest work-list sequence v (of nv) whose first cold tile costs at most tau,
// i.e. prefix[v] + (kc + kh) v hkv + kc <= tau; -1 if there is none.  prefix[v]
// is the number of tiles of the sequences before v.
TQ_HD int split_find_seq(const long long* prefix, int nv, int hkv, SplitPrice k, long long tau) {
  int lo = 0, hi = nv - 1, v = -1;
  while (lo <= hi) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] + (k.cold + k.hot) * mid * hkv + k.cold <= tau) {
      v = mid;
      lo = mid + 1;
    } else {
      hi = mid - 1;
    }
  }
  return v;
}

// Least tile of cost >= tau, given v = split_find_seq(...) >= 0 and tc, the cold
// tiles per row of sequence v.  The row r = v hkv + h is the last one whose first
// cold tile costs at most tau; within it the cold tiles cost base + kc + j and
// the hot ones base + kc + kh + j (j the tile's offset in the row, base = T_r +
// (kc + kh) r); past the row the next row's first tile is the answer.
TQ_HD long long split_tile_in_seq(const long long* prefix, int v, int hkv, int tc, SplitPrice k, long long tau) {
  const long long per_h = (prefix[v + 1] - prefix[v]) / hkv, step = per_h + k.cold + k.hot;
  const long long b0 = prefix[v] + (k.cold + k.hot) * v * hkv;  // base of the row h = 0
  long long h = step > 0 ? (tau - k.cold - b0) / step : hkv - 1;
  if (h > hkv - 1) h = hkv - 1;
  const long long t_row = prefix[v] + h * per_h, base = b0 + h * step;
  const long long jc = tau - base - k.cold;  // offset of the cold tile of cost tau
  if (jc < tc) return t_row + jc;
  const long long jh = tau - base - k.cold - k.hot;  // offset of the hot tile of cost tau
  if (jh <= tc) return t_row + tc;
  if (jh < per_h) return t_row + jh;
  return t_row + per_h;
}

// CTA of cost x (0 <= x < C): floor(x grid / C).  A float estimate of the
// quotient is off by at most one (relative error a few 2^-24, quotient below
// 2^10); exact 64-bit products correct it.
TQ_HD int split_cta(long long x, long long C, int grid) {
  const long long num = x * grid;
  int c = static_cast<int>(static_cast<float>(num) * (1.0f / static_cast<float>(C)));
  c = c < 0 ? 0 : (c > grid - 1 ? grid - 1 : c);
  if (static_cast<long long>(c) * C > num) --c;
  if (static_cast<long long>(c + 1) * C <= num) ++c;
  return c;
}

// Whether CTA c takes a tile whose cost lies in [a, b] (a <= b, the consecutive
// costs of one segment).  When C >= grid consecutive costs never skip a CTA, so
// every CTA from split_cta(a) to split_cta(b) does; below that a CTA may get no
// cost of the segment.
TQ_HD bool split_cta_hits(int c, long long a, long long b, long long C, int grid) {
  if (C >= grid) return true;
  long long x = split_cost_at(C, grid, c);
  if (x < a) x = a;
  return x <= b && x * grid < static_cast<long long>(c + 1) * C;
}

// First cost of the cold and of the hot tiles of row r, whose first tile is hbase.
TQ_HD long long split_cold_cost(long long hbase, long long r, SplitPrice k) {
  return hbase + k.cold * (r + 1) + k.hot * r;
}
TQ_HD long long split_hot_cost(long long hbase, int tc, long long r, SplitPrice k) {
  return hbase + tc + (k.cold + k.hot) * (r + 1);
}

}  // namespace tq
