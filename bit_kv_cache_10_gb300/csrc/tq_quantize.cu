// Quantize-and-append kernel (one launch for K and V of every head) and the
// hot-window evict pass.
//
// Work unit: a "job" is 16 consecutive tokens of one (tensor, batch, KV head).
// Each of the CTA's 32 warps loads its next job into its own padded
// shared-memory tile (272-byte rows) with cp.async as soon as it has finished
// the current one; the other resident warps hide the latency (more warps beat
// a second buffer: the kernel is bound by instruction fetch and issue, and
// 32 warps at 64 registers ran 20 % faster than 20 double-buffered warps at
// 96).  Four lanes share one token
// vector, lane q owning coordinates 32q..32q+31, so that eight vectors are in
// flight per warp step: exact norm (per-lane TwoSum partial sums merged across
// the four lanes), sign flip, FWHT over index bits 0..4 in registers and bits
// 5..6 with shuffles, bucketed threshold lookup, LSB-first packing of the
// lane's 32 codes into exactly `bits` words.
#include <cstring>

#include "tq_device.cuh"
#include "tq_launch.cuh"
#include "tq_internal.h"
#include "tq_debug.h"

namespace tq {
namespace {

constexpr int kWarps = 32;                  // warps per CTA (64 registers each: the register file)
constexpr int kRowBytes = 256;              // one fp16 vector
constexpr int kRowPitch = kRowBytes + 16;   // padded smem pitch
constexpr int kTileRows = 16;
constexpr int kTileBytes = kTileRows * kRowPitch;
constexpr int kLutCopies = 16;              // one LUT copy per lane of a half-warp
constexpr int kSignHeads = 16;              // KV heads whose rotation-sign masks a CTA tabulates once

struct QuantParams {
  const uint16_t* k_src;
  const uint16_t* v_src;
  int64_t stride_b, stride_h, stride_t;
  int n_new;
  const int* start_pos;
  const int* num_new;  // optional per-sequence counts
  int batch, heads, cap, hot;
  int k_mode, k_bits, v_bits;
  uint32_t* k_words;
  float* k_norms;
  uint16_t* k_fp16;
  uint32_t* v_words;
  float* v_norms;
  uint16_t* v_ring;
  RowMap map;  // cache row of (b, h, t): contiguous or through the block table
  uint32_t* status;
  uint64_t seed;
  int layer;
  float k_thr[15];
  float v_thr[15];
  int k_lut_a, v_lut_a;
  int evict;           // 0: append pass, 1: evict ring tokens that turn cold
  int fuse_evict;      // append pass of at most W tokens: each V job evicts its ring slots first
                       // (selects the FUSE variant of the kernel)
  int tiles_per_row;   // jobs per (tensor, batch, head)
  int tensors;         // 2 (K and V) for the append pass, 1 (V) for evict
  long long jobs;
};

struct Job {
  int tensor, b, h, tile;
  bool valid;          // the sequence's range is in bounds
  int start, end;      // append: positions [start, end); evict: [e0, e1)
  int count;           // rows this sequence appends
};

// Sequence fields of a job from its sequence b: append range or evict range.
__device__ __forceinline__ void job_sequence(const QuantParams& p, Job& jb) {
  const int s = p.start_pos[jb.b];
  const int cnt = p.num_new != nullptr ? p.num_new[jb.b] : p.n_new;
  jb.valid = s >= 0 && cnt >= 0 && cnt <= p.n_new && static_cast<long long>(s) + cnt <= p.cap;
  jb.count = cnt;
  if (!p.evict) {
    jb.start = s;
    jb.end = s + cnt;
  } else {
    const int end = s + cnt;
    jb.start = max(0, s - p.hot);
    jb.end = min(s, end - p.hot);
    if (jb.end < jb.start) jb.end = jb.start;
  }
}

// Mixed-radix digits (tensor, b, h, tile) of a job index: tile fastest, then
// head, then sequence, then tensor, so that at any moment nearly all warps run
// the same code width.  (The evict pass has one tensor digit, 0, and
// quantizes V: the walk keeps the digit and the loop sets jb.tensor = 1.)
__device__ __forceinline__ Job job_digits(const QuantParams& p, long long jl) {
  const int j = static_cast<int>(jl);  // the host keeps the job count below 2^31
  Job jb;
  const int rt = j / p.tiles_per_row;
  jb.tile = j - rt * p.tiles_per_row;
  const int bt = rt / p.heads;
  jb.h = rt - bt * p.heads;
  jb.tensor = bt / p.batch;
  jb.b = bt - jb.tensor * p.batch;
  return jb;
}

// jb + d in the mixed radix (every digit of d below its radix): at most one
// carry per digit.
__device__ __forceinline__ void job_advance(const QuantParams& p, Job& jb, const Job& d) {
  jb.tile += d.tile;
  int c = jb.tile >= p.tiles_per_row;
  if (c) jb.tile -= p.tiles_per_row;
  jb.h += d.h + c;
  c = jb.h >= p.heads;
  if (c) jb.h -= p.heads;
  jb.b += d.b + c;
  c = jb.b >= p.batch;
  if (c) jb.b -= p.batch;
  jb.tensor += d.tensor + c;
}

// Whether tile row `row` of a job holds a token (its cache position in *pos_out).
__device__ __forceinline__ bool row_present(const QuantParams& p, const Job& jb, int row, int* pos_out) {
  const int t = jb.tile * kTileRows + row;
  const int pos = jb.start + t;
  *pos_out = pos;
  return p.evict ? pos < jb.end : t < jb.count;
}

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }

__device__ __forceinline__ void issue_tile(const QuantParams& p, const Job& jb, uint8_t* tile, int lane) {
  if (!jb.valid) return;
  const int row0 = lane >> 4, col = lane & 15;
  uint8_t* dst = tile + row0 * kRowPitch + col * 16;
  if (!p.evict) {
    // rows t = 16 tile + 2k + row0 of the source, 2 stride_t apart
    const int t0 = jb.tile * kTileRows + row0;
    const uint16_t* src = (jb.tensor == 0 ? p.k_src : p.v_src) + jb.b * p.stride_b + jb.h * p.stride_h +
                          static_cast<int64_t>(t0) * p.stride_t + col * 8;
    const int64_t step = 2 * p.stride_t;
#pragma unroll
    for (int k = 0; k < kTileRows / 2; ++k)
      if (t0 + 2 * k < jb.count) cp_async16(dst + 2 * k * kRowPitch, src + k * step);
    return;
  }
  const uint16_t* ring = p.v_ring + (static_cast<int64_t>(jb.b) * p.heads + jb.h) * p.hot * D + col * 8;
#pragma unroll
  for (int k = 0; k < kTileRows / 2; ++k) {
    const int pos = jb.start + jb.tile * kTileRows + 2 * k + row0;
    if (pos < jb.end) cp_async16(dst + 2 * k * kRowPitch, ring + (pos % p.hot) * D);
  }
}

// One step: 8 vectors (a staged tile row or a ring row in global memory; rowp
// is the lane's vector), lane = v + 8 q.
template <int BITS>
__device__ __forceinline__ void quantize_step(const uint8_t* rowp, int q, const uint32_t* smask,
                                              const LutEntry* lut, int lut_a, uint32_t* dst_words, float* dst_norm,
                                              bool store) {
  const uint4* src = reinterpret_cast<const uint4*>(rowp) + 4 * q;
  const uint4* msk = reinterpret_cast<const uint4*>(smask) + 4 * q;
  float2 v[16];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint4 a = src[k], m = msk[k];
    v[4 * k] = half2_bits_to_float2(a.x ^ m.x);
    v[4 * k + 1] = half2_bits_to_float2(a.y ^ m.y);
    v[4 * k + 2] = half2_bits_to_float2(a.z ^ m.z);
    v[4 * k + 3] = half2_bits_to_float2(a.w ^ m.w);
  }
  // norm: per-lane partial sums, merged over the 4 lanes of the vector (q ^ 1, then q ^ 2)
  float h, l;
  norm_partial<16>(v, h, l);  // squares of the sign-flipped values
  twosum_merge(h, l, __shfl_xor_sync(0xffffffffu, h, 8), __shfl_xor_sync(0xffffffffu, l, 8));
  twosum_merge(h, l, __shfl_xor_sync(0xffffffffu, h, 16), __shfl_xor_sync(0xffffffffu, l, 16));
  bool exact;  // the rare exact norm is settled after the vector's arithmetic (see norm_decided)
  const float n = norm_decided(h, l, exact);
  // rotation: in-lane bits 0..4, then bits 5 (q ^ 1) and 6 (q ^ 2) across lanes
  fwht32(v);
  // the two halves of a pair are exchanged as two 32-bit values (no 64-bit packing)
  const float s1 = (q & 1) ? -1.0f : 1.0f, s2 = (q & 2) ? -1.0f : 1.0f;
  auto xchg = [](float2 a, int m) {
    return make_float2(__shfl_xor_sync(0xffffffffu, a.x, m), __shfl_xor_sync(0xffffffffu, a.y, m));
  };
#pragma unroll
  for (int j = 0; j < 16; ++j) v[j] = butterfly_pair(v[j], xchg(v[j], 8), make_float2(s1, s1));
#pragma unroll
  for (int j = 0; j < 16; ++j) v[j] = butterfly_pair(v[j], xchg(v[j], 16), make_float2(s2, s2));
  const float inv = n > 0.0f ? frcp(fmul(n, kSqrtD)) : 0.0f;
  uint32_t words[BITS];
  pack_codes32<BITS>(v, inv, lut, kLutCopies, lut_a, words);
  if (store) {
    uint32_t* d = dst_words + q * BITS;
    if constexpr (BITS == 4) {
      *reinterpret_cast<uint4*>(d) = make_uint4(words[0], words[1], words[2], words[3]);
    } else if constexpr (BITS == 2) {
      *reinterpret_cast<uint2*>(d) = make_uint2(words[0], words[1]);
    } else {
#pragma unroll
      for (int k = 0; k < BITS; ++k) d[k] = words[k];
    }
  }
  if (store && q == 0) *dst_norm = exact ? norm_near_midpoint(n, reinterpret_cast<const uint32_t*>(rowp)) : n;
}

// Code of x in the int8 mode for a scale s > 0: the float32 quotient x / s
// (IEEE division) rounded to the nearest integer, ties to even, clamped to
// [-127, 127].
__device__ __forceinline__ uint32_t int8_code(float x, float s) {
  const int c = __float2int_rn(__fdiv_rn(x, s));
  return static_cast<uint32_t>(min(127, max(-127, c)));
}

// One step of the int8 mode ([mlxcel doc] "Available modes": per-token INT8
// absmax): 8 vectors with the lane decomposition of quantize_step
// (lane q holds coordinates 32q .. 32q + 31).  s = fp32(max |x_i|) / 127,
// code_i = int8_code(x_i, s); a zero vector gets s = 0 and zero codes.  The
// lane packs its 32 codes into 8 words, code i in byte i mod 4.
__device__ __forceinline__ void quantize_step_int8(const uint8_t* rowp, int q, uint32_t* dst_words, float* dst_scale,
                                                   bool store) {
  const uint4* src = reinterpret_cast<const uint4*>(rowp) + 4 * q;
  uint32_t w[16];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint4 a = src[k];
    w[4 * k] = a.x;
    w[4 * k + 1] = a.y;
    w[4 * k + 2] = a.z;
    w[4 * k + 3] = a.w;
  }
  // the magnitudes of finite fp16 values order like their bits without the sign
  uint32_t m = 0u;
#pragma unroll
  for (int k = 0; k < 16; ++k) m = __vmaxu2(m, w[k] & 0x7FFF7FFFu);
  m = max(m & 0xFFFFu, m >> 16);
  m = max(m, __shfl_xor_sync(0xffffffffu, m, 8));
  m = max(m, __shfl_xor_sync(0xffffffffu, m, 16));
  const float s = __fdiv_rn(half_bits_to_float(m), 127.0f);
  uint32_t words[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const float2 a = half2_bits_to_float2(w[2 * k]), b = half2_bits_to_float2(w[2 * k + 1]);
    uint32_t word = 0u;
    if (s > 0.0f) {
      const uint32_t lo = __byte_perm(int8_code(a.x, s), int8_code(a.y, s), 0x0040);
      const uint32_t hi = __byte_perm(int8_code(b.x, s), int8_code(b.y, s), 0x0040);
      word = __byte_perm(lo, hi, 0x5410);
    }
    words[k] = word;
  }
  if (store) {
    uint4* d = reinterpret_cast<uint4*>(dst_words + 8 * q);
    d[0] = make_uint4(words[0], words[1], words[2], words[3]);
    d[1] = make_uint4(words[4], words[5], words[6], words[7]);
    if (q == 0) *dst_scale = s;
  }
}

// PLAIN: contiguous layout, no hot window, packed or int8 K, append pass: no row
// goes to the ring or to an fp16 copy, so the step needs neither test.
template <bool PAGED, bool FUSE, bool PLAIN = false>
__global__ void __launch_bounds__(kWarps * 32, 1) quantize_append_kernel(const QuantParams p) {
  asm volatile("griddepcontrol.launch_dependents;\n");  // the next grid may start its prologue
  extern __shared__ __align__(16) uint8_t smem[];
  const int lut_k_n = p.k_lut_a ? lut_size(p.k_lut_a) : 0;
  const int lut_v_n = p.v_lut_a ? lut_size(p.v_lut_a) : 0;  // 0: int8 mode
  LutEntry* lut_k = reinterpret_cast<LutEntry*>(smem);
  LutEntry* lut_v = lut_k + lut_k_n * kLutCopies;
  // rotation-sign masks of every KV head (64 words each) when there are at most
  // kSignHeads heads, else each warp computes its job's head into its own area
  uint32_t* sign_tab = reinterpret_cast<uint32_t*>(lut_v + lut_v_n * kLutCopies);
  const bool tab_signs = p.heads <= kSignHeads && p.k_mode != TQ_KV_INT8;
  uint8_t* warp_area = reinterpret_cast<uint8_t*>(sign_tab + kSignHeads * 64);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int vrow = lane & 7, q = lane >> 3;
  uint8_t* tiles = warp_area + warp * (kTileBytes + 256);
  uint32_t* smask = reinterpret_cast<uint32_t*>(tiles + kTileBytes);

  // threshold lookup tables, kLutCopies interleaved copies (entry j of copy c at
  // j*copies + c): each entry is computed once and written to its copies
  for (int j = threadIdx.x; j < lut_k_n + lut_v_n; j += blockDim.x) {
    const bool is_k = j < lut_k_n;
    const LutEntry e = is_k ? lut_entry(p.k_thr, (1 << p.k_bits) - 1, p.k_lut_a, j)
                            : lut_entry(p.v_thr, (1 << p.v_bits) - 1, p.v_lut_a, j - lut_k_n);
    uint4* dst = reinterpret_cast<uint4*>(lut_k + j * kLutCopies);  // lut_v follows lut_k
    const uint4 two = make_uint4(__float_as_uint(e.thr), e.base, __float_as_uint(e.thr), e.base);
#pragma unroll
    for (int c = 0; c < kLutCopies / 2; ++c) dst[c] = two;
  }
  if (tab_signs)
    for (int i = threadIdx.x; i < p.heads * 64; i += blockDim.x)
      sign_tab[i] = sign_mask_pair(p.seed, p.layer, i >> 6, i & 63);
  __syncthreads();
  // launched as a programmatic dependent grid: everything above uses only the
  // parameters; wait here for the preceding grid (it may produce the inputs or
  // still read the ring slots this launch overwrites)
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  const LutEntry* my_lut_k = lut_k + (lane & (kLutCopies - 1));
  const LutEntry* my_lut_v = lut_v + (lane & (kLutCopies - 1));

  // job j goes to CTA j mod grid: small appends put one job per SM.  The
  // warp's jobs are stride apart, walked in the mixed radix of job_digits
  const long long stride = static_cast<long long>(gridDim.x) * kWarps;
  const Job dstep = job_digits(p, stride < p.jobs ? stride : 0);
  long long j = static_cast<long long>(warp) * gridDim.x + blockIdx.x;
  Job next{};  // the job whose tile is in flight
  if (j < p.jobs) {
    next = job_digits(p, j);
    const int digit = next.tensor;
    if (p.evict) next.tensor = 1;
    job_sequence(p, next);
    issue_tile(p, next, tiles, lane);
    next.tensor = digit;
  }
  cp_async_commit();
  for (; j < p.jobs; j += stride) {
    asm volatile("cp.async.wait_all;\n" ::);
    __syncwarp();

    Job jb = next;
    const int digit = jb.tensor;
    if (p.evict) jb.tensor = 1;  // 0 = K, 1 = V
    if (!jb.valid) {
      if (jb.tile == 0 && jb.tensor == (p.evict ? 1 : 0) && jb.h == 0 && lane == 0 && p.status != nullptr)
        atomicOr(p.status, TQ_DEV_ERR_APPEND_RANGE);
    } else {
      const uint32_t* msk = tab_signs ? sign_tab + jb.h * 64 : smask;  // rotation-sign masks of this head
      if (!tab_signs && p.k_mode != TQ_KV_INT8) {
        smask[lane] = sign_mask_pair(p.seed, p.layer, jb.h, lane);
        smask[lane + 32] = sign_mask_pair(p.seed, p.layer, jb.h, lane + 32);
      }
      __syncwarp();
      const uint8_t* tile = tiles;
      const bool k_tensor = jb.tensor == 0;
      const bool copy_k = !PLAIN && k_tensor && p.k_mode == TQ_K_FP16;
      int cold_end = 1 << 30;
      if (!PLAIN && !k_tensor && p.hot > 0 && !p.evict) cold_end = jb.end - min(p.hot, jb.end);
      auto quantize_row = [&](const uint8_t* rowp, int bits, const LutEntry* lut, int lut_a, uint32_t* dw, float* dn,
                              bool store) {
        switch (bits) {
          case 8: quantize_step_int8(rowp, q, dw, dn, store); break;
          case 2: quantize_step<2>(rowp, q, msk, lut, lut_a, dw, dn, store); break;
          case 3: quantize_step<3>(rowp, q, msk, lut, lut_a, dw, dn, store); break;
          default: quantize_step<4>(rowp, q, msk, lut, lut_a, dw, dn, store); break;
        }
      };
#pragma unroll 1
      for (int step = 0; step < kTileRows / 8; ++step) {
        const int row = 8 * step + vrow;
        int pos = 0;
        bool have;
        if constexpr (PLAIN) {
          pos = jb.start + jb.tile * kTileRows + row;
          have = jb.tile * kTileRows + row < jb.count;
        } else {
          have = row_present(p, jb, row, &pos);
        }
        if (!__any_sync(0xffffffffu, have)) break;  // rows are filled in order: no later step has one
        long long ridx = (static_cast<long long>(jb.b) * p.heads + jb.h) * p.cap + pos;  // cache row
        if constexpr (PAGED) ridx = have ? p.map.row(jb.b, jb.h, pos) : 0;  // through the block table
        const bool to_copy = !PLAIN && (copy_k || (!k_tensor && pos >= cold_end));
        const bool to_ring = !copy_k && to_copy;  // hot V goes to the per-sequence ring, not the pool
        if constexpr (PAGED)
          if (have && ridx < 0 && !to_ring && p.status != nullptr) atomicOr(p.status, TQ_DEV_ERR_BLOCK);
        const bool in_pool = !PAGED || ridx >= 0;  // contiguous rows always are
        const int64_t slot = (static_cast<int64_t>(jb.b) * p.heads + jb.h) * p.hot + (p.hot > 0 ? pos % p.hot : 0);
        if (FUSE && !k_tensor) {
          // appends of at most W tokens: the ring slot this row takes holds
          // position pos - W, which turns cold now; it is quantized from the
          // ring before the slot is overwritten below (one job owns the slot)
          const int old = pos - p.hot;
          long long oidx = (static_cast<long long>(jb.b) * p.heads + jb.h) * p.cap + old;
          if constexpr (PAGED) oidx = have && old >= 0 ? p.map.row(jb.b, jb.h, old) : 0;
          const bool ev = have && old >= 0;
          if (ev && oidx < 0 && p.status != nullptr) atomicOr(p.status, TQ_DEV_ERR_BLOCK);
          if (__any_sync(0xffffffffu, ev && oidx >= 0)) {
            const uint8_t* src = ev ? reinterpret_cast<const uint8_t*>(p.v_ring + slot * D) : tile + row * kRowPitch;
            quantize_row(src, p.v_bits, my_lut_v, p.v_lut_a, p.v_words + oidx * (p.v_bits * 4), p.v_norms + oidx,
                         ev && oidx >= 0);
          }
          __syncwarp();
        }
        if (to_copy && have && (to_ring || in_pool)) {
          // fp16 copy of the row (asym K, or V going to the hot ring): 4 x 16 bytes per lane
          uint4* dst = copy_k ? reinterpret_cast<uint4*>(p.k_fp16 + ridx * D)
                              : reinterpret_cast<uint4*>(p.v_ring + slot * D);
          const uint4* src = reinterpret_cast<const uint4*>(tile + row * kRowPitch);
#pragma unroll
          for (int k = 0; k < 4; ++k) dst[4 * q + k] = src[4 * q + k];
        }
        if (copy_k) continue;  // uniform over the warp (the whole job is fp16 K)
        // every lane takes part in the shuffles of quantize_step; rows that are
        // absent or go to the ring are computed but not stored (a step with no
        // stored row is skipped)
        const bool store = have && !to_copy && in_pool;
        if (!__any_sync(0xffffffffu, store)) continue;
        const int bits = k_tensor ? p.k_bits : p.v_bits;
        quantize_row(tile + row * kRowPitch, bits, k_tensor ? my_lut_k : my_lut_v, k_tensor ? p.k_lut_a : p.v_lut_a,
                     (k_tensor ? p.k_words : p.v_words) + ridx * (bits * 4), (k_tensor ? p.k_norms : p.v_norms) + ridx,
                     store);
      }
    }
    __syncwarp();
    if (j + stride < p.jobs) {
      next = jb;
      next.tensor = digit;
      job_advance(p, next, dstep);
      const int nd = next.tensor;
      if (p.evict) next.tensor = 1;
      if (next.b != jb.b || next.tensor != jb.tensor) job_sequence(p, next);
      issue_tile(p, next, tiles, lane);
      next.tensor = nd;
    }
    cp_async_commit();
  }
  asm volatile("cp.async.wait_all;\n" ::);
}

// ---------------------------------------------------------------------------
// Small appends (at most kSmallMax tokens per sequence: the decode step's one
// token).  The latency of one quantized vector is then the critical path, so
// one warp takes one token vector, lane l holding coordinates 4l..4l+3.  The
// arithmetic is that of quantize_step stage for stage (exact norm, sign flip,
// FWHT over index bits 0..6 in that order, the same scaling; the code is the
// same count of thresholds, found by binary search instead of the bucketed
// table, which this kernel need not build), so the stored words and norms are
// the same.
// ---------------------------------------------------------------------------
int sm_count_q();
constexpr int kSmallMax = 16;   // tokens per sequence appended by the small-append kernel
constexpr int kSmallWarps = 2;  // warps (token vectors in flight) per CTA: small enough to share
                                // an SM with a decode CTA

// Lane l's 4 BITS-bit codes sit at stream offset 4 l BITS; word w of the token
// is the OR of the lanes' contributions to it, and lane w stores it.
template <int BITS>
__device__ __forceinline__ void store_codes_warp(uint32_t val, int lane, uint32_t* dst, bool store) {
  constexpr int kW = 4 * BITS;  // words of a d = 128 vector
  const int off = 4 * BITS * lane;
  const int lo = off >> 5;
  const uint64_t c = static_cast<uint64_t>(val) << (off & 31);
  const uint32_t c_lo = static_cast<uint32_t>(c), c_hi = static_cast<uint32_t>(c >> 32);
  uint32_t mine = 0u;
#pragma unroll
  for (int w = 0; w < kW; ++w) {
    const uint32_t word = __reduce_or_sync(0xffffffffu, (lo == w ? c_lo : 0u) | (lo + 1 == w ? c_hi : 0u));
    if (lane == w) mine = word;
  }
  if (store && lane < kW) dst[lane] = mine;
}

// Code of y: the number of float32 thresholds t_k <= y, by binary search over
// the 2^BITS - 1 sorted thresholds (the same count the bucketed table gives).
template <int BITS>
__device__ __forceinline__ uint32_t threshold_code(float y, const float* thr) {
  uint32_t lo = 0u;
#pragma unroll
  for (int step = 1 << (BITS - 1); step > 0; step >>= 1)
    if (y >= thr[lo + step - 1]) lo += step;
  return lo;
}

// One token vector per warp: x = the lane's 4 fp16 values, sm = their sign
// masks, row = the vector in memory (read only by the rare exact-norm path),
// thr = the codebook's thresholds.
template <int BITS>
__device__ __forceinline__ void quantize_vector_warp(const uint16_t* row, uint2 x, uint2 sm, const float* thr,
                                                     uint32_t* dst_words, float* dst_norm, bool store, int lane) {
  float2 v[2] = {half2_bits_to_float2(x.x ^ sm.x), half2_bits_to_float2(x.y ^ sm.y)};
  float h, l;
  norm_partial<2>(v, h, l);
#pragma unroll
  for (int m = 1; m < 32; m <<= 1)
    twosum_merge(h, l, __shfl_xor_sync(0xffffffffu, h, m), __shfl_xor_sync(0xffffffffu, l, m));
  bool exact;  // the rare exact norm is settled after the vector's arithmetic (see norm_decided)
  const float n = norm_decided(h, l, exact);
  // FWHT: index bits 0 and 1 inside the lane, bits 2..6 across lanes (lane bit k - 2)
  float z[4];
  {
    const float a0 = fadd(v[0].x, v[0].y), a1 = fsub(v[0].x, v[0].y);
    const float a2 = fadd(v[1].x, v[1].y), a3 = fsub(v[1].x, v[1].y);
    z[0] = fadd(a0, a2);
    z[1] = fadd(a1, a3);
    z[2] = fsub(a0, a2);
    z[3] = fsub(a1, a3);
  }
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float o = __shfl_xor_sync(0xffffffffu, z[k], m);
      z[k] = upper ? fsub(o, z[k]) : fadd(z[k], o);
    }
  }
  const float inv = n > 0.0f ? frcp(fmul(n, kSqrtD)) : 0.0f;
  uint32_t val = 0u;
#pragma unroll
  for (int k = 0; k < 4; ++k) val |= threshold_code<BITS>(fmul(z[k], inv), thr) << (BITS * k);
  store_codes_warp<BITS>(val, lane, dst_words, store);
  if (store && lane == 0) *dst_norm = exact ? norm_near_midpoint(n, reinterpret_cast<const uint32_t*>(row)) : n;
}

// The int8 mode for one token vector per warp (arithmetic of quantize_step_int8).
__device__ __forceinline__ void quantize_vector_warp_int8(uint2 x, uint32_t* dst_words, float* dst_scale, bool store,
                                                          int lane) {
  uint32_t m = __vmaxu2(x.x & 0x7FFF7FFFu, x.y & 0x7FFF7FFFu);
  m = __reduce_max_sync(0xffffffffu, max(m & 0xFFFFu, m >> 16));
  const float s = __fdiv_rn(half_bits_to_float(m), 127.0f);
  const float2 a = half2_bits_to_float2(x.x), b = half2_bits_to_float2(x.y);
  uint32_t word = 0u;
  if (s > 0.0f) {
    const uint32_t lo = __byte_perm(int8_code(a.x, s), int8_code(a.y, s), 0x0040);
    const uint32_t hi = __byte_perm(int8_code(b.x, s), int8_code(b.y, s), 0x0040);
    word = __byte_perm(lo, hi, 0x5410);
  }
  if (store) {
    dst_words[lane] = word;
    if (lane == 0) *dst_scale = s;
  }
}

template <bool PAGED>
__global__ void __launch_bounds__(kSmallWarps * 32) quantize_small_kernel(const QuantParams p) {
  asm volatile("griddepcontrol.launch_dependents;\n");
  __shared__ float thr_s[2][16];  // K and V thresholds
  if (threadIdx.x < 32) thr_s[threadIdx.x >> 4][threadIdx.x & 15] = (threadIdx.x & 15) < 15
      ? (threadIdx.x < 16 ? p.k_thr[threadIdx.x & 15] : p.v_thr[threadIdx.x & 15]) : INFINITY;
  __syncthreads();
  asm volatile("griddepcontrol.wait;\n" ::: "memory");  // the inputs and the ring may come from the previous grid
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long per_tensor = static_cast<long long>(p.batch) * p.heads * p.n_new;
  for (long long vi = static_cast<long long>(blockIdx.x) * kSmallWarps + warp; vi < 2 * per_tensor;
       vi += static_cast<long long>(gridDim.x) * kSmallWarps) {
    const int tensor = vi >= per_tensor ? 1 : 0;  // 0 = K, 1 = V
    const long long r = vi - tensor * per_tensor;
    const int t = static_cast<int>(r % p.n_new);
    const int bh = static_cast<int>(r / p.n_new);
    const int b = bh / p.heads, h = bh - b * p.heads;
    // the input row does not depend on the start position: its load overlaps that one
    const uint16_t* src = (tensor ? p.v_src : p.k_src) + b * p.stride_b + h * p.stride_h + t * p.stride_t;
    const uint2 x = reinterpret_cast<const uint2*>(src)[lane];
    const int s = p.start_pos[b];
    const int cnt = p.num_new != nullptr ? p.num_new[b] : p.n_new;
    if (!(s >= 0 && cnt >= 0 && cnt <= p.n_new && static_cast<long long>(s) + cnt <= p.cap)) {
      if (t == 0 && h == 0 && tensor == 0 && lane == 0 && p.status != nullptr)
        atomicOr(p.status, TQ_DEV_ERR_APPEND_RANGE);
      continue;
    }
    if (t >= cnt) continue;
    const int pos = s + t;
    if (tensor == 0 && p.k_mode == TQ_K_FP16) {  // asym K: stored verbatim
      const long long ridx = PAGED ? p.map.row(b, h, pos) : (static_cast<long long>(b) * p.heads + h) * p.cap + pos;
      if (ridx < 0) {
        if (lane == 0 && p.status != nullptr) atomicOr(p.status, TQ_DEV_ERR_BLOCK);
      } else {
        reinterpret_cast<uint2*>(p.k_fp16 + ridx * D)[lane] = x;
      }
      continue;
    }
    const uint2 sm = p.k_mode == TQ_KV_INT8 ? make_uint2(0u, 0u)
                                            : make_uint2(sign_mask_pair(p.seed, p.layer, h, 2 * lane),
                                                         sign_mask_pair(p.seed, p.layer, h, 2 * lane + 1));
    // what to quantize: the new row, or for V with a hot window the ring row
    // position pos - W leaves (the new row takes its slot: at most W tokens
    // are appended, so one vector owns each slot)
    const uint16_t* qrow = src;
    uint2 qx = x;
    int qpos = pos;
    uint16_t* ring = nullptr;
    if (tensor == 1 && p.hot > 0) {
      ring = p.v_ring + ((static_cast<int64_t>(b) * p.heads + h) * p.hot + pos % p.hot) * D;
      qpos = pos - p.hot;
      qrow = ring;
      qx = qpos >= 0 ? reinterpret_cast<const uint2*>(ring)[lane] : make_uint2(0u, 0u);
    }
    if (qpos >= 0) {
      const long long ridx = PAGED ? p.map.row(b, h, qpos) : (static_cast<long long>(b) * p.heads + h) * p.cap + qpos;
      if (ridx < 0 && lane == 0 && p.status != nullptr) atomicOr(p.status, TQ_DEV_ERR_BLOCK);
      const int bits = tensor ? p.v_bits : p.k_bits;
      const float* thr = thr_s[tensor];
      uint32_t* dw = (tensor ? p.v_words : p.k_words) + (ridx < 0 ? 0 : ridx) * (bits * 4);
      float* dn = (tensor ? p.v_norms : p.k_norms) + (ridx < 0 ? 0 : ridx);
      const bool store = ridx >= 0;
      switch (bits) {
        case 8: quantize_vector_warp_int8(qx, dw, dn, store, lane); break;
        case 2: quantize_vector_warp<2>(qrow, qx, sm, thr, dw, dn, store, lane); break;
        case 3: quantize_vector_warp<3>(qrow, qx, sm, thr, dw, dn, store, lane); break;
        default: quantize_vector_warp<4>(qrow, qx, sm, thr, dw, dn, store, lane); break;
      }
    }
    if (ring != nullptr) {  // the slot's old row has been read (and quantized)
      __syncwarp();
      reinterpret_cast<uint2*>(ring)[lane] = x;
    }
  }
}

tq_status launch_small(const QuantParams& p, cudaStream_t stream) {
  const bool paged = p.map.table != nullptr;
  auto kern = paged ? quantize_small_kernel<true> : quantize_small_kernel<false>;
  const int sms = sm_count_q();
  if (sms <= 0) return TQ_ERR_CUDA;
  const long long vectors = 2ll * p.batch * p.heads * p.n_new;
  const long long want = (vectors + kSmallWarps - 1) / kSmallWarps;
  const int grid = static_cast<int>(want < 4ll * sms ? want : 4ll * sms);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kSmallWarps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see griddepcontrol.wait
  attr[0].val.programmaticStreamSerializationAllowed = kProgrammaticLaunch;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, p) != cudaSuccess) return TQ_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

size_t quant_smem_bytes(int k_lut_a, int v_lut_a) {
  const size_t luts = (static_cast<size_t>(k_lut_a ? lut_size(k_lut_a) : 0) + (v_lut_a ? lut_size(v_lut_a) : 0)) *
                      kLutCopies * sizeof(LutEntry);
  return luts + kSignHeads * 64 * sizeof(uint32_t) + static_cast<size_t>(kWarps) * (kTileBytes + 256);
}

int sm_count_q() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

tq_status launch_quantize(QuantParams& p, cudaStream_t stream) {
  if (p.jobs <= 0) return TQ_OK;
  const size_t smem = quant_smem_bytes(p.k_lut_a, p.v_lut_a);
  const bool paged = p.map.table != nullptr;
  const bool plain = !paged && !p.fuse_evict && p.hot == 0 && !p.evict && p.k_mode != TQ_K_FP16;
  auto kern = paged ? (p.fuse_evict ? quantize_append_kernel<true, true> : quantize_append_kernel<true, false>)
                    : (p.fuse_evict ? quantize_append_kernel<false, true>
                                    : (plain ? quantize_append_kernel<false, false, true> : quantize_append_kernel<false, false>));
  // one memo per kernel above; a launch that needs more shared memory than the
  // limit set so far is refused once and retried with the limit raised
  static KernelMemo memos[5];
  KernelMemo& memo = memos[paged ? (p.fuse_evict ? 0 : 1) : (p.fuse_evict ? 2 : (plain ? 3 : 4))];
  const int sms = sm_count_q();
  if (sms <= 0) return TQ_ERR_CUDA;
  const int grid = static_cast<int>(p.jobs < sms ? p.jobs : sms);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kWarps * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see griddepcontrol.wait
  attr[0].val.programmaticStreamSerializationAllowed = kProgrammaticLaunch;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (launch_with_limit(kern, static_cast<int>(smem), memo, current_device(), cfg, p) != cudaSuccess)
    return TQ_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

}  // namespace
}  // namespace tq

extern "C" tq_status tq_quantize_append(const tq_cache_desc* d, const void* k_new, const void* v_new,
                                        int64_t stride_b, int64_t stride_h, int64_t stride_t, int32_t n_new,
                                        const int32_t* d_start_pos, const int32_t* d_num_new,
                                        tq_stream_t stream) {
  using namespace tq;
  const tq_status vs = validate_desc(d);
  if (vs != TQ_OK) return vs;
  if (n_new < 0) return TQ_ERR_INVALID_ARG;
  if (n_new == 0) return TQ_OK;
  if (n_new > d->capacity) return TQ_ERR_CAPACITY;
  if (k_new == nullptr || v_new == nullptr || d_start_pos == nullptr) return TQ_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new)) return TQ_ERR_INVALID_ARG;
  if (stride_b < 0 || stride_h < 0 || stride_t < 0 || (stride_b % 8) || (stride_h % 8) || (stride_t % 8))
    return TQ_ERR_INVALID_ARG;

  if (static_cast<long long>(d->batch) * d->num_kv_heads * ((n_new + kTileRows - 1) / kTileRows) * 2 >= (1ll << 31))
    return TQ_ERR_UNSUPPORTED;  // job indices are 32-bit

  QuantParams p;
  std::memset(&p, 0, sizeof(p));
  p.k_src = static_cast<const uint16_t*>(k_new);
  p.v_src = static_cast<const uint16_t*>(v_new);
  p.stride_b = stride_b;
  p.stride_h = stride_h;
  p.stride_t = stride_t;
  p.n_new = n_new;
  p.start_pos = d_start_pos;
  p.num_new = d_num_new;
  p.batch = d->batch;
  p.heads = d->num_kv_heads;
  p.cap = d->capacity;
  p.hot = d->hot_window;
  p.k_mode = d->k_mode;
  p.k_bits = d->k_mode == TQ_K_FP16 ? 0 : d->k_bits;  // 8 in the int8 mode
  p.v_bits = d->v_bits;
  p.k_words = static_cast<uint32_t*>(d->k_cache);
  p.k_norms = d->k_norms;
  p.k_fp16 = static_cast<uint16_t*>(d->k_cache);
  p.v_words = static_cast<uint32_t*>(d->v_cache);
  p.v_norms = d->v_norms;
  p.v_ring = static_cast<uint16_t*>(d->v_hot);
  p.map = make_row_map(d);
  p.status = d->d_status;
  p.seed = d->seed;
  p.layer = d->layer;
  if (d->k_mode == TQ_K_PACKED) {
    std::memcpy(p.k_thr, d->k_cb.thresholds, sizeof(p.k_thr));
    p.k_lut_a = quant_lut_scale(d->k_cb.thresholds, (1 << d->k_bits) - 1);
  }
  if (d->k_mode != TQ_KV_INT8) {
    std::memcpy(p.v_thr, d->v_cb.thresholds, sizeof(p.v_thr));
    p.v_lut_a = quant_lut_scale(d->v_cb.thresholds, (1 << d->v_bits) - 1);
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  if (n_new <= kSmallMax && (d->hot_window == 0 || n_new <= d->hot_window)) return launch_small(p, s);
  // V tokens leaving the ring are quantized before their slots are reused: by the
  // append launch itself when at most W tokens are appended (every slot is then
  // taken by one new row, whose job evicts it first), else by a launch before it
  p.fuse_evict = d->hot_window > 0 && n_new <= d->hot_window;
  if (d->hot_window > 0 && !p.fuse_evict) {
    QuantParams e = p;
    e.evict = 1;
    e.tensors = 1;
    const int most = n_new < d->hot_window ? n_new : d->hot_window;
    e.tiles_per_row = (most + kTileRows - 1) / kTileRows;
    e.jobs = static_cast<long long>(d->batch) * d->num_kv_heads * e.tiles_per_row;
    const tq_status st = launch_quantize(e, s);
    if (st != TQ_OK) return st;
  }
  p.evict = 0;
  p.tensors = 2;
  p.tiles_per_row = (n_new + kTileRows - 1) / kTileRows;
  p.jobs = static_cast<long long>(d->batch) * d->num_kv_heads * p.tiles_per_row * 2;
  return launch_quantize(p, s);
}

// Host build of the per-vector quantizer (same source as the kernel) for
// verifying the kernel arithmetic on machines without a GPU.  No product
// entry point calls it.
extern "C" tq_status tq_debug_quantize_rows_host(const tq_codebook* cb, uint64_t seed, int32_t layer, int32_t head,
                                                 const uint16_t* rows, int32_t n_rows, uint32_t* words,
                                                 float* norms) {
  using namespace tq;
  if (cb == nullptr || rows == nullptr || words == nullptr || norms == nullptr || n_rows < 0) return TQ_ERR_INVALID_ARG;
  if (cb->head_dim != D || cb->bits < kMinBits || cb->bits > kMaxBits) return TQ_ERR_UNSUPPORTED;
  const int n_thr = (1 << cb->bits) - 1;
  const int a = quant_lut_scale(cb->thresholds, n_thr);
  if (a == 0) return TQ_ERR_UNSUPPORTED;
  LutEntry lut[2 * 4096 + 3];
  for (int j = 0; j < lut_size(a); ++j) lut[j] = lut_entry(cb->thresholds, n_thr, a, j);
  uint32_t smask[64];
  for (int j = 0; j < 64; ++j) smask[j] = sign_mask_pair(seed, layer, head, j);
  // the kernel's four-lane decomposition, with the shuffles done by indexing
  for (int r = 0; r < n_rows; ++r) {
    uint32_t w[64];
    std::memcpy(w, rows + static_cast<size_t>(r) * D, sizeof(w));
    float h[4], l[4];
    float2 v[4][16];
    for (int q = 0; q < 4; ++q) {
      for (int k = 0; k < 16; ++k) v[q][k] = half2_bits_to_float2(w[16 * q + k] ^ smask[16 * q + k]);
      norm_partial<16>(v[q], h[q], l[q]);
      fwht32(v[q]);
    }
    float h1[4], l1[4];
    for (int q = 0; q < 4; ++q) {
      h1[q] = h[q];
      l1[q] = l[q];
      twosum_merge(h1[q], l1[q], h[q ^ 1], l[q ^ 1]);
    }
    float hs = h1[0], ls = l1[0];
    twosum_merge(hs, ls, h1[2], l1[2]);
    bool exact;  // as the kernels: codes from the candidate, the stored norm settled afterwards
    const float n = norm_decided(hs, ls, exact);
    for (int stage = 1; stage <= 2; stage *= 2) {  // index bit 5 (q ^ 1), then bit 6 (q ^ 2)
      float2 prev[4][16];
      std::memcpy(prev, v, sizeof(prev));
      for (int q = 0; q < 4; ++q)
        for (int k = 0; k < 16; ++k) {
          const float sg = (q & stage) ? -1.0f : 1.0f;
          v[q][k] = butterfly_pair(prev[q][k], prev[q ^ stage][k], make_float2(sg, sg));
        }
    }
    const float inv = n > 0.0f ? frcp(fmul(n, kSqrtD)) : 0.0f;
    uint32_t* out = words + static_cast<size_t>(r) * cb->bits * 4;
    for (int q = 0; q < 4; ++q) {
      switch (cb->bits) {
        case 2: pack_codes32<2>(v[q], inv, lut, 1, a, out + 2 * q); break;
        case 3: pack_codes32<3>(v[q], inv, lut, 1, a, out + 3 * q); break;
        default: pack_codes32<4>(v[q], inv, lut, 1, a, out + 4 * q); break;
      }
    }
    norms[r] = exact ? norm_near_midpoint(n, w) : n;
  }
  return TQ_OK;
}
