// Quantize-and-append kernel (one launch for K and V of every head) and the
// hot-window evict pass.
//
// Work unit: a "job" is 32 consecutive tokens of one (tensor, batch, KV head).
// Each warp streams its jobs through a two-stage cp.async pipeline into a
// padded shared-memory tile (272-byte rows, so that the 16-byte row reads of
// the 32 lanes hit distinct banks), then every lane quantizes one token
// vector entirely in registers: exact norm, sign flip, 128-point FWHT,
// bucketed threshold lookup, LSB-first packing.
#include <cstring>

#include "tq_device.cuh"
#include "tq_internal.h"
#include "tq_debug.h"

namespace tq {
namespace {

constexpr int kWarps = 8;                   // warps per CTA
constexpr int kRowBytes = 256;              // one fp16 vector
constexpr int kRowPitch = kRowBytes + 16;   // padded smem pitch
constexpr int kTileRows = 32;
constexpr int kTileBytes = kTileRows * kRowPitch;
constexpr int kLutCopies = 16;              // one LUT copy per lane of a half-warp

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
  uint32_t* status;
  uint64_t seed;
  int layer;
  float k_thr[15];
  float v_thr[15];
  int k_lut_a, v_lut_a;
  int evict;           // 0: append pass, 1: evict ring tokens that turn cold
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

__device__ __forceinline__ Job decode_job(const QuantParams& p, long long j) {
  Job jb;
  jb.tensor = static_cast<int>(j % p.tensors);
  long long r = j / p.tensors;
  jb.tile = static_cast<int>(r % p.tiles_per_row);
  r /= p.tiles_per_row;
  jb.h = static_cast<int>(r % p.heads);
  jb.b = static_cast<int>(r / p.heads);
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
  if (p.evict) jb.tensor = 1;  // 0 = K, 1 = V
  return jb;
}

// Global address of the fp16 source row for tile row `row` of a job, or null.
__device__ __forceinline__ const uint16_t* src_row(const QuantParams& p, const Job& jb, int row, int* pos_out) {
  const int t = jb.tile * kTileRows + row;
  if (!p.evict) {
    if (t >= jb.count) return nullptr;
    *pos_out = jb.start + t;
    const uint16_t* base = jb.tensor == 0 ? p.k_src : p.v_src;
    return base + jb.b * p.stride_b + jb.h * p.stride_h + t * p.stride_t;
  }
  const int pos = jb.start + t;
  if (pos >= jb.end) return nullptr;
  *pos_out = pos;
  return p.v_ring + ((static_cast<int64_t>(jb.b) * p.heads + jb.h) * p.hot + pos % p.hot) * D;
}

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
__device__ __forceinline__ void cp_async_wait1() { asm volatile("cp.async.wait_group 1;\n" ::); }

__device__ __forceinline__ void issue_tile(const QuantParams& p, long long j, uint8_t* tile, int lane) {
  const Job jb = decode_job(p, j);
  if (!jb.valid) return;
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const int row = 2 * k + (lane >> 4), col = lane & 15;
    int pos = 0;
    const uint16_t* src = src_row(p, jb, row, &pos);
    if (src != nullptr) cp_async16(tile + row * kRowPitch + col * 16, src + col * 8);
  }
}

template <int BITS>
__device__ __forceinline__ void quantize_store(const uint32_t* w, const uint32_t* smask, const LutEntry* lut,
                                               int lut_a, uint32_t* dst_words, float* dst_norm, int lane) {
  uint32_t out[BITS * 4];
  const float n = quantize_vector<BITS>(w, smask, lut + (lane & (kLutCopies - 1)), kLutCopies, lut_a, out);
  uint4* d4 = reinterpret_cast<uint4*>(dst_words);
#pragma unroll
  for (int k = 0; k < BITS; ++k) d4[k] = make_uint4(out[4 * k], out[4 * k + 1], out[4 * k + 2], out[4 * k + 3]);
  *dst_norm = n;
}

__device__ __forceinline__ void quantize_any(int bits, const uint32_t* w, const uint32_t* smask, const LutEntry* lut,
                                             int lut_a, uint32_t* dst_words, float* dst_norm, int lane) {
  switch (bits) {
    case 2: quantize_store<2>(w, smask, lut, lut_a, dst_words, dst_norm, lane); break;
    case 3: quantize_store<3>(w, smask, lut, lut_a, dst_words, dst_norm, lane); break;
    default: quantize_store<4>(w, smask, lut, lut_a, dst_words, dst_norm, lane); break;
  }
}

__global__ void __launch_bounds__(kWarps * 32, 1) quantize_append_kernel(const QuantParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int lut_k_n = p.k_lut_a ? lut_size(p.k_lut_a) : 0;
  const int lut_v_n = lut_size(p.v_lut_a);
  LutEntry* lut_k = reinterpret_cast<LutEntry*>(smem);
  LutEntry* lut_v = lut_k + lut_k_n * kLutCopies;
  uint8_t* warp_area = reinterpret_cast<uint8_t*>(lut_v + lut_v_n * kLutCopies);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* tiles = warp_area + warp * (2 * kTileBytes + 256);
  uint32_t* smask = reinterpret_cast<uint32_t*>(tiles + 2 * kTileBytes);

  // threshold lookup tables, kLutCopies interleaved copies (entry j of copy c at j*copies + c)
  for (int i = threadIdx.x; i < lut_k_n * kLutCopies; i += blockDim.x)
    lut_k[i] = lut_entry(p.k_thr, (1 << p.k_bits) - 1, p.k_lut_a, i / kLutCopies);
  for (int i = threadIdx.x; i < lut_v_n * kLutCopies; i += blockDim.x)
    lut_v[i] = lut_entry(p.v_thr, (1 << p.v_bits) - 1, p.v_lut_a, i / kLutCopies);
  __syncthreads();

  const long long stride = static_cast<long long>(gridDim.x) * kWarps;
  long long j = static_cast<long long>(blockIdx.x) * kWarps + warp;
  int buf = 0;
  if (j < p.jobs) issue_tile(p, j, tiles, lane);
  cp_async_commit();
  for (; j < p.jobs; j += stride) {
    const long long jn = j + stride;
    if (jn < p.jobs) issue_tile(p, jn, tiles + (buf ^ 1) * kTileBytes, lane);
    cp_async_commit();
    cp_async_wait1();
    __syncwarp();

    const Job jb = decode_job(p, j);
    if (!jb.valid) {
      if (jb.tile == 0 && jb.tensor == (p.evict ? 1 : 0) && jb.h == 0 && lane == 0 && p.status != nullptr)
        atomicOr(p.status, TQ_DEV_ERR_APPEND_RANGE);
    } else {
      // rotation-sign masks of this head
      smask[lane] = sign_mask_pair(p.seed, p.layer, jb.h, lane);
      smask[lane + 32] = sign_mask_pair(p.seed, p.layer, jb.h, lane + 32);
      __syncwarp();
      int pos = 0;
      const uint16_t* src = src_row(p, jb, lane, &pos);
      if (src != nullptr) {
        const uint4* row = reinterpret_cast<const uint4*>(tiles + buf * kTileBytes + lane * kRowPitch);
        uint32_t w[64];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const uint4 u = row[k];
          w[4 * k] = u.x;
          w[4 * k + 1] = u.y;
          w[4 * k + 2] = u.z;
          w[4 * k + 3] = u.w;
        }
        const int64_t rowidx = (static_cast<int64_t>(jb.b) * p.heads + jb.h) * p.cap + pos;
        if (jb.tensor == 0) {
          if (p.k_mode == TQ_K_FP16) {
            uint4* dst = reinterpret_cast<uint4*>(p.k_fp16 + rowidx * D);
#pragma unroll
            for (int k = 0; k < 16; ++k) dst[k] = row[k];
          } else {
            quantize_any(p.k_bits, w, smask, lut_k, p.k_lut_a, p.k_words + rowidx * (p.k_bits * 4),
                         p.k_norms + rowidx, lane);
          }
        } else {
          bool to_ring = false;
          if (p.hot > 0 && !p.evict) {
            const int cold_end = jb.end - min(p.hot, jb.end);
            to_ring = pos >= cold_end;
          }
          if (to_ring) {
            uint4* dst = reinterpret_cast<uint4*>(
                p.v_ring + ((static_cast<int64_t>(jb.b) * p.heads + jb.h) * p.hot + pos % p.hot) * D);
#pragma unroll
            for (int k = 0; k < 16; ++k) dst[k] = row[k];
          } else {
            quantize_any(p.v_bits, w, smask, lut_v, p.v_lut_a, p.v_words + rowidx * (p.v_bits * 4),
                         p.v_norms + rowidx, lane);
          }
        }
      }
    }
    __syncwarp();
    buf ^= 1;
  }
  asm volatile("cp.async.wait_all;\n" ::);
}

size_t quant_smem_bytes(int k_lut_a, int v_lut_a) {
  const size_t luts = (static_cast<size_t>(k_lut_a ? lut_size(k_lut_a) : 0) + lut_size(v_lut_a)) * kLutCopies *
                      sizeof(LutEntry);
  return luts + static_cast<size_t>(kWarps) * (2 * kTileBytes + 256);
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

tq_status launch_quantize(QuantParams& p, cudaStream_t stream) {
  if (p.jobs <= 0) return TQ_OK;
  const size_t smem = quant_smem_bytes(p.k_lut_a, p.v_lut_a);
  if (cudaFuncSetAttribute(quantize_append_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return TQ_ERR_CUDA;
  const int sms = sm_count();
  if (sms <= 0) return TQ_ERR_CUDA;
  const long long want = (p.jobs + kWarps - 1) / kWarps;
  const int grid = static_cast<int>(want < sms ? want : sms);
  quantize_append_kernel<<<grid, kWarps * 32, smem, stream>>>(p);
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
  p.k_bits = d->k_mode == TQ_K_PACKED ? d->k_bits : 0;
  p.v_bits = d->v_bits;
  p.k_words = static_cast<uint32_t*>(d->k_cache);
  p.k_norms = d->k_norms;
  p.k_fp16 = static_cast<uint16_t*>(d->k_cache);
  p.v_words = static_cast<uint32_t*>(d->v_cache);
  p.v_norms = d->v_norms;
  p.v_ring = static_cast<uint16_t*>(d->v_hot);
  p.status = d->d_status;
  p.seed = d->seed;
  p.layer = d->layer;
  if (d->k_mode == TQ_K_PACKED) {
    std::memcpy(p.k_thr, d->k_cb.thresholds, sizeof(p.k_thr));
    p.k_lut_a = quant_lut_scale(d->k_cb.thresholds, (1 << d->k_bits) - 1);
  }
  std::memcpy(p.v_thr, d->v_cb.thresholds, sizeof(p.v_thr));
  p.v_lut_a = quant_lut_scale(d->v_cb.thresholds, (1 << d->v_bits) - 1);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  if (d->hot_window > 0) {  // V tokens leaving the ring are quantized before their slots are reused
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
  for (int r = 0; r < n_rows; ++r) {
    uint32_t w[64];
    std::memcpy(w, rows + static_cast<size_t>(r) * D, sizeof(w));
    uint32_t* out = words + static_cast<size_t>(r) * cb->bits * 4;
    switch (cb->bits) {
      case 2: norms[r] = quantize_vector<2>(w, smask, lut, 1, a, out); break;
      case 3: norms[r] = quantize_vector<3>(w, smask, lut, 1, a, out); break;
      default: norms[r] = quantize_vector<4>(w, smask, lut, 1, a, out); break;
    }
  }
  return TQ_OK;
}
