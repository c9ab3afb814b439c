// Host-side part of the C ABI: codebook construction, bit budget helpers,
// rotation signs, descriptor set-up and validation.  Needs no GPU.
#include <cmath>
#include <cstring>

#include "tq_internal.h"
#include "tq_signs.h"

namespace {

// n-point Gauss-Legendre nodes and weights on [-1, 1] by Newton iteration on
// the Legendre polynomial P_n (three-term recurrence).
struct GaussLegendre {
  static constexpr int n = 20;
  double x[n];
  double w[n];
  GaussLegendre() {
    const double pi = 3.14159265358979323846;
    for (int i = 0; i < (n + 1) / 2; ++i) {
      double z = std::cos(pi * (i + 0.75) / (n + 0.5));
      double dp = 0.0;
      for (int it = 0; it < 100; ++it) {
        double p1 = 1.0, p0 = 0.0;
        for (int j = 1; j <= n; ++j) {
          double pm = p0;
          p0 = p1;
          p1 = ((2.0 * j - 1.0) * z * p0 - (j - 1.0) * pm) / j;
        }
        dp = n * (z * p1 - p0) / (z * z - 1.0);
        double z_old = z;
        z = z_old - p1 / dp;
        if (std::fabs(z - z_old) < 1e-16) break;
      }
      x[i] = -z;
      x[n - 1 - i] = z;
      w[i] = w[n - 1 - i] = 2.0 / ((1.0 - z * z) * dp * dp);
    }
  }
};

struct Moments {
  double m0 = 0.0, m1 = 0.0, m2 = 0.0;
};

// Integrals of f_d, x f_d and x^2 f_d over [a, b] by composite Gauss-Legendre.
Moments cell_moments(double a, double b, double log_c, double expo, const GaussLegendre& gl) {
  constexpr int panels = 8;
  Moments m;
  const double width = (b - a) / panels;
  for (int p = 0; p < panels; ++p) {
    const double lo = a + width * p;
    const double half = width / 2, mid = lo + half;
    for (int k = 0; k < GaussLegendre::n; ++k) {
      const double x = mid + half * gl.x[k];
      const double f = std::exp(log_c + expo * std::log1p(-x * x));
      const double wf = gl.w[k] * half * f;
      m.m0 += wf;
      m.m1 += wf * x;
      m.m2 += wf * x * x;
    }
  }
  return m;
}

}  // namespace

extern "C" {

const char* tq_status_string(tq_status s) {
  switch (s) {
    case TQ_OK: return "TQ_OK";
    case TQ_ERR_INVALID_ARG: return "TQ_ERR_INVALID_ARG";
    case TQ_ERR_UNSUPPORTED: return "TQ_ERR_UNSUPPORTED";
    case TQ_ERR_CAPACITY: return "TQ_ERR_CAPACITY";
    case TQ_ERR_WORKSPACE: return "TQ_ERR_WORKSPACE";
    case TQ_ERR_CUDA: return "TQ_ERR_CUDA";
    case TQ_ERR_DEVICE: return "TQ_ERR_DEVICE";
  }
  return "TQ_ERR_UNKNOWN";
}

// Lloyd-Max on f_d(x) = C_d (1 - x^2)^((d-3)/2), 2^bits levels.  The density is
// even, so only the levels of the positive half are iterated and the others
// mirror them; the middle threshold is 0.
tq_status tq_build_codebook(int32_t head_dim, int32_t bits, tq_codebook* out) {
  if (out == nullptr) return TQ_ERR_INVALID_ARG;
  if (head_dim < 3 || head_dim > 65536 || bits < 1 || bits > 4) return TQ_ERR_UNSUPPORTED;
  static const GaussLegendre gl;  // constant tables, built once, read-only afterwards
  const double d = head_dim;
  const double log_c = std::lgamma(d / 2) - 0.5 * std::log(3.14159265358979323846) - std::lgamma((d - 1) / 2);
  const double expo = (d - 3) / 2;
  const int levels = 1 << bits, half = levels / 2;

  double c[8];  // positive levels, ascending
  for (int k = 0; k < half; ++k) c[k] = (k + 0.5) / half * 2.5 / std::sqrt(d);
  double edge[9];
  int iters = 0;
  for (iters = 1; iters <= 100000; ++iters) {
    edge[0] = 0.0;
    for (int k = 1; k < half; ++k) edge[k] = 0.5 * (c[k - 1] + c[k]);
    edge[half] = 1.0;
    double step = 0.0;
    for (int k = 0; k < half; ++k) {
      const Moments m = cell_moments(edge[k], edge[k + 1], log_c, expo, gl);
      const double cn = m.m1 / m.m0;
      step = std::fmax(step, std::fabs(cn - c[k]));
      c[k] = cn;
    }
    if (step < 1e-15) break;
  }
  if (iters > 100000) iters = 100000;
  edge[0] = 0.0;
  for (int k = 1; k < half; ++k) edge[k] = 0.5 * (c[k - 1] + c[k]);
  edge[half] = 1.0;
  double mse = 0.0;
  for (int k = 0; k < half; ++k) {
    const Moments m = cell_moments(edge[k], edge[k + 1], log_c, expo, gl);
    mse += 2.0 * (m.m2 - 2.0 * c[k] * m.m1 + c[k] * c[k] * m.m0);
  }

  std::memset(out, 0, sizeof(*out));
  out->head_dim = head_dim;
  out->bits = bits;
  for (int k = 0; k < half; ++k) {
    out->centroids_f64[half + k] = c[k];
    out->centroids_f64[half - 1 - k] = -c[k];
  }
  for (int k = 0; k + 1 < levels; ++k)
    out->thresholds_f64[k] = 0.5 * (out->centroids_f64[k] + out->centroids_f64[k + 1]);
  out->thresholds_f64[half - 1] = 0.0;
  for (int k = 0; k < levels; ++k) out->centroids[k] = static_cast<float>(out->centroids_f64[k]);
  for (int k = 0; k + 1 < levels; ++k) out->thresholds[k] = static_cast<float>(out->thresholds_f64[k]);
  out->mse_per_coord = mse;
  out->iterations = iters;
  return TQ_OK;
}

tq_status tq_split_bits(double bits, int32_t* k_bits, int32_t* v_bits) {
  if (k_bits == nullptr || v_bits == nullptr || !std::isfinite(bits) || bits <= 0.0 || bits > 16.0)
    return TQ_ERR_INVALID_ARG;
  *k_bits = static_cast<int32_t>(std::floor(bits));
  *v_bits = static_cast<int32_t>(std::ceil(bits));
  return TQ_OK;
}

int32_t tq_turboquant_enabled(double bits, int32_t has_bits, int32_t scheme_is_turboquant) {
  if (!has_bits) return 0;
  if (scheme_is_turboquant) return 1;
  return std::fabs(bits - std::nearbyint(bits)) > 1e-6 ? 1 : 0;
}

tq_status tq_rotation_signs(uint64_t seed, int32_t layer, int32_t head, int32_t head_dim, int8_t* out) {
  if (out == nullptr) return TQ_ERR_INVALID_ARG;
  if (layer < 0 || head < 0 || head >= (1 << 16) || head_dim < 1 || head_dim > (1 << 16)) return TQ_ERR_INVALID_ARG;
  for (int i = 0; i < head_dim; ++i) out[i] = tq::sign_negative(seed, layer, head, i) ? -1 : 1;
  return TQ_OK;
}

tq_status tq_cache_desc_init(tq_cache_desc* desc, int32_t batch, int32_t num_kv_heads, int32_t num_q_heads,
                             int32_t head_dim, int32_t capacity, int32_t k_mode, int32_t k_bits, int32_t v_bits,
                             int32_t hot_window, uint64_t seed, int32_t layer) {
  if (desc == nullptr) return TQ_ERR_INVALID_ARG;
  std::memset(desc, 0, sizeof(*desc));
  desc->batch = batch;
  desc->num_kv_heads = num_kv_heads;
  desc->num_q_heads = num_q_heads;
  desc->head_dim = head_dim;
  desc->capacity = capacity;
  desc->k_mode = k_mode;
  desc->k_bits = k_mode == TQ_K_FP16 ? 16 : k_bits;
  desc->v_bits = v_bits;
  desc->hot_window = hot_window;
  desc->layer = layer;
  desc->seed = seed;
  if (k_mode == TQ_KV_INT8) {  // no codebooks
    if (head_dim != tq::kHeadDim || k_bits != 8 || v_bits != 8) return TQ_ERR_UNSUPPORTED;
    return tq::validate_shape(desc);
  }
  if (head_dim != tq::kHeadDim || v_bits < tq::kMinBits || v_bits > tq::kMaxBits) return TQ_ERR_UNSUPPORTED;
  if (k_mode == TQ_K_PACKED) {
    if (k_bits < tq::kMinBits || k_bits > tq::kMaxBits) return TQ_ERR_UNSUPPORTED;
    tq_status s = tq_build_codebook(head_dim, k_bits, &desc->k_cb);
    if (s != TQ_OK) return s;
  }
  tq_status s = tq_build_codebook(head_dim, v_bits, &desc->v_cb);
  if (s != TQ_OK) return s;
  return tq::validate_shape(desc);  // the buffer pointers are still NULL here
}

tq_status tq_cache_desc_set_paged(tq_cache_desc* d, int32_t block_size, int32_t max_blocks_per_seq,
                                  int32_t num_blocks, const int32_t* d_block_table) {
  if (d == nullptr || d_block_table == nullptr || (reinterpret_cast<uintptr_t>(d_block_table) & 3u) != 0)
    return TQ_ERR_INVALID_ARG;
  if (block_size < 16 || block_size > 4096 || (block_size & (block_size - 1)) != 0) return TQ_ERR_INVALID_ARG;
  if (max_blocks_per_seq < 1 || num_blocks < 1) return TQ_ERR_INVALID_ARG;
  if (static_cast<long long>(max_blocks_per_seq) * block_size != d->capacity) return TQ_ERR_INVALID_ARG;
  d->block_size = block_size;
  d->max_blocks_per_seq = max_blocks_per_seq;
  d->num_blocks = num_blocks;
  d->block_table = d_block_table;
  return tq::validate_shape(d);
}

tq_status tq_cache_buffer_bytes(const tq_cache_desc* d, size_t* k_cache_bytes, size_t* k_norms_bytes,
                                size_t* v_cache_bytes, size_t* v_norms_bytes, size_t* v_hot_bytes) {
  if (d == nullptr || d->batch < 1 || d->num_kv_heads < 1 || d->capacity < 1 || d->head_dim < 1)
    return TQ_ERR_INVALID_ARG;
  const size_t rows = d->block_size > 0
                          ? static_cast<size_t>(d->num_blocks) * d->num_kv_heads * d->block_size
                          : static_cast<size_t>(d->batch) * d->num_kv_heads * d->capacity;
  const bool kfp16 = d->k_mode == TQ_K_FP16;
  if (k_cache_bytes)
    *k_cache_bytes = kfp16 ? rows * d->head_dim * 2 : rows * tq::words_per_token(d->head_dim, d->k_bits) * 4;
  if (k_norms_bytes) *k_norms_bytes = kfp16 ? 0 : rows * 4;
  if (v_cache_bytes) *v_cache_bytes = rows * tq::words_per_token(d->head_dim, d->v_bits) * 4;
  if (v_norms_bytes) *v_norms_bytes = rows * 4;
  if (v_hot_bytes)
    *v_hot_bytes = static_cast<size_t>(d->batch) * d->num_kv_heads * (d->hot_window > 0 ? d->hot_window : 0) *
                   d->head_dim * 2;
  return TQ_OK;
}

}  // extern "C"

namespace tq {

static bool codebook_matches(const tq_codebook& cb, int d, int bits) {
  if (cb.head_dim != d || cb.bits != bits) return false;
  const int levels = 1 << bits;
  for (int k = 0; k + 1 < levels; ++k)
    if (!(cb.centroids[k] < cb.centroids[k + 1]) || !(cb.thresholds[k] > cb.centroids[k]) ||
        !(cb.thresholds[k] < cb.centroids[k + 1]))
      return false;
  return true;
}

tq_status validate_shape(const tq_cache_desc* d) {
  if (d == nullptr) return TQ_ERR_INVALID_ARG;
  if (d->head_dim < 1 || (d->head_dim & (d->head_dim - 1)) != 0) return TQ_ERR_UNSUPPORTED;  // WHT needs 2^k
  if (d->head_dim != kHeadDim) return TQ_ERR_UNSUPPORTED;
  if (d->batch < 1 || d->num_kv_heads < 1 || d->num_kv_heads >= (1 << 16) || d->num_q_heads < 1 ||
      d->capacity < 1 || d->layer < 0)
    return TQ_ERR_INVALID_ARG;
  if (d->num_q_heads % d->num_kv_heads != 0) return TQ_ERR_INVALID_ARG;
  const int g = d->num_q_heads / d->num_kv_heads;
  if (g != 1 && g != 2 && g != 4) return TQ_ERR_UNSUPPORTED;
  if (d->k_mode != TQ_K_PACKED && d->k_mode != TQ_K_FP16 && d->k_mode != TQ_KV_INT8) return TQ_ERR_INVALID_ARG;
  if (d->k_mode == TQ_KV_INT8) {
    if (d->k_bits != 8 || d->v_bits != 8) return TQ_ERR_UNSUPPORTED;
  } else {
    if (d->k_mode == TQ_K_PACKED) {
      if (d->k_bits < kMinBits || d->k_bits > kMaxBits) return TQ_ERR_UNSUPPORTED;
      if (!codebook_matches(d->k_cb, d->head_dim, d->k_bits)) return TQ_ERR_INVALID_ARG;
    }
    if (d->v_bits < kMinBits || d->v_bits > kMaxBits) return TQ_ERR_UNSUPPORTED;
    if (!codebook_matches(d->v_cb, d->head_dim, d->v_bits)) return TQ_ERR_INVALID_ARG;
    if (quant_lut_scale(d->v_cb.thresholds, (1 << d->v_bits) - 1) == 0) return TQ_ERR_UNSUPPORTED;
    if (d->k_mode == TQ_K_PACKED && quant_lut_scale(d->k_cb.thresholds, (1 << d->k_bits) - 1) == 0)
      return TQ_ERR_UNSUPPORTED;
  }
  if (d->hot_window < 0 || d->hot_window > d->capacity) return TQ_ERR_INVALID_ARG;
  if (d->block_size != 0) {  // paged layout
    if (d->block_size < 16 || d->block_size > 4096 || (d->block_size & (d->block_size - 1)) != 0)
      return TQ_ERR_INVALID_ARG;
    if (d->max_blocks_per_seq < 1 || d->num_blocks < 1 || d->block_table == nullptr) return TQ_ERR_INVALID_ARG;
    if (static_cast<long long>(d->max_blocks_per_seq) * d->block_size != d->capacity) return TQ_ERR_INVALID_ARG;
    if (static_cast<long long>(d->num_blocks) * d->num_kv_heads * d->block_size >= (1ll << 40))
      return TQ_ERR_UNSUPPORTED;
  }
  return TQ_OK;
}

tq_status validate_desc(const tq_cache_desc* d) {
  const tq_status s = validate_shape(d);
  if (s != TQ_OK) return s;
  if (d->k_cache == nullptr || d->v_cache == nullptr || d->v_norms == nullptr) return TQ_ERR_INVALID_ARG;
  if (!aligned16(d->k_cache) || !aligned16(d->v_cache) || !aligned16(d->v_norms)) return TQ_ERR_INVALID_ARG;
  if (d->k_mode != TQ_K_FP16 && (d->k_norms == nullptr || !aligned16(d->k_norms))) return TQ_ERR_INVALID_ARG;
  if (d->hot_window > 0 && (d->v_hot == nullptr || !aligned16(d->v_hot))) return TQ_ERR_INVALID_ARG;
  if (!(d->sparse_v_threshold >= 0.0f && d->sparse_v_threshold <= 1.0f)) return TQ_ERR_INVALID_ARG;  // NaN too
  return TQ_OK;
}

size_t decode_workspace_slots(const tq_cache_desc* d, int nq) {
  return static_cast<size_t>(kMaxDecodeCtas) + 2 * static_cast<size_t>(d->batch) * nq * d->num_kv_heads;
}

size_t decode_workspace_bytes(const tq_cache_desc* d, int nq) {
  const size_t g = static_cast<size_t>(d->num_q_heads / d->num_kv_heads);
  return decode_workspace_slots(d, nq) * g * (kHeadDim + 2) * sizeof(float);
}

int quant_lut_scale(const float* t, int n) {
  for (int a = 8; a <= 4096; a *= 2) {
    bool ok = true;
    for (int k = 0; k + 1 < n && ok; ++k) {
      // bucket of y is RN(y * a) (exact product, single rounding); neighbours must differ
      const float b0 = std::nearbyint(t[k] * static_cast<float>(a));
      const float b1 = std::nearbyint(t[k + 1] * static_cast<float>(a));
      ok = b1 > b0;
    }
    if (ok) return a;
  }
  return 0;
}

}  // namespace tq
