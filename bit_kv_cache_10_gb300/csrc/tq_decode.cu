// Decode attention over the packed cache: the host entry points, the merge
// kernel and the dense contiguous instantiations of the split-K kernel (the
// kernel itself is in tq_decode_mma.cuh; its sparse-V, paged and multi-token
// instantiations are in tq_decode_sparse.cu, tq_decode_paged.cu,
// tq_decode_paged_sparse.cu, tq_decode_multi.cu and tq_decode_multi_paged.cu,
// the cluster variant's in tq_decode_cluster.cu).
#include <atomic>
#include <cstring>
#include <vector>

#include "tq_decode_dispatch.cuh"
#include "tq_debug.h"

namespace tq {
namespace {

// Merge kernel: one warp per (sequence b, query head), the G warps of a CTA
// sharing the KV head h.  Lane l holds coordinates 4 l .. 4 l + 3: it finds the
// CTAs that covered the (b, h) rows, log-sum-exp combines their partials, rotates
// the cold sum back (sign flips and a Hadamard transform over index bits 0..1 in
// registers and 2..6 across lanes, 1/sqrt d; not in the int8 mode), adds the hot
// sum and divides by the softmax mass.
__global__ void __launch_bounds__(4 * 32) decode_merge_kernel(const DecodeParams p) {
  // a following programmatic dependent grid (the next append) may start its
  // parameter-only prologue now; it waits for this grid before touching memory
  asm volatile("griddepcontrol.launch_dependents;\n");
  const int g = p.hq / p.hkv;
  const int jj = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x, b = blockIdx.y;
  if (jj >= g) return;
  // rotation signs of the lane's coordinates 4 lane .. 4 lane + 3 (parameters only)
  unsigned neg4 = 0u;
  if (p.rotated)
#pragma unroll
    for (int i = 0; i < 4; ++i) neg4 |= sign_negative(p.seed, p.layer, h, 4 * lane + i) ? 1u << i : 0u;
  // the lengths may be written by a grid before the split kernel and the partials
  // by the split kernel: wait for the preceding grids before reading either
  // (programmatic dependent launch lets this grid start while they finish)
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  float4* out = reinterpret_cast<float4*>(p.out + (static_cast<int64_t>(b) * p.hq + h * g + jj) * D);
  // tiles of the sequences before b, and of all sequences
  long long before = 0, total = 0;
  for (int bb = lane; bb < p.batch; bb += 32) {
    const SeqTiles sq = seq_tiles<true>(p, bb);  // the general form also holds for one query token
    const long long c = static_cast<long long>(p.hkv) * (sq.tc + sq.th);
    total += c;
    if (bb < b) before += c;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    before += __shfl_xor_sync(0xffffffffu, before, o);
    total += __shfl_xor_sync(0xffffffffu, total, o);
  }
  const SeqTiles st = seq_tiles<true>(p, b);
  if (st.len == 0) {
    out[lane] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    return;
  }
  const int per_h = st.tc + st.th;
  const long long hbase = before + static_cast<long long>(h) * per_h;
  // rows of this (b, h): cold [hbase, hbase + tc), hot [hbase + tc, hbase + per_h),
  // at the costs of the split kernel's weighted split (tq_split_plan.h); partial
  // i < n0 comes from cold CTA c0 + i, partial n0 + i from hot CTA c1 + i
  const long long r = static_cast<long long>(b) * p.hkv + h;
  const long long cost_all = split_total_cost(total, static_cast<long long>(p.batch) * p.hkv, p.price);
  const long long a0 = split_cold_cost(hbase, r, p.price), e0 = a0 + st.tc - 1;        // cold costs [a0, e0]
  const long long a1 = split_hot_cost(hbase, st.tc, r, p.price), e1 = a1 + st.th - 1;  // hot costs [a1, e1]
  int c0 = 0, n0 = 0, c1 = 0, n1 = 0;
  if (st.tc > 0) {
    c0 = split_cta(a0, cost_all, p.grid);
    n0 = split_cta(e0, cost_all, p.grid) - c0 + 1;
  }
  if (st.th > 0) {
    c1 = split_cta(a1, cost_all, p.grid);
    n1 = split_cta(e1, cost_all, p.grid) - c1 + 1;
  }
  const int row0 = (b * p.hkv + h) * 2;
  auto slot_of = [&](int i) {
    return i < n0 ? static_cast<long long>(c0 + i) + row0 : static_cast<long long>(c1 + i - n0) + row0 + 1;
  };
  auto live = [&](int i) {  // a CTA that took no tile of the segment wrote no partial for it
    return i < n0 ? split_cta_hits(c0 + i, a0, e0, cost_all, p.grid) : split_cta_hits(c1 + i - n0, a1, e1, cost_all, p.grid);
  };
  const int n = n0 + n1;
  const unsigned live32 = __ballot_sync(0xffffffffu, lane < n && live(lane));
  auto is_live = [&](int i) { return i < 32 ? ((live32 >> i) & 1u) != 0 : live(i); };
  float mm = -INFINITY, l = 0.0f;
  float y[4] = {0.0f, 0.0f, 0.0f, 0.0f}, hv[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  auto add_partial = [&](int i, float sc, const float4 a) {
    const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if (i >= n0) hv[k] = ffma(av[k], sc, hv[k]);
      else y[k] = ffma(av[k], sc, y[k]);
    }
  };
  if (n <= 16) {
    // one partial per lane: its (max, mass) read once, its scale shared by
    // shuffles; every accumulator load is issued before the scales are known, so
    // the whole merge waits for one round of loads (a partial that was not
    // written has scale 0 and its loaded values are not used)
    float2 ml = make_float2(-INFINITY, 0.0f);
    if (lane < n && ((live32 >> lane) & 1u))
      ml = reinterpret_cast<const float2*>(p.ws_ml)[slot_of(lane) * g + jj];
    float4 a[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
      if (i < n) a[i] = reinterpret_cast<const float4*>(p.ws_acc + (slot_of(i) * g + jj) * D)[lane];
    mm = ml.x;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mm = fmaxf(mm, __shfl_xor_sync(0xffffffffu, mm, o));
    const float sc_l = ml.x == -INFINITY ? 0.0f : exp2f(ml.x - mm);
    l = fmul(ml.y, sc_l);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l = fadd(l, __shfl_xor_sync(0xffffffffu, l, o));
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (i >= n) break;
      const float sc = __shfl_sync(0xffffffffu, sc_l, i);
      if (sc != 0.0f) add_partial(i, sc, a[i]);
    }
  } else if (n <= 32) {
    // as above with the loads in two rounds of 16
    float2 ml = make_float2(-INFINITY, 0.0f);
    if (lane < n && ((live32 >> lane) & 1u))
      ml = reinterpret_cast<const float2*>(p.ws_ml)[slot_of(lane) * g + jj];
    float4 a[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) a[i] = reinterpret_cast<const float4*>(p.ws_acc + (slot_of(i) * g + jj) * D)[lane];
    mm = ml.x;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mm = fmaxf(mm, __shfl_xor_sync(0xffffffffu, mm, o));
    const float sc_l = ml.x == -INFINITY ? 0.0f : exp2f(ml.x - mm);
    l = fmul(ml.y, sc_l);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l = fadd(l, __shfl_xor_sync(0xffffffffu, l, o));
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float sc = __shfl_sync(0xffffffffu, sc_l, i);
      const float4 nxt = 16 + i < n ? reinterpret_cast<const float4*>(p.ws_acc + (slot_of(16 + i) * g + jj) * D)[lane]
                                    : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      if (sc != 0.0f) add_partial(i, sc, a[i]);
      a[i] = nxt;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (16 + i >= n) break;
      const float sc = __shfl_sync(0xffffffffu, sc_l, 16 + i);
      if (sc != 0.0f) add_partial(16 + i, sc, a[i]);
    }
  } else {
    // (max, mass) of the partials, several per lane, then across the warp
    for (int i = lane; i < n; i += 32)
      if (is_live(i)) mm = fmaxf(mm, p.ws_ml[(slot_of(i) * g + jj) * 2]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mm = fmaxf(mm, __shfl_xor_sync(0xffffffffu, mm, o));
    for (int i = lane; i < n; i += 32) {
      if (!is_live(i)) continue;
      const float ms = p.ws_ml[(slot_of(i) * g + jj) * 2];
      if (ms != -INFINITY) l = ffma(p.ws_ml[(slot_of(i) * g + jj) * 2 + 1], exp2f(ms - mm), l);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l = fadd(l, __shfl_xor_sync(0xffffffffu, l, o));
    for (int i = 0; i < n; ++i) {  // accumulators, partial by partial
      if (!is_live(i)) continue;
      const long long slot = slot_of(i);
      const float ms = p.ws_ml[(slot * g + jj) * 2];
      if (ms == -INFINITY) continue;
      add_partial(i, exp2f(ms - mm), reinterpret_cast<const float4*>(p.ws_acc + (slot * g + jj) * D)[lane]);
    }
  }
  merge_finish(y, hv, l, neg4, p.rotated, p.out + (static_cast<int64_t>(b) * p.hq + h * g + jj) * D, lane);
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

}  // namespace
}  // namespace tq

namespace tq {
namespace {

// Decode path selection for tests: 0 automatic, 1 always the persistent split
// kernel and the merge kernel, 2 the cluster variant wherever the mode allows it.
std::atomic<int> g_decode_path{0};
// Longest context the automatic selection sends to the cluster variant: about
// four 16-token tiles per warp of a row's kClusterCtas CTAs.
constexpr int kClusterMaxLen = kClusterCtas * 12 * 4 * kTile;

// Segment start prices of the weighted split (tq_split_plan.h), in tiles,
// chosen by timing the decode calls over a sweep of prices on GB300 (the
// optimum is broad): 56 per segment with a hot window (long-context 3.5-bit
// decode, 159 -> 152 us), 32 per row without one (the hot parts are empty; fp16
// K with 4-bit V at context 16384: 69.7 -> 68.2 us; the int8 mode within 1 %).
SplitPrice split_price(const tq_cache_desc* d, int nq) {
  (void)nq;  // the multi-token work list has rows of the same tiles
  return d->hot_window > 0 ? SplitPrice{56, 56} : SplitPrice{32, 0};
}

// Split-K attention of nq query tokens per sequence (the newest nq positions,
// causal; nq = 1 is decode) over the cache: the work list holds B nq
// sequences, sequence b nq + i being query token i of cache sequence b.
tq_status run_attention(const tq_cache_desc* d, const void* q, int nq, const int32_t* d_seq_lens, int32_t max_seq_len,
                        float* out, void* workspace, size_t workspace_bytes, cudaStream_t s) {
  if (q == nullptr || d_seq_lens == nullptr || out == nullptr || max_seq_len < 0 || nq < 1) return TQ_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(out)) return TQ_ERR_INVALID_ARG;
  if (static_cast<long long>(d->batch) * nq > kMaxDecodeBatch) return TQ_ERR_UNSUPPORTED;
  if (nq > 1 && d->sparse_v_threshold > 0.0f) return TQ_ERR_UNSUPPORTED;  // several query tokens: dense V
  if (static_cast<long long>(d->num_kv_heads) * (d->capacity / 32 + d->hot_window / 32 + 2) >= (1ll << 31))
    return TQ_ERR_UNSUPPORTED;  // tiles of one sequence must fit in 32 bits
  const size_t out_bytes = static_cast<size_t>(d->batch) * nq * d->num_q_heads * D * sizeof(float);
  if (max_seq_len == 0) return cudaMemsetAsync(out, 0, out_bytes, s) == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
  const size_t need = decode_workspace_bytes(d, nq);
  if (workspace == nullptr || !aligned16(workspace) || workspace_bytes < need) return TQ_ERR_WORKSPACE;
  const int sms = sm_count();
  if (sms <= 0) return TQ_ERR_CUDA;

  DecodeParams p;
  std::memset(&p, 0, sizeof(p));
  p.q = static_cast<const uint16_t*>(q);
  p.seq_lens = d_seq_lens;
  p.max_seq_len = max_seq_len;
  p.batch = d->batch * nq;
  p.nq = nq;
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
  p.map = make_row_map(d);
  p.status = d->d_status;
  p.seed = d->seed;
  p.layer = d->layer;
  if (d->k_mode == TQ_K_PACKED) std::memcpy(p.k_cent, d->k_cb.centroids, sizeof(p.k_cent));
  if (d->k_mode != TQ_KV_INT8) std::memcpy(p.v_cent, d->v_cb.centroids, sizeof(p.v_cent));
  const int g = d->num_q_heads / d->num_kv_heads;
  const size_t slots = decode_workspace_slots(d, nq);
  p.ws_acc = static_cast<float*>(workspace);
  p.ws_ml = p.ws_acc + slots * g * D;
  p.grid = sms < kMaxDecodeCtas ? sms : kMaxDecodeCtas;
  p.price = split_price(d, nq);
  p.sparse_tau = d->sparse_v_threshold;
  p.rotated = d->k_mode != TQ_KV_INT8;
  p.out = out;

  const int kb = d->k_mode == TQ_K_FP16 ? 16 : d->k_bits;
  tq_status st;
  const bool sparse = p.sparse_tau > 0.0f, paged = d->block_size > 0;
  // small work (rows of at most kClusterMaxLen positions, every row's cluster
  // resident at once): one thread-block cluster per (b, h) row, no merge launch
  const int path = g_decode_path.load(std::memory_order_relaxed);
  if (nq == 1 && !paged && !sparse && path != 1 && (path == 2 || max_seq_len <= kClusterMaxLen)) {
    st = dispatch_cluster(p, g, kb, d->v_bits, s);
    if (st != TQ_ERR_UNSUPPORTED) return st;
  }
  if (nq > 1) {
    st = paged ? dispatch_split_multi_paged(p, g, kb, d->v_bits, s) : dispatch_split_multi(p, g, kb, d->v_bits, s);
  } else if (paged) {
    st = sparse ? dispatch_split_paged_sparse(p, g, kb, d->v_bits, s) : dispatch_split_paged(p, g, kb, d->v_bits, s);
  } else {
    st = sparse ? dispatch_split_sparse(p, g, kb, d->v_bits, s) : dispatch_split_variant<false, false>(p, g, kb, d->v_bits, s);
  }
  if (st != TQ_OK) return st;
  // with programmatic dependent launch (kProgrammaticLaunch) the merge grid would be
  // scheduled as the split kernel's CTAs retire and wait (griddepcontrol.wait) for
  // its completion; without it, it starts after the split kernel
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(d->num_kv_heads, p.batch);
  cfg.blockDim = dim3(4 * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = kProgrammaticLaunch;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, decode_merge_kernel, p) != cudaSuccess) return TQ_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
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
  return run_attention(d, q, 1, d_seq_lens, max_seq_len, out, workspace, workspace_bytes,
                       reinterpret_cast<cudaStream_t>(stream));
}

extern "C" size_t tq_multi_query_workspace_bytes(const tq_cache_desc* d, int32_t n_query, int32_t max_seq_len) {
  using namespace tq;
  if (validate_shape(d) != TQ_OK || max_seq_len < 0 || n_query < 1) return 0;
  if (max_seq_len == 0) return 0;
  return decode_workspace_bytes(d, n_query);
}

extern "C" tq_status tq_multi_query_attention(const tq_cache_desc* d, const void* q, int32_t n_query,
                                              const int32_t* d_seq_lens, int32_t max_seq_len, float* out,
                                              void* workspace, size_t workspace_bytes, tq_stream_t stream) {
  using namespace tq;
  const tq_status vs = validate_desc(d);
  if (vs != TQ_OK) return vs;
  return run_attention(d, q, n_query, d_seq_lens, max_seq_len, out, workspace, workspace_bytes,
                       reinterpret_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------------------
// Decode without a caller workspace: the split-K partials live in a fixed
// device array of this file, for callers that cannot allocate device memory.
// ---------------------------------------------------------------------------
namespace {

static __device__ __align__(256) unsigned char g_no_alloc_scratch[TQ_NO_ALLOC_WORKSPACE_BYTES];

// Device address of the scratch array in the current context.  In host code the
// array's name only stands in for the symbol, so the address is looked up with
// the caller's device current, on every call: the module can be loaded at another
// address in another context (or after a device reset), so no address is kept
// between calls.  The lookup is host-side and allocates nothing.
tq_status no_alloc_scratch(void** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_no_alloc_scratch) != cudaSuccess || p == nullptr) return TQ_ERR_CUDA;
  *out = p;
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

extern "C" void tq_debug_set_decode_path(int32_t path) {
  tq::g_decode_path.store(path == 1 || path == 2 ? path : 0, std::memory_order_relaxed);
}

extern "C" tq_status tq_debug_split_plan(const int32_t* tiles_cold, const int32_t* tiles_hot, int32_t nv, int32_t hkv,
                                         int32_t grid, int32_t price_cold, int32_t price_hot, int64_t* starts,
                                         uint8_t* seg_ctas) {
  using namespace tq;
  if (tiles_cold == nullptr || tiles_hot == nullptr || starts == nullptr || nv < 1 || hkv < 1 || grid < 1 ||
      price_cold < 0 || price_hot < 0)
    return TQ_ERR_INVALID_ARG;
  const SplitPrice price{price_cold, price_hot};
  std::vector<long long> prefix(static_cast<size_t>(nv) + 1, 0);
  for (int v = 0; v < nv; ++v) {
    if (tiles_cold[v] < 0 || tiles_hot[v] < 0) return TQ_ERR_INVALID_ARG;
    prefix[v + 1] = prefix[v] + static_cast<long long>(hkv) * (tiles_cold[v] + tiles_hot[v]);
    if (prefix[v + 1] >= (1ll << 40)) return TQ_ERR_INVALID_ARG;
  }
  const long long total = prefix[nv], rows = static_cast<long long>(nv) * hkv;
  const long long cost_all = split_total_cost(total, rows, price);
  // the split kernel's ranges (its start_of)
  for (int c = 0; c <= grid; ++c) {
    if (c == grid) {
      starts[c] = total;
      continue;
    }
    const long long tau = split_cost_at(cost_all, grid, c);
    const int v = split_find_seq(prefix.data(), nv, hkv, price, tau);
    starts[c] = v < 0 ? 0 : split_tile_in_seq(prefix.data(), v, hkv, tiles_cold[v], price, tau);
  }
  if (seg_ctas == nullptr) return TQ_OK;
  // the merge kernel's choice of partials per row
  std::memset(seg_ctas, 0, static_cast<size_t>(2 * rows) * grid);
  for (int v = 0; v < nv; ++v) {
    const int tc = tiles_cold[v], th = tiles_hot[v];
    for (int h = 0; h < hkv; ++h) {
      const long long r = static_cast<long long>(v) * hkv + h;
      const long long hbase = prefix[v] + static_cast<long long>(h) * (tc + th);
      const long long a[2] = {split_cold_cost(hbase, r, price), split_hot_cost(hbase, tc, r, price)};
      const int n_t[2] = {tc, th};
      for (int part = 0; part < 2; ++part) {
        if (n_t[part] == 0) continue;
        const long long e = a[part] + n_t[part] - 1;
        const int c_first = split_cta(a[part], cost_all, grid), c_last = split_cta(e, cost_all, grid);
        for (int c = c_first; c <= c_last; ++c)
          if (split_cta_hits(c, a[part], e, cost_all, grid)) seg_ctas[(2 * r + part) * grid + c] = 1;
      }
    }
  }
  return TQ_OK;
}
