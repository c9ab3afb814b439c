/*
 * tq.h -- C ABI of the TurboQuant packed KV-cache library (GB300, sm_103a).
 *
 * The library implements the data-parallel hot path of TurboQuant KV-cache
 * quantization as the pages below describe it, in hand-written CUDA:
 *
 *   [MLX-VLM deep-dive]  "TurboQuant KV Cache Quantization in MLX-VLM: Low-Bit
 *                         Compression for Efficient Generation"
 *   [MLX-VLM CLI guide]  "How to Use TurboQuant with the MLX-VLM CLI:
 *                         KV-Cache Compression Guide"
 *   [mlxcel doc]         "TurboQuant KV cache" (mlxcel docs/turbo-kv-cache.md)
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Ownership.   The caller allocates every device buffer (cache, queries,
 *              outputs, workspace) and keeps it alive while work that uses it
 *              is queued.  The library allocates no device memory, keeps no
 *              global state (the one exception is the fixed scratch array of
 *              tq_decode_attention_no_alloc, part of the library's device
 *              image), and may be called from several host threads.
 * Asynchrony.  Functions taking a stream enqueue kernels on it and return at
 *              once; results are ready when the stream is.  A NULL stream is
 *              the legacy default stream.  The host-only helpers are
 *              synchronous and need no GPU.  The stream functions only
 *              launch kernels (no allocation, no synchronisation, no reads of
 *              device data on the host), so a sequence of appends and decodes
 *              may be captured into a CUDA graph and replayed; the captured
 *              kernels keep the arguments of the capture (pointers, sizes,
 *              max_seq_len), while device-side inputs such as start
 *              positions and lengths are read when the graph runs.
 * Errors.      Argument errors are found on the host and returned before any
 *              launch (nothing is enqueued).  A failed launch returns
 *              TQ_ERR_CUDA.  Errors that only the device can see (a start
 *              position or a sequence length outside the cache) set bits of
 *              the optional device status word `d_status` (atomic OR) and the
 *              offending sequence is skipped; kernels never trap and never
 *              spin-wait.
 * Layouts.     All index arithmetic is row-major.  "[B, Hkv, cap, W]" means a
 *              contiguous array with W fastest.  Device pointers must be
 *              16-byte aligned (cudaMalloc and torch give 256 bytes).
 */
#ifndef TQ_H_
#define TQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t (declared here so that the header needs no CUDA headers). */
typedef struct CUstream_st *tq_stream_t;

typedef enum tq_status {
  TQ_OK = 0,
  TQ_ERR_INVALID_ARG = -1, /* null pointer, bad shape, misaligned pointer or stride */
  TQ_ERR_UNSUPPORTED = -2, /* valid request outside what the kernels implement
                              (head_dim not a power of two, bits outside 2..4, ...) */
  TQ_ERR_CAPACITY = -3,    /* a host-visible size exceeds the cache capacity */
  TQ_ERR_WORKSPACE = -4,   /* workspace pointer missing, misaligned or too small */
  TQ_ERR_CUDA = -5,        /* a CUDA runtime call or launch failed */
  TQ_ERR_DEVICE = -6       /* reserved: device-side error reported through d_status */
} tq_status;

/* Bits of the device status word (OR-ed together by the kernels). */
#define TQ_DEV_ERR_APPEND_RANGE 0x1u /* start_pos < 0, bad per-sequence count, or past capacity */
#define TQ_DEV_ERR_SEQ_LEN 0x2u      /* seq_len < 0 or seq_len > capacity (or > max_seq_len) */
#define TQ_DEV_ERR_LAYOUT 0x4u       /* internal: a kernel's shared-memory layout did not fit (not expected) */
#define TQ_DEV_ERR_BLOCK 0x8u        /* paged layout: a block-table entry outside [0, num_blocks) */

/* Human-readable name of a status code (static string, never NULL). */
const char *tq_status_string(tq_status status);

/* ------------------------------------------------------------------------ */
/* Codebook                                                                   */
/* ------------------------------------------------------------------------ */

/*
 * Lloyd-Max scalar codebook for one coordinate of a randomly rotated unit
 * vector in R^d, whose density is f_d(x) = C_d (1 - x^2)^((d-3)/2) on [-1, 1]
 * ([MLX-VLM deep-dive] "How TurboQuant KV Cache Quantization Works": a
 * Beta-PDF-based Lloyd-Max quantizer; [MLX-VLM CLI guide] "What Is
 * TurboQuant?": the codebook generator).  2^bits reconstruction levels in
 * ascending order; thresholds are the midpoints of neighbouring levels.
 * The kernels use the float32 fields; the float64 fields record the fixed
 * point before rounding.
 */
typedef struct tq_codebook {
  int32_t head_dim;
  int32_t bits;               /* 1..4 */
  float centroids[16];        /* first 2^bits used, ascending */
  float thresholds[15];       /* first 2^bits - 1 used: (c[k] + c[k+1]) / 2 */
  double centroids_f64[16];
  double thresholds_f64[15];
  double mse_per_coord;       /* E[(x - c(x))^2] under f_d */
  int32_t iterations;         /* Lloyd iterations taken */
} tq_codebook;

/*
 * Build the codebook for (head_dim, bits).  Host only, synchronous, needs no
 * GPU; takes up to about a second for bits = 4.  Lloyd's two conditions are
 * iterated with cell integrals by composite Gauss-Legendre quadrature until
 * no level moves by more than 1e-15.
 *   head_dim  3 .. 65536 (the density needs d >= 3)
 *   bits      1 .. 4
 *   out       written on success
 * Returns TQ_ERR_INVALID_ARG for a NULL `out`, TQ_ERR_UNSUPPORTED for values
 * outside the ranges above.
 */
tq_status tq_build_codebook(int32_t head_dim, int32_t bits, tq_codebook *out);

/*
 * Fractional bit budget split: K gets floor(bits), V gets ceil(bits)
 * ([MLX-VLM deep-dive] "Quantization Codecs and Bit Splitting").
 * bits must be finite and in (0, 16]; both outputs must be non-NULL.
 */
tq_status tq_split_bits(double bits, int32_t *k_bits, int32_t *v_bits);

/*
 * Whether the TurboQuant scheme is selected ([MLX-VLM CLI guide] "Activation
 * Logic and CLI Integration"): 0 when no bit width is given (has_bits == 0);
 * 1 when the scheme is explicitly "turboquant"; otherwise 1 exactly when
 * `bits` is more than 1e-6 away from the nearest integer.
 */
int32_t tq_turboquant_enabled(double bits, int32_t has_bits, int32_t scheme_is_turboquant);

/*
 * The library's rotation signs for one KV head: out[i] = +1 or -1, i < head_dim.
 * s_i = -1 when bit 63 of SplitMix64's first output from state
 * seed + (layer << 32 | head << 16 | i) is set ([MLX-VLM deep-dive] "How
 * TurboQuant KV Cache Quantization Works" names a deterministic random
 * rotation but no generator; this reading fixes one).  Host only.
 * layer in [0, 2^31), head in [0, 2^16), head_dim in [1, 2^16].
 */
tq_status tq_rotation_signs(uint64_t seed, int32_t layer, int32_t head, int32_t head_dim, int8_t *out);

/* ------------------------------------------------------------------------ */
/* Cache descriptor                                                           */
/* ------------------------------------------------------------------------ */

enum { TQ_K_PACKED = 0, /* K quantized like V (symmetric turbo modes) */
       TQ_K_FP16 = 1,   /* K kept fp16, V packed (the "asym" modes of [mlxcel doc] "Available modes") */
       TQ_KV_INT8 = 2   /* K and V both per-token INT8 absmax, no rotation and no codebook (the int8
                           mode of [mlxcel doc] "Available modes"); k_bits = v_bits = 8 */ };

/*
 * Describes one layer's KV cache.  All pointers are caller-owned device
 * buffers; sizes follow from the shape fields (see tq_cache_buffer_bytes).
 *
 *   k_cache  TQ_K_PACKED: uint32 [B, Hkv, cap, head_dim*k_bits/32] packed codes
 *            TQ_K_FP16:   fp16   [B, Hkv, cap, head_dim]
 *   k_norms  float [B, Hkv, cap] per-token K norms (TQ_K_PACKED only)
 *   v_cache  uint32 [B, Hkv, cap, head_dim*v_bits/32] packed V codes
 *   v_norms  float [B, Hkv, cap]
 *   v_hot    fp16 [B, Hkv, hot_window, head_dim] ring of the newest V tokens
 *            (hot_window > 0 only): position p lives in slot p mod hot_window
 *            ([mlxcel doc] "Available modes", turbo4-delegated: recent V in
 *            fp16, the cold tail packed)
 *   d_status optional device uint32 status word (may be NULL)
 *
 * Packed layout: code i of a token occupies bits [i*b, i*b+b) of that
 * token's bitstream, stream bit j is bit (j mod 32) of word j/32, codes may
 * straddle words ([MLX-VLM deep-dive] "The TurboQuantKVCache Class" and
 * "Manual Cache Operations": packed uint32 buffers, several codes per word).
 * The per-token norm is the correctly rounded float32 of the exact norm.
 *
 * TQ_KV_INT8: k_cache and v_cache hold [B, Hkv, cap, head_dim/4] uint32 words
 * of int8 codes (code i in byte i mod 4 of word i/4, two's complement: the
 * bitstream above with b = 8), and k_norms / v_norms the per-token float32
 * scales s = fp32(max_i |x_i|) / 127; code_i = round-half-even(fp32(x_i) / s)
 * in [-127, 127] (a zero vector has s = 0 and zero codes), dequantized as
 * s * code_i.  The hot V window works as in the packed modes.
 *
 * GQA: query head hq reads KV head hq / (num_q_heads / num_kv_heads).
 */
typedef struct tq_cache_desc {
  int32_t batch;         /* B >= 1 */
  int32_t num_kv_heads;  /* Hkv >= 1 */
  int32_t num_q_heads;   /* Hq, a multiple of Hkv */
  int32_t head_dim;      /* d; the kernels implement d = 128 */
  int32_t capacity;      /* cap >= 1 tokens per (sequence, KV head) */
  int32_t k_mode;        /* TQ_K_PACKED, TQ_K_FP16 or TQ_KV_INT8 */
  int32_t k_bits;        /* 2..4 when K is packed, 8 for TQ_KV_INT8 (ignored for TQ_K_FP16) */
  int32_t v_bits;        /* 2..4, 8 for TQ_KV_INT8 */
  int32_t hot_window;    /* 0 = none; else 1..cap fp16 V ring length */
  int32_t layer;         /* rotation-sign stream, [0, 2^31) */
  uint64_t seed;         /* rotation-sign seed */
  tq_codebook k_cb;      /* built for (head_dim, k_bits) when K is packed (unused for TQ_KV_INT8) */
  tq_codebook v_cb;      /* built for (head_dim, v_bits) (unused for TQ_KV_INT8) */
  void *k_cache;
  float *k_norms;
  void *v_cache;
  float *v_norms;
  void *v_hot;
  uint32_t *d_status;
  /* Sparse-V threshold tau of decode ([mlxcel doc] "Environment variables":
   * a threshold setting whose zero value turns sparse V off).  0 (the default of
   * tq_cache_desc_init) decodes densely.  With 0 < tau <= 1 decode skips the V
   * accumulation of every (token, query head) whose softmax weight relative to
   * the running maximum of its row is below tau; the weight still counts in
   * the normalization.  Each skipped token then has a normalized weight below
   * tau, so each output coordinate moves by at most sum_{p_j < tau} p_j |v_j|
   * from the dense result.  NaN, negative or > 1 values are TQ_ERR_INVALID_ARG. */
  float sparse_v_threshold;
  /* Paged layout (tq_cache_desc_set_paged; all zero / NULL = contiguous).
   * Token t of (sequence b, KV head h) lives in block
   * block_table[b * max_blocks_per_seq + t / block_size] of the pools, at row
   * (block * Hkv + h) * block_size + t % block_size of k_cache, k_norms,
   * v_cache and v_norms.  The fp16 hot ring stays per sequence. */
  int32_t block_size;          /* tokens per block: a power of two in [16, 4096] */
  int32_t max_blocks_per_seq;  /* capacity = max_blocks_per_seq * block_size */
  int32_t num_blocks;          /* blocks in each pool */
  int32_t reserved;
  const int32_t *block_table;  /* device int32 [B, max_blocks_per_seq] */
} tq_cache_desc;

/*
 * Fill the shape and mode fields of `desc`, build both codebooks (host, as
 * tq_build_codebook; none for TQ_KV_INT8, which needs k_bits = v_bits = 8)
 * and set every pointer to NULL.  The caller then sets the buffer pointers.
 * Validates like the launch entry points.
 */
tq_status tq_cache_desc_init(tq_cache_desc *desc, int32_t batch, int32_t num_kv_heads, int32_t num_q_heads,
                             int32_t head_dim, int32_t capacity, int32_t k_mode, int32_t k_bits,
                             int32_t v_bits, int32_t hot_window, uint64_t seed, int32_t layer);

/*
 * Switch a descriptor from tq_cache_desc_init to the paged layout: the
 * packed K/V (or fp16 K) and norm buffers become pools of num_blocks blocks of
 * block_size tokens per KV head, and each sequence maps its positions to
 * blocks through d_block_table (device int32 [B, max_blocks_per_seq], owned
 * by the caller, read at every launch, so blocks can be remapped between
 * calls).  block_size must be a power of two in [16, 4096] and
 * max_blocks_per_seq * block_size must equal the descriptor's capacity
 * (TQ_ERR_INVALID_ARG otherwise).  This is the block-table layout of the
 * serving paths of [mlxcel doc] "Paged cache and server batching" (blocks adopted
 * and donated between sequences; paged decode equal to the contiguous one).
 * A block-table entry outside [0, num_blocks) met by a kernel sets
 * TQ_DEV_ERR_BLOCK and that token is skipped (decode: treated as absent).
 */
tq_status tq_cache_desc_set_paged(tq_cache_desc *desc, int32_t block_size, int32_t max_blocks_per_seq,
                                  int32_t num_blocks, const int32_t *d_block_table);

/*
 * Bytes of each buffer the descriptor needs (0 for a buffer the mode does
 * not use; in the paged layout the pools of num_blocks blocks).  Any output
 * pointer may be NULL.  Host only.
 */
tq_status tq_cache_buffer_bytes(const tq_cache_desc *desc, size_t *k_cache_bytes, size_t *k_norms_bytes,
                                size_t *v_cache_bytes, size_t *v_norms_bytes, size_t *v_hot_bytes);

/* ------------------------------------------------------------------------ */
/* Quantize / append                                                          */
/* ------------------------------------------------------------------------ */

/*
 * Append n_new fp16 token vectors of K and of V to every (sequence, KV head)
 * of the cache, at positions [start_b, start_b + n_new) of sequence b, with
 * start_b = d_start_pos[b] (device int32 [B]).  This is the update step of
 * [MLX-VLM deep-dive] "Manual Cache Operations" (update_and_fetch) and, with
 * start 0, the bulk conversion of an existing fp16 cache.
 *
 * Each packed vector x gets its norm n = ||x|| (correctly rounded float32)
 * and codes of y = R (x / n), R = (1/sqrt(d)) H diag(s): the sign flip, a
 * fast Walsh-Hadamard transform and the 1/sqrt(d) scale ([MLX-VLM
 * deep-dive] "How TurboQuant KV Cache Quantization Works"); code_i is the
 * number of float32 thresholds t_k <= y_i, i.e. the nearest level with ties
 * going up.  K and V of all heads are processed by one launch
 * ([MLX-VLM deep-dive] "Fused vs. Separate Quantization Paths").
 *
 *   k_new, v_new  fp16 device arrays viewed as [B, Hkv, n_new, head_dim] with
 *                 the given element strides (stride over batch, head, token;
 *                 the last dimension is contiguous).  Both use the same
 *                 strides; strides and base pointers must be multiples of 8
 *                 elements / 16 bytes.
 *   n_new         >= 0 (0 is a no-op)
 *   d_start_pos   device int32 [B]: number of tokens already stored for each
 *                 sequence (appends must continue a sequence)
 *   d_num_new     optional device int32 [B] (NULL = n_new for every
 *                 sequence): sequence b appends its first d_num_new[b] <=
 *                 n_new rows, so that sequences of different lengths can be
 *                 filled in one launch (ragged prefill)
 *   stream        CUDA stream
 *
 * TQ_K_FP16: K rows are copied into the fp16 K cache.
 * TQ_KV_INT8: K and V rows get their absmax scale and int8 codes (see the
 * descriptor); no rotation.
 * hot_window W > 0: after the call positions [end - W, end) of V (end =
 * start + n_new) are in the fp16 ring and [0, end - W) are packed; V tokens
 * that leave the ring are quantized before their slot is reused: inside the
 * append launch when n_new <= W (each new row takes exactly one slot), else
 * by one extra launch before the append launch, on the same stream.
 * Appends of at most 16 tokens per sequence use a one-warp-per-vector kernel
 * with the same arithmetic (identical words and norms).
 *
 * A start position < 0, a count outside [0, n_new] or start + count >
 * capacity sets TQ_DEV_ERR_APPEND_RANGE in d_status and skips that sequence.
 * Before any launch: TQ_ERR_CAPACITY for n_new > capacity, TQ_ERR_UNSUPPORTED
 * when B * Hkv * ceil(n_new / 16) * 2 reaches 2^31 (32-bit job indices),
 * TQ_ERR_INVALID_ARG for NULL or misaligned pointers and strides.
 */
tq_status tq_quantize_append(const tq_cache_desc *desc, const void *k_new, const void *v_new, int64_t stride_b,
                             int64_t stride_h, int64_t stride_t, int32_t n_new, const int32_t *d_start_pos,
                             const int32_t *d_num_new, tq_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Decode attention                                                           */
/* ------------------------------------------------------------------------ */

/*
 * Workspace bytes tq_decode_attention needs for this descriptor when no
 * sequence is longer than max_seq_len (>= 0).  Host only; 0 on bad input.
 */
size_t tq_decode_workspace_bytes(const tq_cache_desc *desc, int32_t max_seq_len);

/*
 * One decode step of attention for every query head, reading the packed
 * cache directly ([MLX-VLM deep-dive] "How TurboQuant KV Cache Quantization
 * Works": scores from the compressed form; [MLX-VLM CLI guide] "What Is
 * TurboQuant?": fused scoring kernels with query-head repeat):
 *
 *   out[b, hq] = sum_j softmax_j(q.k_j / sqrt(d)) v_j,   j < seq_len_b
 *
 * with k_j, v_j the dequantized tokens n_j R^T c[codes_j] (or the raw fp16 K
 * in TQ_K_FP16 mode, s_j code_j in TQ_KV_INT8 mode, and the raw fp16 V of the
 * hot ring for the newest min(W, L) positions).  With packed K the query is
 * rotated once and scores are n_j * sum_i (R q)_i c[code_ji] (fp16 and int8 K
 * use the raw query); the softmax runs online over split-K
 * chunks of the context, V is accumulated in the rotated domain and rotated
 * back once per output by a reduction kernel.
 *
 *   q            fp16 device [B, Hq, head_dim] (contiguous)
 *   d_seq_lens   device int32 [B], each in [0, min(capacity, max_seq_len)]
 *   max_seq_len  host upper bound of the lengths (sizes the split grid)
 *   out          float32 device [B, Hq, head_dim]; zeros for an empty sequence
 *   workspace    device scratch of >= tq_decode_workspace_bytes(desc,
 *                max_seq_len) bytes, 16-byte aligned; contents are
 *                overwritten, nothing needs clearing
 *
 * Launches two kernels on `stream`.  A length outside [0, capacity] or above
 * max_seq_len sets TQ_DEV_ERR_SEQ_LEN and that sequence's output is zero.
 */
tq_status tq_decode_attention(const tq_cache_desc *desc, const void *q, const int32_t *d_seq_lens,
                              int32_t max_seq_len, float *out, void *workspace, size_t workspace_bytes,
                              tq_stream_t stream);

/*
 * Attention of the n_query newest tokens of every sequence over the cache, each
 * query causal over the positions up to its own: the multi-token (prefill chunk
 * or speculative verification) counterpart of tq_decode_attention, whose
 * prefill ratios [mlxcel doc] "Measured speed and the memory trade-off" reports
 * for every mode.  The new tokens' K/V must already be appended.  With
 * L_b = d_seq_lens[b], query i (0 <= i < n_query) of sequence b sits at
 * position L_b - n_query + i and
 *
 *   out[b, i, hq] = sum_{j <= L_b - n_query + i} softmax_j(q[b, i, hq].k_j / sqrt(d)) v_j
 *
 * (zeros when L_b - n_query + i < 0), with k_j, v_j as in tq_decode_attention;
 * n_query = 1 computes what tq_decode_attention computes.  Each query token
 * is one more sequence of the split-K work list, so a call costs about
 * n_query decode calls of the same lengths.
 *
 *   q            fp16 device [B, n_query, Hq, head_dim] (contiguous)
 *   n_query      >= 1; B * n_query <= 512
 *   d_seq_lens   device int32 [B]: positions stored per sequence, the new
 *                tokens included; each in [0, min(capacity, max_seq_len)]
 *   out          float32 device [B, n_query, Hq, head_dim]
 *   workspace    >= tq_multi_query_workspace_bytes(desc, n_query, max_seq_len)
 *
 * Errors as tq_decode_attention; TQ_ERR_UNSUPPORTED when B * n_query > 512
 * or, with n_query > 1, when the descriptor's sparse-V threshold is nonzero
 * (several query tokens accumulate V densely).
 */
size_t tq_multi_query_workspace_bytes(const tq_cache_desc *desc, int32_t n_query, int32_t max_seq_len);
tq_status tq_multi_query_attention(const tq_cache_desc *desc, const void *q, int32_t n_query,
                                   const int32_t *d_seq_lens, int32_t max_seq_len, float *out, void *workspace,
                                   size_t workspace_bytes, tq_stream_t stream);

/*
 * Decode attention for callers that cannot allocate device memory.  The pages
 * have no counterpart of this entry point; it exists for hosts that hand a
 * library only input and output pointers (plugin interfaces with no scratch
 * allocator, runtimes whose memory pool owns all of the GPU's memory, serving
 * loops that must not call cudaMalloc because it can synchronize the device
 * and fail under a full pool).  It computes exactly what tq_decode_attention
 * computes, with the same arguments minus the workspace: the split-K partials
 * go to a scratch array of TQ_NO_ALLOC_WORKSPACE_BYTES that the library holds
 * in device memory on every GPU where it is loaded, until the process exits.
 *
 *   Limit      the call needs tq_decode_workspace_bytes(desc, max_seq_len) <=
 *              TQ_NO_ALLOC_WORKSPACE_BYTES; a larger request returns
 *              TQ_ERR_WORKSPACE before any launch.
 *   Device     the current device.  Every call looks up the scratch array's
 *              device address in the current context (a host-side runtime
 *              call that allocates nothing; the first one on a device may
 *              load the library's device code), so make the first call on a
 *              device before any stream capture.
 *   Sharing    every call uses the same array and leaves its contents behind;
 *              nothing in it needs to start at zero.  Calls whose kernels can
 *              overlap on the GPU (different streams, no ordering between
 *              them) race on the array and give wrong results: order them.
 * No cudaMalloc, cudaFree or other allocating call is made.
 */
#define TQ_NO_ALLOC_WORKSPACE_BYTES ((size_t)16 << 20)
tq_status tq_decode_attention_no_alloc(const tq_cache_desc *desc, const void *q, const int32_t *d_seq_lens,
                                       int32_t max_seq_len, float *out, tq_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Dequantize                                                                 */
/* ------------------------------------------------------------------------ */

/*
 * Dequantize positions [token_start, token_start + n_tokens) of sequence b
 * for all KV heads: x_hat = n R^T c[codes] as float32 ([MLX-VLM deep-dive]
 * FAQ "Where is the dequantization logic implemented?"); TQ_KV_INT8: the
 * float32 product s * code.  which = 0 reads
 * K, 1 reads V.  For V with a hot window, positions >= seq_len - min(W,
 * seq_len) return the fp16 ring value; seq_len is the host-known length of
 * sequence b (only used for that split).  TQ_K_FP16 K returns the stored
 * fp16 values.
 *
 *   out  float32 device [Hkv, n_tokens, head_dim]
 * Requires 0 <= token_start, token_start + n_tokens <= capacity and
 * token_start + n_tokens <= seq_len when a hot window is used.
 */
tq_status tq_dequantize(const tq_cache_desc *desc, int32_t which, int32_t b, int32_t seq_len,
                        int32_t token_start, int32_t n_tokens, float *out, tq_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* TQ_H_ */
