"""ctypes binding of the C ABI in ``include/tq.h`` (argument marshalling only).

Every function here forwards to ``libtq.so`` with the same name.  Device
buffers are passed as integer device pointers (``tensor.data_ptr()``) and
streams as raw ``cudaStream_t`` handles.  Loading fails loudly if the library
has not been built; there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import (POINTER, c_double, c_float, c_int8, c_int32, c_int64, c_size_t, c_uint8, c_uint16, c_uint32, c_uint64,
                    c_void_p)

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libtq.so")

TQ_OK = 0
TQ_ERR_INVALID_ARG = -1
TQ_ERR_UNSUPPORTED = -2
TQ_ERR_CAPACITY = -3
TQ_ERR_WORKSPACE = -4
TQ_ERR_CUDA = -5
TQ_ERR_DEVICE = -6
TQ_K_PACKED = 0
TQ_K_FP16 = 1
TQ_KV_INT8 = 2
TQ_DEV_ERR_APPEND_RANGE = 0x1
TQ_DEV_ERR_SEQ_LEN = 0x2

# every symbol the public headers declare (include/tq.h, include/tq_debug.h)
EXPORTED = (
    "tq_status_string", "tq_build_codebook", "tq_split_bits", "tq_turboquant_enabled", "tq_rotation_signs",
    "tq_cache_desc_init", "tq_cache_buffer_bytes", "tq_quantize_append", "tq_decode_workspace_bytes",
    "tq_decode_attention", "tq_dequantize", "tq_debug_quantize_rows_host", "tq_decode_attention_no_alloc",
    "tq_cache_desc_set_paged", "tq_multi_query_workspace_bytes", "tq_multi_query_attention",
    "tq_debug_set_decode_path", "tq_debug_split_plan",
)
TQ_DEV_ERR_APPEND_RANGE, TQ_DEV_ERR_SEQ_LEN, TQ_DEV_ERR_LAYOUT, TQ_DEV_ERR_BLOCK = 0x1, 0x2, 0x4, 0x8
TQ_NO_ALLOC_WORKSPACE_BYTES = 16 << 20


class TQCodebook(ctypes.Structure):
    _fields_ = [
        ("head_dim", c_int32), ("bits", c_int32),
        ("centroids", c_float * 16), ("thresholds", c_float * 15),
        ("centroids_f64", c_double * 16), ("thresholds_f64", c_double * 15),
        ("mse_per_coord", c_double), ("iterations", c_int32),
    ]


class TQCacheDesc(ctypes.Structure):
    _fields_ = [
        ("batch", c_int32), ("num_kv_heads", c_int32), ("num_q_heads", c_int32), ("head_dim", c_int32),
        ("capacity", c_int32), ("k_mode", c_int32), ("k_bits", c_int32), ("v_bits", c_int32),
        ("hot_window", c_int32), ("layer", c_int32), ("seed", c_uint64),
        ("k_cb", TQCodebook), ("v_cb", TQCodebook),
        ("k_cache", c_void_p), ("k_norms", c_void_p), ("v_cache", c_void_p), ("v_norms", c_void_p),
        ("v_hot", c_void_p), ("d_status", c_void_p), ("sparse_v_threshold", ctypes.c_float),
        ("block_size", c_int32), ("max_blocks_per_seq", c_int32), ("num_blocks", c_int32), ("reserved", c_int32),
        ("block_table", c_void_p),
    ]


class TQError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__("%s failed: %s (%d)" % (what, tq_status_string(status), status))
        self.status = status


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library (loads it on first use; raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libtq.so is not built (%s); run bit_kv_cache_10_gb300.build.build()" % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        L.tq_status_string.restype = ctypes.c_char_p
        L.tq_status_string.argtypes = [c_int32]
        L.tq_build_codebook.restype = c_int32
        L.tq_build_codebook.argtypes = [c_int32, c_int32, POINTER(TQCodebook)]
        L.tq_split_bits.restype = c_int32
        L.tq_split_bits.argtypes = [c_double, POINTER(c_int32), POINTER(c_int32)]
        L.tq_turboquant_enabled.restype = c_int32
        L.tq_turboquant_enabled.argtypes = [c_double, c_int32, c_int32]
        L.tq_rotation_signs.restype = c_int32
        L.tq_rotation_signs.argtypes = [c_uint64, c_int32, c_int32, c_int32, POINTER(c_int8)]
        L.tq_cache_desc_init.restype = c_int32
        L.tq_cache_desc_init.argtypes = [POINTER(TQCacheDesc)] + [c_int32] * 9 + [c_uint64, c_int32]
        L.tq_cache_desc_set_paged.restype = c_int32
        L.tq_cache_desc_set_paged.argtypes = [POINTER(TQCacheDesc), c_int32, c_int32, c_int32, c_void_p]
        L.tq_cache_buffer_bytes.restype = c_int32
        L.tq_cache_buffer_bytes.argtypes = [POINTER(TQCacheDesc)] + [POINTER(c_size_t)] * 5
        L.tq_quantize_append.restype = c_int32
        L.tq_quantize_append.argtypes = [POINTER(TQCacheDesc), c_void_p, c_void_p, c_int64, c_int64, c_int64,
                                         c_int32, c_void_p, c_void_p, c_void_p]
        L.tq_decode_workspace_bytes.restype = c_size_t
        L.tq_decode_workspace_bytes.argtypes = [POINTER(TQCacheDesc), c_int32]
        L.tq_decode_attention.restype = c_int32
        L.tq_decode_attention.argtypes = [POINTER(TQCacheDesc), c_void_p, c_void_p, c_int32, c_void_p, c_void_p,
                                          c_size_t, c_void_p]
        L.tq_multi_query_workspace_bytes.restype = c_size_t
        L.tq_multi_query_workspace_bytes.argtypes = [POINTER(TQCacheDesc), c_int32, c_int32]
        L.tq_multi_query_attention.restype = c_int32
        L.tq_multi_query_attention.argtypes = [POINTER(TQCacheDesc), c_void_p, c_int32, c_void_p, c_int32, c_void_p,
                                               c_void_p, c_size_t, c_void_p]
        L.tq_decode_attention_no_alloc.restype = c_int32
        L.tq_decode_attention_no_alloc.argtypes = [POINTER(TQCacheDesc), c_void_p, c_void_p, c_int32, c_void_p,
                                                   c_void_p]
        L.tq_dequantize.restype = c_int32
        L.tq_dequantize.argtypes = [POINTER(TQCacheDesc), c_int32, c_int32, c_int32, c_int32, c_int32, c_void_p,
                                    c_void_p]
        L.tq_debug_set_decode_path.restype = None
        L.tq_debug_set_decode_path.argtypes = [c_int32]
        L.tq_debug_split_plan.restype = c_int32
        L.tq_debug_split_plan.argtypes = [POINTER(c_int32), POINTER(c_int32), c_int32, c_int32, c_int32, c_int32,
                                          c_int32, POINTER(c_int64), POINTER(c_uint8)]
        L.tq_debug_quantize_rows_host.restype = c_int32
        L.tq_debug_quantize_rows_host.argtypes = [POINTER(TQCodebook), c_uint64, c_int32, c_int32, POINTER(c_uint16),
                                                  c_int32, POINTER(c_uint32), POINTER(c_float)]
        _lib = L
    return _lib


def _check(status: int, what: str) -> None:
    if status != TQ_OK:
        raise TQError(status, what)


def tq_status_string(status: int) -> str:
    return lib().tq_status_string(status).decode()


def tq_build_codebook(head_dim: int, bits: int) -> TQCodebook:
    cb = TQCodebook()
    _check(lib().tq_build_codebook(head_dim, bits, ctypes.byref(cb)), "tq_build_codebook")
    return cb


def tq_split_bits(bits: float) -> tuple[int, int]:
    k, v = c_int32(), c_int32()
    _check(lib().tq_split_bits(bits, ctypes.byref(k), ctypes.byref(v)), "tq_split_bits")
    return k.value, v.value


def tq_turboquant_enabled(bits, scheme=None) -> bool:
    has = bits is not None
    return bool(lib().tq_turboquant_enabled(float(bits) if has else 0.0, int(has), int(scheme == "turboquant")))


def tq_rotation_signs(seed: int, layer: int, head: int, head_dim: int):
    buf = (c_int8 * head_dim)()
    _check(lib().tq_rotation_signs(seed, layer, head, head_dim, buf), "tq_rotation_signs")
    return list(buf)


def tq_cache_desc_init(batch, num_kv_heads, num_q_heads, head_dim, capacity, k_mode, k_bits, v_bits,
                       hot_window=0, seed=0, layer=0) -> TQCacheDesc:
    d = TQCacheDesc()
    _check(lib().tq_cache_desc_init(ctypes.byref(d), batch, num_kv_heads, num_q_heads, head_dim, capacity, k_mode,
                                    k_bits, v_bits, hot_window, seed, layer), "tq_cache_desc_init")
    return d


def tq_cache_desc_set_paged(desc: TQCacheDesc, block_size: int, max_blocks_per_seq: int, num_blocks: int,
                            block_table_ptr: int) -> None:
    _check(lib().tq_cache_desc_set_paged(ctypes.byref(desc), block_size, max_blocks_per_seq, num_blocks,
                                         block_table_ptr), "tq_cache_desc_set_paged")


def tq_cache_buffer_bytes(desc: TQCacheDesc) -> dict:
    vals = [c_size_t() for _ in range(5)]
    _check(lib().tq_cache_buffer_bytes(ctypes.byref(desc), *[ctypes.byref(v) for v in vals]), "tq_cache_buffer_bytes")
    return dict(zip(("k_cache", "k_norms", "v_cache", "v_norms", "v_hot"), (v.value for v in vals)))


def tq_quantize_append(desc, k_new_ptr, v_new_ptr, stride_b, stride_h, stride_t, n_new, d_start_pos_ptr,
                       d_num_new_ptr, stream):
    _check(lib().tq_quantize_append(ctypes.byref(desc), k_new_ptr, v_new_ptr, stride_b, stride_h, stride_t, n_new,
                                    d_start_pos_ptr, d_num_new_ptr, stream), "tq_quantize_append")


def tq_decode_workspace_bytes(desc, max_seq_len: int) -> int:
    return int(lib().tq_decode_workspace_bytes(ctypes.byref(desc), max_seq_len))


def tq_decode_attention(desc, q_ptr, d_seq_lens_ptr, max_seq_len, out_ptr, ws_ptr, ws_bytes, stream):
    _check(lib().tq_decode_attention(ctypes.byref(desc), q_ptr, d_seq_lens_ptr, max_seq_len, out_ptr, ws_ptr,
                                     ws_bytes, stream), "tq_decode_attention")


def tq_multi_query_workspace_bytes(desc, n_query: int, max_seq_len: int) -> int:
    return int(lib().tq_multi_query_workspace_bytes(ctypes.byref(desc), n_query, max_seq_len))


def tq_multi_query_attention(desc, q_ptr, n_query, d_seq_lens_ptr, max_seq_len, out_ptr, ws_ptr, ws_bytes, stream):
    _check(lib().tq_multi_query_attention(ctypes.byref(desc), q_ptr, n_query, d_seq_lens_ptr, max_seq_len, out_ptr,
                                          ws_ptr, ws_bytes, stream), "tq_multi_query_attention")


def tq_decode_attention_no_alloc(desc, q_ptr, d_seq_lens_ptr, max_seq_len, out_ptr, stream):
    """Decode attention with the library's fixed device scratch (no workspace argument)."""
    _check(lib().tq_decode_attention_no_alloc(ctypes.byref(desc), q_ptr, d_seq_lens_ptr, max_seq_len, out_ptr,
                                              stream), "tq_decode_attention_no_alloc")


def tq_dequantize(desc, which, b, seq_len, token_start, n_tokens, out_ptr, stream):
    _check(lib().tq_dequantize(ctypes.byref(desc), which, b, seq_len, token_start, n_tokens, out_ptr, stream),
           "tq_dequantize")


def tq_debug_quantize_rows_host(cb: TQCodebook, seed: int, layer: int, head: int, rows_fp16):
    """Host build of the kernels' per-vector quantizer (verification only).
    ``rows_fp16``: numpy float16 [n, 128].  Returns (words uint32 [n, bits*4], norms float32 [n])."""
    import numpy as np

    rows = np.ascontiguousarray(rows_fp16, dtype=np.float16)
    n = rows.shape[0]
    words = np.zeros((n, cb.bits * 4), np.uint32)
    norms = np.zeros(n, np.float32)
    _check(lib().tq_debug_quantize_rows_host(
        ctypes.byref(cb), seed, layer, head, rows.view(np.uint16).ctypes.data_as(POINTER(c_uint16)), n,
        words.ctypes.data_as(POINTER(c_uint32)), norms.ctypes.data_as(POINTER(c_float))), "tq_debug_quantize_rows_host")
    return words, norms


def tq_debug_set_decode_path(path: int) -> None:
    """Decode path for tests (process-wide): 0 automatic, 1 persistent split-K
    kernel + merge kernel, 2 the thread-block-cluster variant where allowed."""
    lib().tq_debug_set_decode_path(int(path))


def tq_debug_split_plan(tiles_cold, tiles_hot, hkv: int, grid: int, price_cold: int, price_hot: int,
                        with_segments: bool = True):
    """Host computation of the persistent decode path's split (verification only).
    ``tiles_cold`` / ``tiles_hot``: per work-list sequence, the cold and hot tiles
    of each of its hkv rows; ``price_cold`` / ``price_hot``: tiles' worth of a
    cold / hot segment start.  Returns (starts int64 [grid + 1], seg_ctas uint8
    [2 nv hkv, grid] or None): CTA c takes tiles [starts[c], starts[c + 1]);
    seg_ctas[2 r + part, c] = 1 when the merge reads CTA c for that row part."""
    import numpy as np

    tc = np.ascontiguousarray(tiles_cold, dtype=np.int32)
    th = np.ascontiguousarray(tiles_hot, dtype=np.int32)
    nv = tc.shape[0]
    starts = np.zeros(grid + 1, np.int64)
    seg = np.zeros((2 * nv * hkv, grid), np.uint8) if with_segments else None
    _check(lib().tq_debug_split_plan(
        tc.ctypes.data_as(POINTER(c_int32)), th.ctypes.data_as(POINTER(c_int32)), nv, hkv, grid, price_cold, price_hot,
        starts.ctypes.data_as(POINTER(c_int64)),
        seg.ctypes.data_as(POINTER(c_uint8)) if seg is not None else None), "tq_debug_split_plan")
    return starts, seg
