"""The C-ABI library on a machine without a GPU: it builds, loads and exports
every declared symbol; its host-side code (codebook builder, signs, bit
helpers, validation, sizes) agrees with the oracle; and the host build of the
kernels' per-vector quantizer reproduces the oracle's words and norms."""
import math
import os
import re

import numpy as np
import pytest

import oracle
from bit_kv_cache_10_gb300 import native as N
from bit_kv_cache_10_gb300 import synth

from helpers import RealBuffers, compare_packed

INCLUDE = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")


@pytest.fixture(scope="session", autouse=True)
def built_library():
    from bit_kv_cache_10_gb300 import build
    build.build()
    N.lib()


def _declared_functions():
    names = set()
    for f in os.listdir(INCLUDE):
        if f.endswith(".h"):
            text = open(os.path.join(INCLUDE, f)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(tq_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_every_declared_symbol_is_exported():
    declared = _declared_functions()
    assert len(declared) >= 11
    lib = N.lib()
    for name in declared:
        assert hasattr(lib, name), name
    assert set(declared) == set(N.EXPORTED)


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
@pytest.mark.parametrize("d", [16, 64, 128, 256])
def test_codebook_matches_oracle(d, bits):
    cb = N.tq_build_codebook(d, bits)
    ref = oracle.codebook(d, bits)
    k = 1 << bits
    np.testing.assert_allclose(np.array(cb.centroids_f64[:k]), ref.centroids, atol=1e-12, rtol=0)
    np.testing.assert_allclose(np.array(cb.thresholds_f64[:k - 1]), ref.thresholds, atol=1e-12, rtol=0)
    np.testing.assert_array_equal(np.array(cb.centroids[:k], np.float32), ref.centroids32)
    np.testing.assert_array_equal(np.array(cb.thresholds[:k - 1], np.float32), ref.thresholds32)
    assert cb.mse_per_coord == pytest.approx(ref.mse_per_coord, rel=1e-10)


def test_codebook_argument_errors():
    with pytest.raises(N.TQError) as e:
        N.tq_build_codebook(2, 3)
    assert e.value.status == N.TQ_ERR_UNSUPPORTED
    with pytest.raises(N.TQError):
        N.tq_build_codebook(128, 5)
    assert N.lib().tq_build_codebook(128, 3, None) == N.TQ_ERR_INVALID_ARG


def test_status_strings():
    """Every status code has its own name; any other value maps to one fallback
    name (never NULL), and an error raised by the binding carries the name."""
    codes = [N.TQ_OK, N.TQ_ERR_INVALID_ARG, N.TQ_ERR_UNSUPPORTED, N.TQ_ERR_CAPACITY, N.TQ_ERR_WORKSPACE,
             N.TQ_ERR_CUDA, N.TQ_ERR_DEVICE]
    names = [N.tq_status_string(c) for c in codes]
    assert names[0] == "TQ_OK" and len(set(names)) == len(codes)
    assert all(n.startswith("TQ_") for n in names)
    assert N.tq_status_string(42) == N.tq_status_string(-99) == "TQ_ERR_UNKNOWN"
    assert "TQ_ERR_UNKNOWN" not in names
    with pytest.raises(N.TQError) as e:
        N.tq_build_codebook(2, 3)
    assert "TQ_ERR_UNSUPPORTED" in str(e.value)


@pytest.mark.parametrize("seed,layer,head", [(0, 0, 0), (0, 0, 7), (123456789, 3, 2), (2**63 + 5, 31, 65535)])
def test_rotation_signs_match_oracle(seed, layer, head):
    np.testing.assert_array_equal(np.array(N.tq_rotation_signs(seed, layer, head, 128)),
                                  oracle.rotation_signs(seed, layer, head, 128))


def test_bit_split_and_scheme_gate_match_pages():
    for bits in (2.5, 3, 3.5, 4, 4.2):
        assert N.tq_split_bits(bits) == oracle.split_bits(bits)
    for bits, scheme in [(None, None), (None, "turboquant"), (4, "turboquant"), (3.5, None), (4, None),
                         (4.0000001, None), (4.2, None), (2, "uniform")]:
        assert N.tq_turboquant_enabled(bits, scheme) == oracle.turboquant_enabled(bits, scheme)
    with pytest.raises(N.TQError):
        N.tq_split_bits(float("nan"))


def test_descriptor_validation():
    # head_dim 80 (the pages' Phi-2 example) is not a power of two: rejected, not padded
    for d in (80, 96, 64, 256):
        with pytest.raises(N.TQError) as e:
            N.tq_cache_desc_init(1, 8, 32, d, 16, N.TQ_K_PACKED, 3, 4)
        assert e.value.status == N.TQ_ERR_UNSUPPORTED
    for kb, vb in [(1, 4), (5, 4), (3, 1), (3, 8)]:
        with pytest.raises(N.TQError) as e:
            N.tq_cache_desc_init(1, 8, 32, 128, 16, N.TQ_K_PACKED, kb, vb)
        assert e.value.status == N.TQ_ERR_UNSUPPORTED
    with pytest.raises(N.TQError) as e:
        N.tq_cache_desc_init(1, 8, 30, 128, 16, N.TQ_K_PACKED, 3, 4)
    assert e.value.status == N.TQ_ERR_INVALID_ARG
    with pytest.raises(N.TQError) as e:
        N.tq_cache_desc_init(1, 4, 32, 128, 16, N.TQ_K_PACKED, 3, 4)  # 8 query heads per KV head
    assert e.value.status == N.TQ_ERR_UNSUPPORTED
    with pytest.raises(N.TQError) as e:
        N.tq_cache_desc_init(1, 8, 32, 128, 16, N.TQ_K_PACKED, 3, 4, hot_window=17)
    assert e.value.status == N.TQ_ERR_INVALID_ARG
    d = N.tq_cache_desc_init(2, 8, 32, 128, 4096, N.TQ_K_PACKED, 3, 4, hot_window=256, seed=9, layer=1)
    assert (d.k_bits, d.v_bits, d.hot_window, d.seed, d.layer) == (3, 4, 256, 9, 1)


def test_entry_points_reject_bad_arguments_before_launch():
    B, HK, HQ, CAP = 1, 8, 32, 64
    d = N.tq_cache_desc_init(B, HK, HQ, 128, CAP, N.TQ_K_PACKED, 3, 4)
    # buffers not set: every launching entry point refuses without touching the GPU
    L = N.lib()
    assert L.tq_quantize_append(d, None, None, 0, 0, 0, 1, None, None, None) == N.TQ_ERR_INVALID_ARG
    assert L.tq_decode_attention(d, None, None, 4, None, None, 0, None) == N.TQ_ERR_INVALID_ARG
    assert L.tq_dequantize(d, 0, 0, 0, 0, 1, None, None) == N.TQ_ERR_INVALID_ARG
    # real buffers of the sizes each call would use; validation must refuse before any launch
    mem = RealBuffers()
    mem.cache(d)
    new = mem.alloc(B * HK * (CAP + 1) * 128 * 2)  # fp16 [B, Hkv, 65, d]
    pos = mem.alloc(4 * B)
    q = mem.alloc(B * HQ * 128 * 2)
    lens = mem.alloc(4 * B)
    out = mem.alloc(B * HQ * 128 * 4)
    ws_need = N.tq_decode_workspace_bytes(d, CAP)
    ws = mem.alloc(ws_need)
    deq = mem.alloc(HK * 5 * 128 * 4)
    assert L.tq_quantize_append(d, new, new, 0, 0, 0, -1, pos, None, None) == N.TQ_ERR_INVALID_ARG
    assert L.tq_quantize_append(d, new, new, 0, 0, 0, CAP + 1, pos, None, None) == N.TQ_ERR_CAPACITY
    assert L.tq_quantize_append(d, new + 8, new, 0, 0, 0, 1, pos, None, None) == N.TQ_ERR_INVALID_ARG
    assert L.tq_quantize_append(d, new, new, 0, 0, 3, 1, pos, None, None) == N.TQ_ERR_INVALID_ARG
    assert L.tq_decode_attention(d, q, lens, CAP, out, ws, 16, None) == N.TQ_ERR_WORKSPACE
    assert L.tq_decode_attention(d, q, lens, CAP, out, None, ws_need, None) == N.TQ_ERR_WORKSPACE
    assert L.tq_dequantize(d, 2, 0, 0, 0, 1, deq, None) == N.TQ_ERR_INVALID_ARG
    assert L.tq_dequantize(d, 0, 0, 0, CAP - 4, 5, deq, None) == N.TQ_ERR_CAPACITY
    k_norms = d.k_norms
    d.k_norms = k_norms + 4
    assert L.tq_quantize_append(d, new, new, 0, 0, 0, 1, pos, None, None) == N.TQ_ERR_INVALID_ARG
    d.k_norms = k_norms
    # the sparse-V threshold must lie in [0, 1] (NaN included in the refusal)
    for tau in (float("nan"), -1e-6, 1.5, float("inf")):
        d.sparse_v_threshold = tau
        assert L.tq_decode_attention(d, q, lens, CAP, out, ws, ws_need, None) == N.TQ_ERR_INVALID_ARG
    assert N.tq_cache_desc_init(1, 8, 32, 128, 64, N.TQ_K_PACKED, 3, 4).sparse_v_threshold == 0.0


def test_workspace_and_buffer_sizes():
    d = N.tq_cache_desc_init(4, 8, 32, 128, 131072, N.TQ_K_PACKED, 3, 4, hot_window=256)
    # one partial of 4 query heads per (split-K CTA, row) pair: 512 CTAs + cold and hot rows of 4 x 8 (b, h)
    assert N.tq_decode_workspace_bytes(d, 131072) == (512 + 2 * 4 * 8) * 4 * 130 * 4
    assert N.tq_decode_workspace_bytes(d, 7) == N.tq_decode_workspace_bytes(d, 131072)
    assert N.tq_decode_workspace_bytes(d, 0) == 0
    sizes = N.tq_cache_buffer_bytes(d)
    rows = 4 * 8 * 131072
    assert sizes == {"k_cache": rows * 48, "k_norms": rows * 4, "v_cache": rows * 64, "v_norms": rows * 4,
                     "v_hot": 4 * 8 * 256 * 256}
    # bytes per token-head equal the oracle's storage formula
    assert (sizes["k_cache"] + sizes["k_norms"]) // rows == oracle.bytes_per_token_head(3, 128)
    assert (sizes["v_cache"] + sizes["v_norms"]) // rows == oracle.bytes_per_token_head(4, 128)
    a = N.tq_cache_desc_init(8, 8, 32, 128, 16384, N.TQ_K_FP16, 0, 4)
    assert N.tq_cache_buffer_bytes(a)["k_cache"] == 8 * 8 * 16384 * 256


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_host_build_of_kernel_quantizer_matches_oracle(bits):
    x = synth.kv_fp16(5, synth.STREAM_K, 1, 2, 3000, 128, scales=synth.channel_scales(5, 4, 2, 128))
    cb = N.tq_build_codebook(128, bits)
    ref_cb = oracle.codebook(128, bits)
    for h in range(2):
        words, norms = N.tq_debug_quantize_rows_host(cb, 7, 2, h, x[0, h])
        codes, ref_n, y = oracle.quantize_rows(x[0, h], oracle.rotation(7, 2, h, 128), ref_cb)
        np.testing.assert_array_equal(norms, ref_n)
        compare_packed(words, oracle.pack(codes, bits), y, bits, ref_cb.thresholds32, "bits %d head %d" % (bits, h))


def test_host_quantizer_special_vectors():
    cb = N.tq_build_codebook(128, 3)
    rows = np.zeros((6, 128), np.float16)
    rows[1, 0] = 1.0                        # one-hot
    rows[2, :4] = [1.0, 2.0 ** -12, 2.0 ** -12, 2.0 ** -24]  # |x|^2 = (1 + 2^-24)^2 exactly: a rounding tie
    rows[3, :] = 65504.0                    # largest fp16
    rows[4, :] = 2.0 ** -24                 # smallest subnormal
    rows[5, ::2] = -3.0
    words, norms = N.tq_debug_quantize_rows_host(cb, 0, 0, 0, rows)
    codes, ref_n, y = oracle.quantize_rows(rows, oracle.rotation(0, 0, 0, 128), oracle.codebook(128, 3))
    np.testing.assert_array_equal(norms, ref_n)
    assert norms[2] == np.float32(1.0)      # tie goes to the even neighbour
    assert norms[0] == 0 and np.all(oracle.unpack(words[:1], 3, 128) == 4)
    compare_packed(words, oracle.pack(codes, 3), y, 3, oracle.codebook(128, 3).thresholds32, "special")


def test_paged_layout_validation_and_pool_sizes():
    d = N.tq_cache_desc_init(2, 8, 32, 128, 4096, N.TQ_K_PACKED, 3, 4, hot_window=64)
    mem = RealBuffers()
    tab = mem.alloc(2 * 4096 // 8 * 4)  # the largest table of the cases below
    for bs, mb, nb, t in [(24, 4096 // 24, 10, tab), (8, 512, 10, tab), (8192, 1, 10, tab),
                          (64, 63, 10, tab), (64, 64, 0, tab), (64, 64, 10, None), (64, 64, 10, tab + 2)]:
        with pytest.raises(N.TQError) as e:
            N.tq_cache_desc_set_paged(d, bs, mb, nb, t)
        assert e.value.status == N.TQ_ERR_INVALID_ARG
    N.tq_cache_desc_set_paged(d, 64, 64, 200, tab)
    assert (d.block_size, d.max_blocks_per_seq, d.num_blocks, d.block_table) == (64, 64, 200, tab)
    sizes = N.tq_cache_buffer_bytes(d)
    rows = 200 * 8 * 64  # pools of 200 blocks of 64 tokens per KV head
    assert sizes == {"k_cache": rows * 48, "k_norms": rows * 4, "v_cache": rows * 64, "v_norms": rows * 4,
                     "v_hot": 2 * 8 * 64 * 256}
    # a corrupted paged descriptor (no table) is refused before any launch
    L = N.lib()
    mem.cache(d)
    d.block_table = None
    q, lens, out = mem.alloc(2 * 32 * 128 * 2), mem.alloc(8), mem.alloc(2 * 32 * 128 * 4)
    need = N.tq_decode_workspace_bytes(d, 64)
    assert L.tq_decode_attention(d, q, lens, 64, out, mem.alloc(need), need, None) == N.TQ_ERR_INVALID_ARG


def test_int8_mode_descriptor_and_sizes():
    d = N.tq_cache_desc_init(4, 8, 32, 128, 4096, N.TQ_KV_INT8, 8, 8)
    rows = 4 * 8 * 4096
    sizes = N.tq_cache_buffer_bytes(d)
    # 128 one-byte codes and a float32 scale per token-head (the ~2x of the int8 mode)
    assert sizes == {"k_cache": rows * 128, "k_norms": rows * 4, "v_cache": rows * 128, "v_norms": rows * 4,
                     "v_hot": 0}
    assert (sizes["k_cache"] + sizes["k_norms"]) // rows == 128 + 4
    for kb, vb in ((4, 8), (8, 4), (8, 3), (16, 8)):
        with pytest.raises(N.TQError) as e:
            N.tq_cache_desc_init(4, 8, 32, 128, 4096, N.TQ_KV_INT8, kb, vb)
        assert e.value.status == N.TQ_ERR_UNSUPPORTED
    with pytest.raises(N.TQError):  # a mode value the library does not know
        N.tq_cache_desc_init(4, 8, 32, 128, 4096, 3, 8, 8)


def test_multi_query_arguments_and_workspace():
    d = N.tq_cache_desc_init(4, 8, 32, 128, 4096, N.TQ_K_PACKED, 3, 4, hot_window=256)
    # one partial slot per (split CTA, row): rows = 2 (cold, hot) x B x n_query x Hkv
    per_slot = 4 * (128 + 2) * 4
    assert N.tq_multi_query_workspace_bytes(d, 1, 100) == N.tq_decode_workspace_bytes(d, 100)
    assert N.tq_multi_query_workspace_bytes(d, 8, 100) == (512 + 2 * 4 * 8 * 8) * per_slot
    assert N.tq_multi_query_workspace_bytes(d, 0, 100) == 0
    L = N.lib()
    mem = RealBuffers()
    mem.cache(d)
    B, HQ = 4, 32
    q = mem.alloc(B * 129 * HQ * 128 * 2)  # room for the largest query count of the cases below
    lens = mem.alloc(4 * B)
    out = mem.alloc(B * 129 * HQ * 128 * 4)
    big = N.tq_multi_query_workspace_bytes(d, 129, 64)
    ws = mem.alloc(big)
    assert L.tq_multi_query_attention(d, q, 0, lens, 64, out, ws, big, None) == N.TQ_ERR_INVALID_ARG
    assert L.tq_multi_query_attention(d, q, 129, lens, 64, out, ws, big, None) == N.TQ_ERR_UNSUPPORTED
    assert L.tq_multi_query_attention(d, q + 8, 2, lens, 64, out, ws, big, None) == N.TQ_ERR_INVALID_ARG
    need = N.tq_multi_query_workspace_bytes(d, 4, 64)
    assert L.tq_multi_query_attention(d, q, 4, lens, 64, out, ws, need - 16, None) == N.TQ_ERR_WORKSPACE


def test_multi_query_refuses_sparse_v():
    d = N.tq_cache_desc_init(2, 8, 32, 128, 4096, N.TQ_K_PACKED, 3, 4)
    mem = RealBuffers()
    mem.cache(d)
    d.sparse_v_threshold = 1e-3
    q, lens, out = mem.alloc(2 * 4 * 32 * 128 * 2), mem.alloc(8), mem.alloc(2 * 4 * 32 * 128 * 4)
    need = N.tq_multi_query_workspace_bytes(d, 4, 64)
    L = N.lib()
    assert L.tq_multi_query_attention(d, q, 4, lens, 64, out, mem.alloc(need), need, None) == N.TQ_ERR_UNSUPPORTED
