"""GPU parity of the per-token INT8 absmax mode (the int8 mode of the mlxcel
page, "Available modes") through the C ABI against the oracle.

Scales and codes are decided in float32 on both sides (the scale absmax / 127
and the quotient x / s are IEEE divisions, rounded half to even), so words and
scales must be bit-exact; dequantized values are float32 products s * code and
must be bit-exact too; attention outputs must agree within 2e-3 max-abs and
1e-3 relative-L2 of the float64 oracle.
"""
import numpy as np
import pytest

import oracle
from bit_kv_cache_10_gb300 import native as N
from bit_kv_cache_10_gb300 import synth

from helpers import assert_attention_close

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

D = 128


@pytest.fixture(scope="module", autouse=True)
def gpu_library():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from bit_kv_cache_10_gb300 import build
    build.build()
    N.lib()


def _cache(**kw):
    from bit_kv_cache_10_gb300.cache import TurboQuantKVCache
    return TurboQuantKVCache(bits="int8", **kw)


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def upload(tc, oc):
    tc.k_cache.copy_(_dev(oc.k_words.view(np.int32)))
    tc.k_norms.copy_(_dev(oc.k_norms))
    tc.v_cache.copy_(_dev(oc.v_words.view(np.int32)))
    tc.v_norms.copy_(_dev(oc.v_norms))
    if oc.v_hot is not None:
        tc.v_hot.copy_(_dev(oc.v_hot))
    torch.cuda.synchronize()


def check_rows(tc, x16, which, lengths, what):
    """GPU words and scales of positions [0, L_b) equal the oracle's, bit for bit."""
    gw = (tc.k_cache if which == 0 else tc.v_cache).cpu().numpy().view(np.uint32)
    gs = (tc.k_norms if which == 0 else tc.v_norms).cpu().numpy()
    for b in range(x16.shape[0]):
        L = int(lengths[b])
        for h in range(x16.shape[1]):
            codes, s = oracle.int8_quantize_rows(x16[b, h, :L])
            np.testing.assert_array_equal(gs[b, h, :L], s, err_msg="%s scales b=%d h=%d" % (what, b, h))
            np.testing.assert_array_equal(gw[b, h, :L], oracle.int8_words(codes),
                                          err_msg="%s codes b=%d h=%d" % (what, b, h))


def decode_both(tc, oc, q16, lengths, max_len, pairs=None):
    got = tc.decode(_dev(q16), _dev(np.asarray(lengths, np.int32)), max_len).cpu().numpy()
    ref = oracle.decode_attention(oc, q16, lengths, pairs)
    if pairs is not None:
        idx = tuple(np.array(pairs).T)
        return got[idx], ref[idx]
    return got, ref


def test_int8_llama_like_layer():
    """Llama-3-8B-like layer (B1, 32 q / 8 KV heads, context 4096): append,
    bit-exact codes and scales, decode and dequantize."""
    B, HQ, HK, L = 1, 32, 8, 4096
    k = synth.kv_fp16(2, synth.STREAM_K, B, HK, L, D, synth.channel_scales(2, synth.STREAM_SCALE_K, HK, D))
    v = synth.kv_fp16(2, synth.STREAM_V, B, HK, L, D, synth.channel_scales(2, synth.STREAM_SCALE_V, HK, D))
    q = synth.queries_fp16(2, B, HQ, D)
    tc = _cache(batch=B, num_kv_heads=HK, num_q_heads=HQ, capacity=L)
    tc.append(_dev(k), _dev(v), _dev(np.zeros(B, np.int32)))
    assert tc.device_status() == 0
    check_rows(tc, k, 0, [L], "K")
    check_rows(tc, v, 1, [L], "V")
    oc = oracle.build_cache(k, v, [L], L, 8, 8, codec="int8")
    got, ref = decode_both(tc, oc, q, [L], L)
    assert_attention_close(got, ref, "int8 decode")
    for which in (0, 1):
        g = tc.dequantize(which, 0, L, 100, 3000).cpu().numpy()
        for h in range(HK):
            kr, vr = oracle.dequantized_kv(oc, 0, h, L)
            ref_h = (kr if which == 0 else vr)[100:3100].astype(np.float32)  # exact products, rounded once
            np.testing.assert_array_equal(g[h], ref_h)


def test_int8_ragged_append_hot_window():
    """Ragged prefill, then token-by-token appends that push V out of a 64-token ring."""
    B, HQ, HK, CAP, W, STEPS = 3, 16, 4, 1500, 64, 9
    lens = np.array([1500, 700, 80], np.int32)
    k = synth.kv_fp16(12, synth.STREAM_K, B, HK, CAP, D, synth.channel_scales(12, 4, HK, D))
    v = synth.kv_fp16(12, synth.STREAM_V, B, HK, CAP, D, synth.channel_scales(12, 5, HK, D))
    q = synth.queries_fp16(12, B, HQ, D)
    tc = _cache(batch=B, num_kv_heads=HK, num_q_heads=HQ, capacity=CAP, hot_window=W)
    kd, vd = _dev(k), _dev(v)
    pre = lens - STEPS
    tc.append(kd, vd, _dev(np.zeros(B, np.int32)), _dev(pre))
    for s in range(STEPS):
        start = (pre + s).astype(np.int32)
        kn = torch.stack([kd[b, :, int(start[b])] for b in range(B)])[:, :, None].contiguous()
        vn = torch.stack([vd[b, :, int(start[b])] for b in range(B)])[:, :, None].contiguous()
        tc.append(kn, vn, _dev(start))
    assert tc.device_status() == 0
    check_rows(tc, k, 0, lens, "ragged K")
    check_rows(tc, v, 1, lens - np.minimum(W, lens), "ragged cold V")
    oc = oracle.build_cache(k, v, lens, CAP, 8, 8, hot_window=W, codec="int8")
    np.testing.assert_array_equal(tc.v_hot.cpu().numpy(), oc.v_hot)
    got, ref = decode_both(tc, oc, q, lens, CAP)
    assert_attention_close(got, ref, "int8 ragged decode")
    gv = tc.dequantize(1, 1, 700, 600, 100).cpu().numpy()  # 636 .. 699 come from the ring
    for h in range(HK):
        _, vr = oracle.dequantized_kv(oc, 1, h, 700)
        np.testing.assert_array_equal(gv[h], vr[600:700].astype(np.float32))


@pytest.mark.parametrize("hq", [8, 16, 32])
def test_int8_edge_lengths_and_group_sizes(hq):
    HK, CAP = 8, 2100
    lens = np.array([0, 1, 15, 17, 1024, 1025, 2100], np.int32)
    B = len(lens)
    k = synth.kv_fp16(13, 1, B, HK, CAP, D, synth.channel_scales(13, 4, HK, D))
    v = synth.kv_fp16(13, 2, B, HK, CAP, D, synth.channel_scales(13, 5, HK, D))
    q = synth.queries_fp16(13, B, hq, D)
    oc = oracle.build_cache(k, v, lens, CAP, 8, 8, codec="int8")
    tc = _cache(batch=B, num_kv_heads=HK, num_q_heads=hq, capacity=CAP)
    upload(tc, oc)
    got, ref = decode_both(tc, oc, q, lens, CAP)
    assert np.all(got[0] == 0)
    assert_attention_close(got[1:], ref[1:], "int8 edge lengths G=%d" % (hq // HK))


def test_int8_zero_and_extreme_rows():
    """All-zero vectors (scale 0), fp16 extremes and subnormals quantize exactly like the oracle."""
    B, HK, T = 1, 2, 48
    x = synth.kv_fp16(14, 1, B, HK, T, D)
    x[0, 0, 3] = 0.0
    x[0, 1, 5] = np.float16(65504.0) * np.sign(x[0, 1, 5]).astype(np.float16)
    x[0, 1, 6, :] = np.float16(6e-8)  # fp16 subnormal
    x[0, 0, 7, 0] = np.float16(-65504.0)
    tc = _cache(batch=B, num_kv_heads=HK, num_q_heads=HK, capacity=T)
    tc.append(_dev(x), _dev(x), _dev(np.zeros(B, np.int32)))
    assert tc.device_status() == 0
    check_rows(tc, x, 0, [T], "extreme K")
    assert tc.k_norms[0, 0, 3].item() == 0.0


def test_int8_long_context_full_size_sampled():
    """The long-context shape (B4, 32 q / 8 KV heads, contexts in [64K, 128K],
    256-token fp16 V window) on random int8 records: any byte is a valid code."""
    B, HQ, HK, CAP, W = 4, 32, 8, 131072, 256
    lens = synth.seq_lengths(5, B, 65536, 131072)
    rk = synth.rng(15, synth.STREAM_CODES_K)
    rv = synth.rng(15, synth.STREAM_CODES_V)
    k_words = rk.integers(0, 2 ** 32, size=(B, HK, CAP, 32), dtype=np.uint32)
    v_words = rv.integers(0, 2 ** 32, size=(B, HK, CAP, 32), dtype=np.uint32)
    # scales putting K and V at the magnitude of the packed workload (|k| ~ 12, |v| ~ 30)
    k_scales = synth.random_norms(15, synth.STREAM_NORMS_K, (B, HK, CAP), median=12.0 / (73.3 * 11.3))
    v_scales = synth.random_norms(15, synth.STREAM_NORMS_V, (B, HK, CAP), median=30.0 / (73.3 * 11.3))
    v_hot = synth.kv_fp16(15, synth.STREAM_V, B, HK, W, D, synth.channel_scales(15, synth.STREAM_SCALE_V, HK, D))
    oc = oracle.PackedCache(0, 0, D, 8, 8, k_words, k_scales, None, v_words, v_scales, W, v_hot, "int8")
    q = synth.queries_fp16(15, B, HQ, D)
    tc = _cache(batch=B, num_kv_heads=HK, num_q_heads=HQ, capacity=CAP, hot_window=W)
    upload(tc, oc)
    pairs = [(0, 0), (1, 13), (2, 22), (3, 31), (3, 4), (0, 27)]
    got, ref = decode_both(tc, oc, q, lens, CAP, pairs)
    assert_attention_close(got, ref, "int8 long-context decode (sampled heads)")
    assert tc.device_status() == 0


def test_int8_quantize_full_size_sampled():
    """The quantize throughput shape (B16 x 8192 tokens x 8 heads): two full
    (batch, head) rows and random token samples, bit-exact."""
    B, HK, T = 16, 8, 8192
    k = synth.kv_fp16(4, synth.STREAM_K, B, HK, T, D, synth.channel_scales(4, synth.STREAM_SCALE_K, HK, D))
    v = synth.kv_fp16(4, synth.STREAM_V, B, HK, T, D, synth.channel_scales(4, synth.STREAM_SCALE_V, HK, D))
    tc = _cache(batch=B, num_kv_heads=HK, num_q_heads=HK * 4, capacity=T)
    tc.append(_dev(k), _dev(v), _dev(np.zeros(B, np.int32)))
    assert tc.device_status() == 0
    rng = np.random.default_rng(8)
    for which, x in ((0, k), (1, v)):
        gw = (tc.k_cache if which == 0 else tc.v_cache).cpu().numpy().view(np.uint32)
        gs = (tc.k_norms if which == 0 else tc.v_norms).cpu().numpy()
        for b, h in [(0, 0), (B - 1, HK - 1)]:
            codes, s = oracle.int8_quantize_rows(x[b, h])
            np.testing.assert_array_equal(gs[b, h], s)
            np.testing.assert_array_equal(gw[b, h], oracle.int8_words(codes))
        for b, h in zip(rng.integers(0, B, 8), rng.integers(0, HK, 8)):
            t_idx = rng.choice(T, 512, replace=False)
            codes, s = oracle.int8_quantize_rows(x[b, h, t_idx])
            np.testing.assert_array_equal(gs[b, h, t_idx], s)
            np.testing.assert_array_equal(gw[b, h, t_idx], oracle.int8_words(codes))


def test_int8_paged_sparse_and_reproducible():
    """Paged int8 decode equals the contiguous one bit for bit; a vanishing
    sparse-V threshold changes nothing; repeated calls are identical."""
    B, HQ, HK, cap, bs = 3, 8, 2, 1024, 64
    lens = np.array([1000, 577, 70], np.int32)
    k = synth.kv_fp16(16, 1, B, HK, cap, D, synth.channel_scales(16, 4, HK, D))
    v = synth.kv_fp16(16, 2, B, HK, cap, D, synth.channel_scales(16, 5, HK, D))
    q = _dev(synth.queries_fp16(16, B, HQ, D))
    sl = _dev(lens)
    flat = _cache(batch=B, num_kv_heads=HK, num_q_heads=HQ, capacity=cap, hot_window=32)
    mb = cap // bs
    paged = _cache(batch=B, num_kv_heads=HK, num_q_heads=HQ, capacity=cap, hot_window=32, block_size=bs,
                   num_blocks=B * mb + 5)
    perm = np.random.default_rng(3).permutation(B * mb + 5)[:B * mb].astype(np.int32).reshape(B, mb)
    paged.block_table.copy_(_dev(perm))
    for tc in (flat, paged):
        tc.append(_dev(k), _dev(v), _dev(np.zeros(B, np.int32)), sl)
    assert flat.device_status() == 0 and paged.device_status() == 0
    # the paged layout and sparse V run the persistent kernel: the contiguous dense
    # decode they must equal bit for bit is taken through the same kernel
    N.tq_debug_set_decode_path(1)
    try:
        ref = flat.decode(q, sl, cap).cpu().numpy()
        np.testing.assert_array_equal(paged.decode(q, sl, cap).cpu().numpy(), ref)
        np.testing.assert_array_equal(flat.decode(q, sl, cap).cpu().numpy(), ref)
        flat.desc.sparse_v_threshold = 1e-30
        np.testing.assert_array_equal(flat.decode(q, sl, cap).cpu().numpy(), ref)
    finally:
        N.tq_debug_set_decode_path(0)
    oc = oracle.build_cache(k, v, lens, cap, 8, 8, hot_window=32, codec="int8")
    assert_attention_close(ref, oracle.decode_attention(oc, synth.queries_fp16(16, B, HQ, D), lens), "int8 paged")
