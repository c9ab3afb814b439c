"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Words and norms must be bit-exact except for codes whose oracle float32
rotated coordinate lies within 1e-6 of a threshold (counted, < 1e-5 of all
codes); attention outputs must agree within 2e-3 max-abs and 1e-3 relative-L2.
Decode is checked on the oracle's own packed cache uploaded to the GPU (so
that it is independent of quantize exceptions) and on the GPU's own cache.
"""
import numpy as np
import pytest

import oracle
from bit_kv_cache_10_gb300 import native as N
from bit_kv_cache_10_gb300 import synth

from helpers import assert_attention_close, assert_code_rate, compare_packed

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
    return TurboQuantKVCache(**kw)


def _dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.cuda()


def upload(tc, oc: oracle.PackedCache):
    """Copy an oracle cache state into the device buffers of a TurboQuantKVCache."""
    if oc.k_fp16 is not None:
        tc.k_cache.copy_(_dev(oc.k_fp16))
    else:
        tc.k_cache.copy_(_dev(oc.k_words.view(np.int32)))
        tc.k_norms.copy_(_dev(oc.k_norms))
    tc.v_cache.copy_(_dev(oc.v_words.view(np.int32)))
    tc.v_norms.copy_(_dev(oc.v_norms))
    if oc.v_hot is not None:
        tc.v_hot.copy_(_dev(oc.v_hot))
    torch.cuda.synchronize()


def quantize_reference(x16, seed, layer, bits, heads=None):
    """Oracle words, norms and rotated coordinates of x16 [B, H, T, d];
    ``heads`` gives the KV-head index of each H slice (default 0..H-1)."""
    b_, h_, t_, _ = x16.shape
    cb = oracle.codebook(D, bits)
    words = np.empty((b_, h_, t_, D * bits // 32), np.uint32)
    norms = np.empty((b_, h_, t_), np.float32)
    ys = np.empty((b_, h_, t_, D))
    for h in range(h_):
        rot = oracle.rotation(seed, layer, heads[h] if heads is not None else h, D)
        for b in range(b_):
            c, n, y = oracle.quantize_rows(x16[b, h], rot, cb)
            words[b, h] = oracle.pack(c, bits)
            norms[b, h] = n
            ys[b, h] = y
    return words, norms, ys


def check_quantized(tc, x16, which, bits, lengths, seed=0, layer=0, what=""):
    """GPU words/norms of positions [0, L_b) against the oracle."""
    ref_w, ref_n, ys = quantize_reference(x16, seed, layer, bits)
    gw = (tc.k_cache if which == 0 else tc.v_cache).cpu().numpy().view(np.uint32)
    gn = (tc.k_norms if which == 0 else tc.v_norms).cpu().numpy()
    thr = oracle.codebook(D, bits).thresholds32
    total_mism, total_codes = 0, 0
    for b in range(x16.shape[0]):
        L = int(lengths[b])
        np.testing.assert_array_equal(gn[b, :, :L], ref_n[b, :, :L], err_msg=what + " norms")
        m, c = compare_packed(gw[b, :, :L].reshape(-1, gw.shape[-1]), ref_w[b, :, :L].reshape(-1, ref_w.shape[-1]),
                              ys[b, :, :L].reshape(-1, D), bits, thr, what, check_rate=False)
        total_mism, total_codes = total_mism + m, total_codes + c
    assert_code_rate(total_mism, total_codes, what)
    return total_mism


def decode_both(tc, oc, q16, lengths, max_len, pairs=None):
    ql = _dev(q16)
    sl = _dev(np.asarray(lengths, np.int32))
    got = tc.decode(ql, sl, max_len).cpu().numpy()
    ref = oracle.decode_attention(oc, q16, lengths, pairs)
    if pairs is not None:
        idx = tuple(np.array(pairs).T)
        return got[idx], ref[idx]
    return got, ref


def end_to_end(tc, oc, q16, lengths, max_len, flips, what):
    """Decode parity on the oracle's own cache (the decode claim), and on the
    GPU-quantized cache when it equals the oracle's bit for bit.  With counted
    threshold-near code flips the GPU cache is a different (equally valid)
    quantization, and a flipped code of a token that dominates a peaked
    softmax can move an output by more than the attention tolerance; the two
    claims are then checked separately."""
    ql = _dev(q16)
    sl = _dev(np.asarray(lengths, np.int32))
    own = tc.decode(ql, sl, max_len).cpu().numpy()
    ref = oracle.decode_attention(oc, q16, lengths)
    if flips == 0:
        assert_attention_close(own, ref, what + " decode on the GPU-quantized cache")
    upload(tc, oc)
    got = tc.decode(ql, sl, max_len).cpu().numpy()
    assert_attention_close(got, ref, what + " decode on the oracle cache")


# --------------------------------------------------------------------------
# workload 1: tiny, K4/V4, 1 head, 512 tokens, N(0,1), seed 0
# --------------------------------------------------------------------------

def test_tiny_k4v4():
    L = 512
    k = synth.kv_fp16(0, synth.STREAM_K, 1, 1, L, D)
    v = synth.kv_fp16(0, synth.STREAM_V, 1, 1, L, D)
    q = synth.queries_fp16(0, 1, 1, D)
    tc = _cache(batch=1, num_kv_heads=1, num_q_heads=1, capacity=L, bits=(4, 4))
    tc.append(_dev(k), _dev(v), _dev(np.zeros(1, np.int32)))
    assert tc.device_status() == 0
    flips = check_quantized(tc, k, 0, 4, [L], what="tiny K") + check_quantized(tc, v, 1, 4, [L], what="tiny V")
    oc = oracle.build_cache(k, v, [L], L, 4, 4)
    end_to_end(tc, oc, q, [L], L, flips, "tiny")


# --------------------------------------------------------------------------
# workload 2: Llama-3-8B-like layer at 3.5 bits (K3/V4), GQA 4, context 4096
# --------------------------------------------------------------------------

def test_llama_like_3p5_bit():
    B, HQ, HK, L = 1, 32, 8, 4096
    k = synth.kv_fp16(2, synth.STREAM_K, B, HK, L, D, synth.channel_scales(2, synth.STREAM_SCALE_K, HK, D))
    v = synth.kv_fp16(2, synth.STREAM_V, B, HK, L, D, synth.channel_scales(2, synth.STREAM_SCALE_V, HK, D))
    q = synth.queries_fp16(2, B, HQ, D)
    tc = _cache(batch=B, num_kv_heads=HK, num_q_heads=HQ, capacity=L, bits=3.5)
    tc.append(_dev(k), _dev(v), _dev(np.zeros(B, np.int32)))
    flips = check_quantized(tc, k, 0, 3, [L], what="3.5-bit K") + check_quantized(tc, v, 1, 4, [L], what="3.5-bit V")
    oc = oracle.build_cache(k, v, [L], L, 3, 4)
    end_to_end(tc, oc, q, [L], L, flips, "3.5-bit")


# --------------------------------------------------------------------------
# workload 3: asym, fp16 K + 4-bit V, batch 8, GQA 4, context 16384
# --------------------------------------------------------------------------

def test_asym_fp16k_v4_full_size():
    B, HQ, HK, L = 8, 32, 8, 16384
    k = synth.kv_fp16(3, synth.STREAM_K, B, HK, L, D, synth.channel_scales(3, synth.STREAM_SCALE_K, HK, D))
    v = synth.kv_fp16(3, synth.STREAM_V, B, HK, L, D, synth.channel_scales(3, synth.STREAM_SCALE_V, HK, D))
    q = synth.queries_fp16(3, B, HQ, D)
    tc = _cache(batch=B, num_kv_heads=HK, num_q_heads=HQ, capacity=L, bits=(0, 4), k_fp16=True)
    tc.append(_dev(k), _dev(v), _dev(np.zeros(B, np.int32)))
    np.testing.assert_array_equal(tc.k_cache.cpu().numpy(), k)  # fp16 K stored verbatim
    # V parity on a sample of rows (the whole set is checked on smaller workloads)
    sub = v[[0, 5]][:, [0, 7]]
    ref_w, ref_n, ys = quantize_reference(sub, 0, 0, 4, heads=[0, 7])
    gw = tc.v_cache.cpu().numpy().view(np.uint32)[[0, 5]][:, [0, 7]]
    gn = tc.v_norms.cpu().numpy()[[0, 5]][:, [0, 7]]
    np.testing.assert_array_equal(gn, ref_n)
    compare_packed(gw.reshape(-1, 16), ref_w.reshape(-1, 16), ys.reshape(-1, D), 4,
                   oracle.codebook(D, 4).thresholds32, "asym V")
    pairs = [(0, 0), (0, 31), (3, 9), (5, 17), (7, 30), (2, 4)]
    oc = _asym_reference_cache(k, v, L, {(b, hq // 4) for b, hq in pairs})
    got, ref = decode_both(tc, oc, q, [L] * B, L, pairs)
    assert_attention_close(got, ref, "asym decode (sampled heads)")


def _asym_reference_cache(k, v, L, needed):
    """Oracle cache with fp16 K and the oracle's own 4-bit V for the (b, h) rows in ``needed``."""
    B, HK = k.shape[:2]
    cb = oracle.codebook(D, 4)
    words = np.zeros((B, HK, L, 16), np.uint32)
    norms = np.zeros((B, HK, L), np.float32)
    for b, h in needed:
        c, n, _ = oracle.quantize_rows(v[b, h], oracle.rotation(0, 0, h, D), cb)
        words[b, h] = oracle.pack(c, 4)
        norms[b, h] = n
    return oracle.PackedCache(0, 0, D, 16, 4, None, None, k, words, norms)


# --------------------------------------------------------------------------
# workload 4: quantize/append throughput shape, bits 3, 4 and 3.5
# --------------------------------------------------------------------------

@pytest.mark.parametrize("bits", [(3, 3), (4, 4), (3, 4)])
def test_quantize_full_size(bits):
    B, HK, T = 16, 8, 8192
    k = synth.kv_fp16(4, synth.STREAM_K, B, HK, T, D, synth.channel_scales(4, synth.STREAM_SCALE_K, HK, D))
    v = synth.kv_fp16(4, synth.STREAM_V, B, HK, T, D, synth.channel_scales(4, synth.STREAM_SCALE_V, HK, D))
    tc = _cache(batch=B, num_kv_heads=HK, num_q_heads=HK * 4, capacity=T, bits=bits)
    tc.append(_dev(k), _dev(v), _dev(np.zeros(B, np.int32)))
    assert tc.device_status() == 0
    kb, vb = bits
    rng = np.random.default_rng(sum(bits))
    n_mism, n_codes = 0, 0
    for which, x, nb in ((0, k, kb), (1, v, vb)):
        gw = (tc.k_cache if which == 0 else tc.v_cache).cpu().numpy().view(np.uint32)
        gn = (tc.k_norms if which == 0 else tc.v_norms).cpu().numpy()
        thr = oracle.codebook(D, nb).thresholds32
        # two full (batch, head) rows and 8 x 512 random token vectors
        sel = [(0, 0), (B - 1, HK - 1)] + [(int(b), int(h)) for b, h in zip(rng.integers(0, B, 8), rng.integers(0, HK, 8))]
        for b, h in sel[:2]:
            ref_w, ref_n, ys = quantize_reference(x[b:b + 1, h:h + 1], 0, 0, nb, heads=[h])
            np.testing.assert_array_equal(gn[b, h], ref_n[0, 0])
            m, c = compare_packed(gw[b, h], ref_w[0, 0], ys[0, 0], nb, thr, "full row", check_rate=False)
            n_mism, n_codes = n_mism + m, n_codes + c
        for b, h in sel[2:]:
            t_idx = rng.choice(T, 512, replace=False)
            c_, n, y = oracle.quantize_rows(x[b, h, t_idx], oracle.rotation(0, 0, h, D), oracle.codebook(D, nb))
            np.testing.assert_array_equal(gn[b, h, t_idx], n)
            m, c = compare_packed(gw[b, h, t_idx], oracle.pack(c_, nb), y, nb, thr, "sampled rows", check_rate=False)
            n_mism, n_codes = n_mism + m, n_codes + c
    assert_code_rate(n_mism, n_codes, "quantize %s" % (bits,))


# --------------------------------------------------------------------------
# workload 5: long context, K3 + V4 cold + 256-token fp16 V window, ragged
# --------------------------------------------------------------------------

def test_long_context_full_size_sampled():
    B, HQ, HK, CAP, W = 4, 32, 8, 131072, 256
    lens = synth.seq_lengths(5, B, 65536, 131072)
    rk = synth.rng(5, synth.STREAM_CODES_K)
    rv = synth.rng(5, synth.STREAM_CODES_V)
    # any bit pattern is a valid packed record: random words stand in for a full cache
    k_words = rk.integers(0, 2 ** 32, size=(B, HK, CAP, 12), dtype=np.uint32)
    v_words = rv.integers(0, 2 ** 32, size=(B, HK, CAP, 16), dtype=np.uint32)
    k_norms = synth.random_norms(5, synth.STREAM_NORMS_K, (B, HK, CAP), median=12.0)
    v_norms = synth.random_norms(5, synth.STREAM_NORMS_V, (B, HK, CAP), median=30.0)
    v_hot = synth.kv_fp16(5, synth.STREAM_V, B, HK, W, D, synth.channel_scales(5, synth.STREAM_SCALE_V, HK, D))
    oc = oracle.PackedCache(0, 0, D, 3, 4, k_words, k_norms, None, v_words, v_norms, W, v_hot)
    tc = _cache(batch=B, num_kv_heads=HK, num_q_heads=HQ, capacity=CAP, bits=3.5, hot_window=W)
    upload(tc, oc)
    # every query head of the shortest sequence (all 8 KV heads, 32 outputs), and
    # heads of the other sequences; with the plain queries and with queries scaled
    # by 2.5, whose softmax concentrates on a few tokens
    b_all = int(np.argmin(lens))
    pairs = [(b_all, hq) for hq in range(HQ)] + [(b, hq) for b, hq in ((0, 27), (1, 13), (2, 22), (3, 31), (3, 4))
                                                 if b != b_all]
    for scale in (1.0, 2.5):
        q = (synth.queries_fp16(5, B, HQ, D) * np.float16(scale)).astype(np.float16)
        got, ref = decode_both(tc, oc, q, lens, CAP, pairs)
        assert_attention_close(got, ref, "long-context decode, query scale %g" % scale)
    assert tc.device_status() == 0


def test_long_context_ragged_append_then_decode():
    """Reduced long-context workload built through the append path: a ragged
    prefill, then token-by-token appends that push V tokens out of the hot ring."""
    B, HQ, HK, CAP, W, STEPS = 4, 32, 8, 6144, 256, 12
    lens = synth.seq_lengths(6, B, 2048, 6000)
    k = synth.kv_fp16(6, synth.STREAM_K, B, HK, int(lens.max()), D, synth.channel_scales(6, 4, HK, D))
    v = synth.kv_fp16(6, synth.STREAM_V, B, HK, int(lens.max()), D, synth.channel_scales(6, 5, HK, D))
    q = synth.queries_fp16(6, B, HQ, D)
    tc = _cache(batch=B, num_kv_heads=HK, num_q_heads=HQ, capacity=CAP, bits=3.5, hot_window=W)
    kd, vd = _dev(k), _dev(v)
    pre = lens - STEPS
    tc.append(kd, vd, _dev(np.zeros(B, np.int32)), _dev(pre.astype(np.int32)))
    for s in range(STEPS):
        start = (pre + s).astype(np.int32)
        idx = torch.from_numpy(start.astype(np.int64)).cuda()
        kn = torch.stack([kd[b, :, idx[b]] for b in range(B)])[:, :, None].contiguous()
        vn = torch.stack([vd[b, :, idx[b]] for b in range(B)])[:, :, None].contiguous()
        tc.append(kn, vn, _dev(start))
    assert tc.device_status() == 0
    oc = oracle.build_cache(k, v, lens, CAP, 3, 4, hot_window=W)
    flips = check_quantized(tc, k, 0, 3, lens, what="ragged K")
    # cold V region and the ring
    ce = lens - np.minimum(W, lens)
    flips += check_quantized(tc, v, 1, 4, ce, what="ragged cold V")
    np.testing.assert_array_equal(tc.v_hot.cpu().numpy(), oc.v_hot)
    end_to_end(tc, oc, q, lens, CAP, flips, "ragged")


# --------------------------------------------------------------------------
# edge cases
# --------------------------------------------------------------------------

@pytest.mark.parametrize("kb,vb,hq", [(2, 2, 8), (4, 3, 16), (3, 4, 8), (2, 4, 32)])
def test_edge_lengths_and_group_sizes(kb, vb, hq):
    HK, CAP = 8, 2100
    lens = np.array([0, 1, 31, 33, 1024, 1025, 2100], np.int32)
    B = len(lens)
    k = synth.kv_fp16(7, 1, B, HK, CAP, D, synth.channel_scales(7, 4, HK, D))
    v = synth.kv_fp16(7, 2, B, HK, CAP, D, synth.channel_scales(7, 5, HK, D))
    q = synth.queries_fp16(7, B, hq, D)
    oc = oracle.build_cache(k, v, lens, CAP, kb, vb)
    tc = _cache(batch=B, num_kv_heads=HK, num_q_heads=hq, capacity=CAP, bits=(kb, vb))
    upload(tc, oc)
    got, ref = decode_both(tc, oc, q, lens, CAP)
    assert np.all(got[0] == 0)
    assert_attention_close(got[1:], ref[1:], "edge lengths kb=%d vb=%d G=%d" % (kb, vb, hq // HK))


@pytest.mark.parametrize("hot", [8, 64])
def test_hot_window_longer_and_shorter_than_sequences(hot):
    HK, HQ, CAP = 2, 8, 300
    lens = np.array([3, 8, 9, 64, 65, 300], np.int32)
    B = len(lens)
    k = synth.kv_fp16(8, 1, B, HK, CAP, D, synth.channel_scales(8, 4, HK, D))
    v = synth.kv_fp16(8, 2, B, HK, CAP, D, synth.channel_scales(8, 5, HK, D))
    q = synth.queries_fp16(8, B, HQ, D)
    tc = _cache(batch=B, num_kv_heads=HK, num_q_heads=HQ, capacity=CAP, bits=3.5, hot_window=hot)
    tc.append(_dev(k), _dev(v), _dev(np.zeros(B, np.int32)), _dev(lens))
    oc = oracle.build_cache(k, v, lens, CAP, 3, 4, hot_window=hot)
    np.testing.assert_array_equal(tc.v_hot.cpu().numpy(), oc.v_hot)
    got, ref = decode_both(tc, oc, q, lens, CAP)
    assert_attention_close(got, ref, "hot window %d" % hot)
    for b in (0, 4, 5):
        L = int(lens[b])
        gv = tc.dequantize(1, b, L, 0, L).cpu().numpy()
        for h in range(HK):
            _, ref_v = oracle.dequantized_kv(oc, b, h, L)
            scale = np.maximum(np.linalg.norm(ref_v, axis=1, keepdims=True), 1e-30)
            assert np.all(np.abs(gv[h] - ref_v) <= 1e-5 * scale)


def test_strided_inputs_and_partial_tiles():
    # K/V given as a [B, T, H, d] buffer viewed as [B, H, T, d]; 45 tokens appended at offset 19
    B, HK, T, CAP = 2, 4, 45, 100
    kt = synth.kv_fp16(9, 1, B, T, HK, D)  # drawn [B, T, H, d]
    vt = synth.kv_fp16(9, 2, B, T, HK, D)
    kd = _dev(kt).permute(0, 2, 1, 3)
    vd = _dev(vt).permute(0, 2, 1, 3)
    tc = _cache(batch=B, num_kv_heads=HK, num_q_heads=HK, capacity=CAP, bits=(3, 2))
    tc.append(kd, vd, _dev(np.array([19, 0], np.int32)))
    assert tc.device_status() == 0
    k = np.ascontiguousarray(kt.transpose(0, 2, 1, 3))
    v = np.ascontiguousarray(vt.transpose(0, 2, 1, 3))
    gw = tc.k_cache.cpu().numpy().view(np.uint32)
    gn = tc.k_norms.cpu().numpy()
    ref_w, ref_n, ys = quantize_reference(k, 0, 0, 3)
    np.testing.assert_array_equal(gn[0, :, 19:64], ref_n[0])
    np.testing.assert_array_equal(gn[1, :, :45], ref_n[1])
    assert np.all(gn[0, :, :19] == 0) and np.all(gn[0, :, 64:] == 0) and np.all(gn[1, :, 45:] == 0)
    compare_packed(gw[0, :, 19:64].reshape(-1, 12), ref_w[0].reshape(-1, 12), ys[0].reshape(-1, D), 3,
                   oracle.codebook(D, 3).thresholds32, "strided K")
    vw, vn, vy = quantize_reference(v, 0, 0, 2)
    np.testing.assert_array_equal(tc.v_norms.cpu().numpy()[1, :, :45], vn[1])
    compare_packed(tc.v_cache.cpu().numpy().view(np.uint32)[1, :, :45].reshape(-1, 8), vw[1].reshape(-1, 8),
                   vy[1].reshape(-1, D), 2, oracle.codebook(D, 2).thresholds32, "strided V")


def test_device_status_on_bad_positions_and_lengths():
    B, HK, CAP = 3, 2, 64
    k = synth.kv_fp16(10, 1, B, HK, 40, D)
    v = synth.kv_fp16(10, 2, B, HK, 40, D)
    tc = _cache(batch=B, num_kv_heads=HK, num_q_heads=HK, capacity=CAP, bits=(4, 4))
    tc.append(_dev(k), _dev(v), _dev(np.array([0, 30, -1], np.int32)))  # 30+40 > 64, -1 < 0
    assert tc.device_status() == N.TQ_DEV_ERR_APPEND_RANGE
    gn = tc.k_norms.cpu().numpy()
    assert np.all(gn[0, :, :40] > 0) and np.all(gn[1] == 0) and np.all(gn[2] == 0)
    tc.status.zero_()
    q = synth.queries_fp16(10, B, HK, D)
    out = tc.decode(_dev(q), _dev(np.array([40, 65, -3], np.int32)), CAP).cpu().numpy()
    assert tc.device_status() == N.TQ_DEV_ERR_SEQ_LEN
    assert np.all(out[1:] == 0) and np.all(np.isfinite(out[0]))
    tc.status.zero_()
    tc.decode(_dev(q), _dev(np.array([40, 50, 10], np.int32)), 45)  # 50 > max_seq_len
    assert tc.device_status() == N.TQ_DEV_ERR_SEQ_LEN


def test_dequantize_matches_oracle():
    B, HK, L = 2, 3, 300
    k = synth.kv_fp16(11, 1, B, HK, L, D, synth.channel_scales(11, 4, HK, D))
    v = synth.kv_fp16(11, 2, B, HK, L, D, synth.channel_scales(11, 5, HK, D))
    for kfp16 in (False, True):
        oc = oracle.build_cache(k, v, [L, L], L, 16 if kfp16 else 3, 4, k_fp16=kfp16)
        tc = _cache(batch=B, num_kv_heads=HK, num_q_heads=HK, capacity=L, bits=(0, 4) if kfp16 else (3, 4),
                    k_fp16=kfp16)
        upload(tc, oc)
        for which in (0, 1):
            got = tc.dequantize(which, 1, L, 7, 250).cpu().numpy()
            for h in range(HK):
                kr, vr = oracle.dequantized_kv(oc, 1, h, L)
                ref = (kr if which == 0 else vr)[7:257]
                scale = np.maximum(np.linalg.norm(ref, axis=1, keepdims=True), 1e-30)
                assert np.all(np.abs(got[h] - ref) <= 1e-5 * scale), (kfp16, which, h)


@pytest.mark.parametrize("bits", [3.5, "int8"])
def test_append_chunks_within_the_hot_window(bits):
    """Appends of at most W tokens evict the ring slots they take inside the same
    launch; rows whose slot held a position (pos - W >= 0) turn cold, the others
    do not.  Chunks of 8 and 40 (= W) tokens on sequences shorter and longer
    than W."""
    HK, HQ, CAP, W = 2, 8, 400, 40
    pre = np.array([10, 39, 100, 0], np.int32)
    B = len(pre)
    k = synth.kv_fp16(41, 1, B, HK, CAP, D, synth.channel_scales(41, 4, HK, D))
    v = synth.kv_fp16(41, 2, B, HK, CAP, D, synth.channel_scales(41, 5, HK, D))
    tc = _cache(batch=B, num_kv_heads=HK, num_q_heads=HQ, capacity=CAP, bits=bits, hot_window=W)
    kd, vd = _dev(k), _dev(v)
    tc.append(kd, vd, _dev(np.zeros(B, np.int32)), _dev(pre))
    lens = pre.copy()
    for n in (8, 40, 1, 8):
        idx = torch.from_numpy(lens.astype(np.int64)).cuda()
        kn = torch.stack([kd[b, :, idx[b]:idx[b] + n] for b in range(B)]).contiguous()
        vn = torch.stack([vd[b, :, idx[b]:idx[b] + n] for b in range(B)]).contiguous()
        tc.append(kn, vn, _dev(lens))
        lens = lens + n
    assert tc.device_status() == 0
    if bits == "int8":
        oc = oracle.build_cache(k, v, lens, CAP, 8, 8, hot_window=W, codec="int8")
        gw = tc.v_cache.cpu().numpy().view(np.uint32)
        gs = tc.v_norms.cpu().numpy()
        for b in range(B):
            ce = int(lens[b]) - min(W, int(lens[b]))
            np.testing.assert_array_equal(gw[b, :, :ce], oc.v_words[b, :, :ce])
            np.testing.assert_array_equal(gs[b, :, :ce], oc.v_norms[b, :, :ce])
    else:
        oc = oracle.build_cache(k, v, lens, CAP, 3, 4, hot_window=W)
        check_quantized(tc, v, 1, 4, lens - np.minimum(W, lens), what="chunked cold V")
    np.testing.assert_array_equal(tc.v_hot.cpu().numpy(), oc.v_hot)
    q = synth.queries_fp16(41, B, HQ, D)
    upload(tc, oc)
    got, ref = decode_both(tc, oc, q, lens, CAP)
    assert_attention_close(got, ref, "chunked appends")


@pytest.mark.parametrize("bits", [(2, 3), 3.5, (4, 4), "int8"])
def test_small_and_bulk_appends_store_the_same_words(bits):
    """Appends of at most 16 tokens use the one-warp-per-vector kernel, longer
    ones the four-lanes-per-vector kernel; both must store identical words and
    norms (same arithmetic, stage for stage)."""
    B, HK, T = 3, 4, 48
    k = synth.kv_fp16(51, 1, B, HK, T, D, synth.channel_scales(51, 4, HK, D))
    v = synth.kv_fp16(51, 2, B, HK, T, D, synth.channel_scales(51, 5, HK, D))
    k[0, 1, 5] = 0.0  # a zero vector
    bulk = _cache(batch=B, num_kv_heads=HK, num_q_heads=HK, capacity=T, bits=bits)
    small = _cache(batch=B, num_kv_heads=HK, num_q_heads=HK, capacity=T, bits=bits)
    bulk.append(_dev(k), _dev(v), _dev(np.zeros(B, np.int32)))
    for c in range(0, T, 16):
        small.append(_dev(k[:, :, c:c + 16]), _dev(v[:, :, c:c + 16]), _dev(np.full(B, c, np.int32)))
    assert bulk.device_status() == 0 and small.device_status() == 0
    for name in ("k_cache", "k_norms", "v_cache", "v_norms"):
        np.testing.assert_array_equal(getattr(small, name).cpu().numpy(), getattr(bulk, name).cpu().numpy(),
                                      err_msg=name)


@pytest.mark.parametrize("hk", [16, 17, 24])
def test_many_kv_heads_rotation_signs(hk):
    """The bulk append kernel tabulates the rotation signs of up to 16 KV heads
    once per CTA and computes them per job beyond that; both must give the
    oracle's words and norms (seed 3, layer 5), and the same words as the
    small-append kernel, which computes the signs per vector."""
    B, T = 2, 40
    k = synth.kv_fp16(71, 1, B, hk, T, D, synth.channel_scales(71, 4, hk, D))
    v = synth.kv_fp16(71, 2, B, hk, T, D, synth.channel_scales(71, 5, hk, D))
    kw = dict(batch=B, num_kv_heads=hk, num_q_heads=hk, capacity=T, bits=(3, 4), seed=3, layer=5)
    bulk, small = _cache(**kw), _cache(**kw)
    bulk.append(_dev(k), _dev(v), _dev(np.zeros(B, np.int32)))
    for c in range(0, T, 16):
        small.append(_dev(k[:, :, c:c + 16]), _dev(v[:, :, c:c + 16]), _dev(np.full(B, c, np.int32)))
    assert bulk.device_status() == 0 and small.device_status() == 0
    for name in ("k_cache", "k_norms", "v_cache", "v_norms"):
        np.testing.assert_array_equal(getattr(small, name).cpu().numpy(), getattr(bulk, name).cpu().numpy(),
                                      err_msg=name)
    lens = np.full(B, T)
    check_quantized(bulk, k, 0, 3, lens, seed=3, layer=5, what="K, %d KV heads" % hk)
    check_quantized(bulk, v, 1, 4, lens, seed=3, layer=5, what="V, %d KV heads" % hk)


def test_largest_batch_of_ragged_sequences():
    """The largest batch one decode call takes (512 sequences: the per-sequence tile
    prefix is held in shared memory), lengths 0..200 including empty sequences,
    G = 4, K4/V4 with a 16-token hot window."""
    B, HK, HQ, CAP, W = 512, 1, 4, 200, 16
    rng = np.random.default_rng(61)
    lens = rng.integers(0, CAP + 1, size=B).astype(np.int32)
    lens[:3] = [0, 1, CAP]
    k = synth.kv_fp16(61, 1, B, HK, CAP, D)
    v = synth.kv_fp16(61, 2, B, HK, CAP, D)
    q = synth.queries_fp16(61, B, HQ, D)
    oc = oracle.build_cache(k, v, lens, CAP, 4, 4, hot_window=W)
    tc = _cache(batch=B, num_kv_heads=HK, num_q_heads=HQ, capacity=CAP, bits=(4, 4), hot_window=W)
    upload(tc, oc)
    got, ref = decode_both(tc, oc, q, lens, CAP)
    empty = lens == 0
    assert np.all(got[empty] == 0)
    assert_attention_close(got[~empty], ref[~empty], "512 ragged sequences")
    assert tc.device_status() == 0
    # one sequence more is refused before any launch
    big = _cache(batch=B + 1, num_kv_heads=HK, num_q_heads=HQ, capacity=16, bits=(4, 4))
    with pytest.raises(N.TQError) as e:
        big.decode(_dev(np.zeros((B + 1, HQ, D), np.float16)), _dev(np.zeros(B + 1, np.int32)), 16)
    assert e.value.status == N.TQ_ERR_UNSUPPORTED
