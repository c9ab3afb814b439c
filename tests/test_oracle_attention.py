"""Pins of the oracle's decode attention and bit-budget helpers (CPU only)."""
import math

import numpy as np
import pytest
from scipy import special

import oracle
from bit_kv_cache_10_gb300 import synth


def _cache(b, hk, length, kb, vb, k_fp16=False, hot=0, seed=0, scaled=True, cap=None):
    d = 128
    sk = synth.channel_scales(seed, 4, hk, d) if scaled else None
    sv = synth.channel_scales(seed, 5, hk, d) if scaled else None
    k = synth.kv_fp16(seed, 1, b, hk, length, d, sk)
    v = synth.kv_fp16(seed, 2, b, hk, length, d, sv)
    lens = np.full(b, length)
    c = oracle.build_cache(k, v, lens, cap or length, kb, vb, seed=seed, k_fp16=k_fp16, hot_window=hot)
    return c, k, v, lens


def test_single_token_returns_its_value():
    c, _, _, lens = _cache(1, 1, 1, 4, 4)
    q = synth.queries_fp16(0, 1, 1, 128)
    _, v = oracle.dequantized_kv(c, 0, 0, 1)
    np.testing.assert_allclose(oracle.decode_attention(c, q, lens)[0, 0], v[0], rtol=1e-14)


def test_zero_query_is_mean_of_values():
    c, _, _, lens = _cache(1, 1, 37, 3, 4)
    q = np.zeros((1, 1, 128), np.float16)
    _, v = oracle.dequantized_kv(c, 0, 0, 37)
    np.testing.assert_allclose(oracle.decode_attention(c, q, lens)[0, 0], v.mean(axis=0), rtol=1e-12, atol=1e-13)


def test_identical_keys_give_uniform_weights():
    d = 128
    k = np.tile(synth.kv_fp16(4, 1, 1, 1, 1, d), (1, 1, 20, 1))
    v = synth.kv_fp16(4, 2, 1, 1, 20, d)
    c = oracle.build_cache(k, v, [20], 20, 4, 4)
    q = synth.queries_fp16(4, 1, 1, d)
    _, vh = oracle.dequantized_kv(c, 0, 0, 20)
    np.testing.assert_allclose(oracle.decode_attention(c, q, [20])[0, 0], vh.mean(axis=0), rtol=1e-12, atol=1e-13)


def test_fp16_keys_reduce_to_textbook_softmax_attention():
    c, k, _, lens = _cache(1, 2, 50, 16, 4, k_fp16=True)
    q = synth.queries_fp16(0, 1, 8, 128)
    out = oracle.decode_attention(c, q, lens)
    for hq in range(8):
        h = hq // 4
        _, vh = oracle.dequantized_kv(c, 0, h, 50)
        kf = k[0, h].astype(np.float64)
        p = special.softmax(kf @ q[0, hq].astype(np.float64) / math.sqrt(128))
        np.testing.assert_allclose(out[0, hq], p @ vh, rtol=1e-11, atol=1e-12)


def test_gqa_groups_are_contiguous():
    c, _, _, lens = _cache(1, 2, 40, 3, 4)
    q = np.tile(synth.queries_fp16(1, 1, 1, 128), (1, 4, 1))
    out = oracle.decode_attention(c, q, lens)
    np.testing.assert_array_equal(out[0, 0], out[0, 1])
    np.testing.assert_array_equal(out[0, 2], out[0, 3])
    assert np.abs(out[0, 1] - out[0, 2]).max() > 1e-3


@pytest.mark.parametrize("hot", [0, 16])
def test_rotated_domain_identity(hot):
    c, _, _, lens = _cache(2, 2, 100, 3, 4, hot=hot)
    q = synth.queries_fp16(0, 2, 8, 128)
    dense = oracle.decode_attention(c, q, lens)
    for b, hq in [(0, 0), (1, 5), (1, 7)]:
        np.testing.assert_allclose(oracle.decode_attention_rotated(c, q, lens, b, hq), dense[b, hq],
                                   rtol=1e-11, atol=1e-12)


def test_hot_window_reads_raw_fp16_values():
    d, length, hot = 128, 30, 8
    c, k, v, lens = _cache(1, 1, length, 3, 4, hot=hot)
    q = synth.queries_fp16(2, 1, 1, d)
    kd, vd = oracle.dequantized_kv(c, 0, 0, length)
    np.testing.assert_array_equal(vd[length - hot:], v[0, 0, length - hot:].astype(np.float64))
    full = oracle.build_cache(k, v, lens, length, 3, 4)
    _, v_cold = oracle.dequantized_kv(full, 0, 0, length)
    np.testing.assert_array_equal(vd[:length - hot], v_cold[:length - hot])
    p = special.softmax(kd @ q[0, 0].astype(np.float64) / math.sqrt(d))
    np.testing.assert_allclose(oracle.decode_attention(c, q, lens)[0, 0], p @ vd, rtol=1e-12, atol=1e-12)
    # ring slots: position p sits in slot p mod W
    for p_ in range(length - hot, length):
        np.testing.assert_array_equal(c.v_hot[0, 0, p_ % hot], v[0, 0, p_])


def test_hot_window_longer_than_sequence():
    c, _, v, lens = _cache(1, 1, 5, 3, 4, hot=8, cap=16)
    _, vd = oracle.dequantized_kv(c, 0, 0, 5)
    np.testing.assert_array_equal(vd, v[0, 0, :5].astype(np.float64))


def test_empty_sequence_gives_zero_output():
    c, _, _, _ = _cache(1, 1, 4, 3, 4)
    q = synth.queries_fp16(0, 1, 1, 128)
    assert np.all(oracle.decode_attention(c, q, [0])[0, 0] == 0)


def test_split_bits():
    assert oracle.split_bits(3.5) == (3, 4)
    assert oracle.split_bits(4) == (4, 4)
    assert oracle.split_bits(2.5) == (2, 3)
    assert oracle.split_bits(4.2) == (4, 5)


def test_turboquant_enabled_truth_table():
    assert oracle.turboquant_enabled(None) is False
    assert oracle.turboquant_enabled(None, "turboquant") is False
    assert oracle.turboquant_enabled(4, "turboquant") is True
    assert oracle.turboquant_enabled(3.5) is True
    assert oracle.turboquant_enabled(4) is False
    assert oracle.turboquant_enabled(4.0000001) is False
    assert oracle.turboquant_enabled(4.2) is True
    assert oracle.turboquant_enabled(2, "uniform") is False


# --- sparse-V bound ------------------------------------------------------------

def _dense_weights(q, k):
    s = k @ q / np.sqrt(q.shape[-1])
    p = np.exp(s - s.max())
    return p / p.sum()


def test_sparse_v_bound_is_zero_when_off():
    g = np.random.default_rng(3)
    q, k, v = g.standard_normal(8), g.standard_normal((20, 8)), g.standard_normal((20, 8))
    assert np.all(oracle.sparse_v_bound(q, k, v, 0.0) == 0.0)
    assert np.all(oracle.sparse_v_bound(q, k[:0], v[:0], 0.5) == 0.0)


def test_sparse_v_bound_with_every_token_skippable_is_the_weighted_abs_sum():
    g = np.random.default_rng(4)
    q, k, v = g.standard_normal(8), g.standard_normal((15, 8)), g.standard_normal((15, 8))
    p = _dense_weights(q, k)
    expect = sum(p[j] * np.abs(v[j]) for j in range(15))
    np.testing.assert_allclose(oracle.sparse_v_bound(q, k, v, 1.0 + 1e-9), expect, rtol=1e-12)


def test_sparse_v_bound_covers_every_skipped_subset_by_brute_force():
    # every subset of the tokens below the threshold, its V rows removed with the
    # softmax mass kept, moves each coordinate by no more than the bound
    import itertools
    g = np.random.default_rng(5)
    d, n = 4, 7
    q, k, v = 2.0 * g.standard_normal(d), g.standard_normal((n, d)), g.standard_normal((n, d))
    p = _dense_weights(q, k)
    tau = float(np.sort(p)[4])  # four tokens lie below it
    below = [j for j in range(n) if p[j] < tau]
    assert len(below) == 4
    bound = oracle.sparse_v_bound(q, k, v, tau)
    dense = p @ v
    worst = np.zeros(d)
    for r in range(len(below) + 1):
        for sub in itertools.combinations(below, r):
            kept = [j for j in range(n) if j not in sub]
            out = p[kept] @ v[kept]
            worst = np.maximum(worst, np.abs(out - dense))
    assert np.all(worst <= bound + 1e-15)
    # with values of one sign the bound is reached by skipping all of them
    vp = np.abs(v)
    bound_p = oracle.sparse_v_bound(q, k, vp, tau)
    np.testing.assert_allclose(p[below] @ vp[below], bound_p, rtol=1e-13)


def test_decode_sparse_v_bound_matches_per_row_bound():
    rng = np.random.default_rng(6)
    d, L = 128, 40
    k16 = rng.standard_normal((1, 2, L, d)).astype(np.float16)
    v16 = rng.standard_normal((1, 2, L, d)).astype(np.float16)
    q16 = (3.0 * rng.standard_normal((1, 4, d))).astype(np.float16)
    c = oracle.build_cache(k16, v16, [L], L, 3, 4)
    out = oracle.decode_sparse_v_bound(c, q16, [L], 0.01)
    for hq in range(4):
        k, v = oracle.dequantized_kv(c, 0, hq // 2, L)
        np.testing.assert_array_equal(out[0, hq], oracle.sparse_v_bound(q16[0, hq].astype(np.float64), k, v, 0.01))


def _masked_softmax_attention(q, k, v, pos):
    """Textbook causal attention of a block of queries: scores for every (query,
    key) pair, -inf above the diagonal given by the query positions, row softmax."""
    s = q @ k.T / math.sqrt(q.shape[-1])
    s = np.where(np.arange(k.shape[0])[None, :] <= pos[:, None], s, -np.inf)
    w = np.exp(s - s.max(axis=1, keepdims=True))
    w = np.where(np.isfinite(s), w, 0.0)
    return (w @ v) / w.sum(axis=1, keepdims=True)


@pytest.mark.parametrize("codec", ["turbo", "int8"])
def test_multi_query_attention_is_causal_block_attention(codec):
    rng = np.random.default_rng(21)
    B, HK, HQ, T, D, NQ = 2, 2, 4, 40, 128, 5
    k = rng.standard_normal((B, HK, T, D)).astype(np.float16)
    v = rng.standard_normal((B, HK, T, D)).astype(np.float16)
    lens = np.array([40, 23])
    cache = oracle.build_cache(k, v, lens, T, 3, 4, hot_window=7, codec=codec)
    q = (rng.standard_normal((B, NQ, HQ, D)) * 0.5).astype(np.float16)
    got = oracle.multi_query_attention(cache, q, lens)
    for b in range(B):
        for hq in range(HQ):
            kk, vv = oracle.dequantized_kv(cache, b, hq // 2, int(lens[b]))
            pos = lens[b] - NQ + np.arange(NQ)
            want = _masked_softmax_attention(q[b, :, hq].astype(np.float64), kk, vv, pos)
            np.testing.assert_allclose(got[b, :, hq], want, rtol=1e-12, atol=1e-12)


def test_multi_query_with_one_token_is_decode_and_early_queries_are_zero():
    rng = np.random.default_rng(22)
    B, HK, HQ, T, D = 3, 1, 2, 20, 128
    k = rng.standard_normal((B, HK, T, D)).astype(np.float16)
    v = rng.standard_normal((B, HK, T, D)).astype(np.float16)
    lens = np.array([20, 3, 0])
    cache = oracle.build_cache(k, v, lens, T, 4, 4)
    q = rng.standard_normal((B, 1, HQ, D)).astype(np.float16)
    one = oracle.multi_query_attention(cache, q, lens)[:, 0]
    dec = oracle.decode_attention(cache, q[:, 0], lens)
    np.testing.assert_array_equal(one[:2], dec[:2])
    assert np.all(one[2] == 0)
    q5 = rng.standard_normal((B, 5, HQ, D)).astype(np.float16)
    out = oracle.multi_query_attention(cache, q5, lens)
    assert np.all(out[1, :2] == 0) and np.all(out[2] == 0)  # positions -2, -1 and an empty sequence
    # the last query of a block sees exactly what a decode at the full length sees
    np.testing.assert_array_equal(out[:2, 4], oracle.decode_attention(cache, q5[:, 4], lens)[:2])
