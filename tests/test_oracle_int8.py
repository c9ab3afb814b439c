"""Pins of the oracle's per-token INT8 absmax mode (CPU only).

The int8 mode of the mlxcel page ("Available modes": per-token INT8 absmax
quantization; "Measured speed and the memory trade-off": ~2x compression and a
scale-and-add dequantization).  Each test fixes a value by something other than
the oracle's own formula: hand-derived codes, exact rational arithmetic,
exhaustive search over the 255 codes, or a lossless special case that reduces
int8 attention to plain softmax attention."""
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle
from bit_kv_cache_10_gb300 import synth


def _row(values, d=8):
    x = np.zeros((1, d), np.float16)
    x[0, :len(values)] = values
    return x


def test_hand_derived_codes_scale_one():
    # absmax 127 -> scale exactly 1; codes are x rounded half to even
    x = _row([127.0, -127.0, 2.5, 3.5, -2.5, -3.5, 0.5, 1.5])
    codes, s = oracle.int8_quantize_rows(x)
    assert s[0] == np.float32(1.0)
    assert codes[0].tolist() == [127, -127, 2, 4, -2, -4, 0, 2]


def test_hand_derived_codes_scale_two():
    # absmax 254 -> scale 2; quotients 2.5 and 3.5 go to the even neighbour
    x = _row([254.0, 5.0, 7.0, -5.0, 1.0, 3.0, -253.0, 0.0])
    codes, s = oracle.int8_quantize_rows(x)
    assert s[0] == np.float32(2.0)
    assert codes[0].tolist() == [127, 2, 4, -2, 0, 2, -126, 0]


def test_zero_row_has_zero_scale_and_codes():
    codes, s = oracle.int8_quantize_rows(np.zeros((3, 128), np.float16))
    assert np.all(s == 0) and np.all(codes == 0)


def _fp32_correctly_rounded(num: Fraction) -> np.float32:
    """Nearest float32 to a positive rational (ties to even), by bisection over bit patterns."""
    lo, hi = 0, 0x7F800000
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if Fraction(float(np.array(mid, np.uint32).view(np.float32))) <= num:
            lo = mid
        else:
            hi = mid
    a = Fraction(float(np.array(lo, np.uint32).view(np.float32)))
    b = Fraction(float(np.array(lo + 1, np.uint32).view(np.float32)))
    if num - a < b - num or (num - a == b - num and lo % 2 == 0):
        return np.array(lo, np.uint32).view(np.float32)
    return np.array(lo + 1, np.uint32).view(np.float32)


def test_scale_is_the_correctly_rounded_absmax_over_127():
    x = synth.kv_fp16(5, synth.STREAM_K, 1, 1, 40, 128)[0, 0]
    _, s = oracle.int8_quantize_rows(x)
    for r in range(x.shape[0]):
        amax = max(abs(Fraction(float(v))) for v in x[r])
        assert s[r] == _fp32_correctly_rounded(amax / 127), r


def test_codes_by_exhaustive_search():
    # every code is the nearest of the 255 levels to the float32 quotient (ties to even)
    x = synth.kv_fp16(6, synth.STREAM_V, 1, 2, 24, 128).reshape(-1, 128)
    codes, s = oracle.int8_quantize_rows(x)
    levels = np.arange(-127, 128, dtype=np.float64)
    for r in range(x.shape[0]):
        quot = (x[r].astype(np.float32) / s[r]).astype(np.float64)  # the float32 quotient of the reading
        dist = np.abs(quot[:, None] - levels[None, :])
        best = dist.min(axis=1, keepdims=True)
        cand = dist == best
        want = np.empty(128, np.int64)
        for i in range(128):
            ks = levels[cand[i]].astype(np.int64)
            want[i] = ks[0] if len(ks) == 1 else ks[ks % 2 == 0][0]
        np.testing.assert_array_equal(codes[r].astype(np.int64), want)


def test_invariants_absmax_code_and_error_bound():
    x = synth.kv_fp16(7, synth.STREAM_K, 2, 2, 50, 128, synth.channel_scales(7, synth.STREAM_SCALE_K, 2, 128))
    x = x.reshape(-1, 128)
    codes, s = oracle.int8_quantize_rows(x)
    xf = x.astype(np.float64)
    i = np.abs(xf).argmax(axis=1)
    r = np.arange(x.shape[0])
    assert np.all(np.abs(codes[r, i]) == 127)
    assert np.all(np.sign(codes[r, i]) == np.sign(xf[r, i]))
    assert np.abs(codes.astype(np.int64)).max() == 127
    # |x/s - code| <= 1/2 + half an ulp of the float32 quotient (|x/s| <= 127: ulp <= 2^-17)
    err = np.abs(xf - oracle.int8_dequantize_rows(codes, s))
    assert np.all(err <= s.astype(np.float64)[:, None] * (0.5 + 2.0 ** -18))


def test_dequantize_is_exact_scale_times_code():
    codes = np.array([[-127, -1, 0, 1, 127, 64, -64, 3]], np.int8)
    s = np.array([np.float32(0.1)], np.float32)
    got = oracle.int8_dequantize_rows(codes, s)
    for c, g in zip(codes[0], got[0]):
        assert Fraction(g) == Fraction(float(s[0])) * int(c)


def test_word_layout_bytes_lsb_first_twos_complement():
    codes = np.array([[1, -1, 127, -127, 0, 2, -128 + 1, 5]], np.int8)
    w = oracle.int8_words(codes)
    assert w.dtype == np.uint32 and w.shape == (1, 2)
    assert int(w[0, 0]) == 0x817FFF01
    assert int(w[0, 1]) == 0x05810200
    np.testing.assert_array_equal(oracle.int8_codes(w, 8), codes)


def test_compression_about_two_x():
    # 128 int8 codes + a float32 scale per token-head against 256 fp16 bytes
    d = 128
    stored = d + 4
    assert abs(2 * d / stored - 2.0) < 0.07


def test_lossless_inputs_reduce_to_plain_attention():
    # integer-valued rows with absmax 127 quantize exactly (scale 1), so int8
    # decode must equal textbook softmax attention over the fp16 values
    rng = np.random.default_rng(3)
    B, HK, HQ, T, D = 2, 2, 4, 37, 128
    k = rng.integers(-126, 127, size=(B, HK, T, D)).astype(np.float16)
    v = rng.integers(-126, 127, size=(B, HK, T, D)).astype(np.float16)
    k[..., 5] = 127.0
    v[..., 9] = -127.0
    lens = np.array([37, 20])
    cache = oracle.build_cache(k, v, lens, T, 8, 8, codec="int8")
    assert np.all(cache.k_norms[0, :, :37] == 1.0)
    q = (rng.standard_normal((B, HQ, D)) * 0.02).astype(np.float16)
    got = oracle.decode_attention(cache, q, lens)
    for b in range(B):
        for hq in range(HQ):
            kk = k[b, hq // 2, :lens[b]].astype(np.float64)
            vv = v[b, hq // 2, :lens[b]].astype(np.float64)
            sc = kk @ q[b, hq].astype(np.float64) / math.sqrt(D)
            w = np.exp(sc - sc.max())
            np.testing.assert_allclose(got[b, hq], (w @ vv) / w.sum(), rtol=1e-12, atol=1e-10)


def test_int8_cache_with_hot_window_keeps_newest_v_raw():
    rng = np.random.default_rng(4)
    B, HK, T, D, W = 1, 1, 30, 128, 8
    k = rng.standard_normal((B, HK, T, D)).astype(np.float16)
    v = rng.standard_normal((B, HK, T, D)).astype(np.float16)
    cache = oracle.build_cache(k, v, [30], 32, 8, 8, hot_window=W, codec="int8")
    _, vv = oracle.dequantized_kv(cache, 0, 0, 30)
    np.testing.assert_array_equal(vv[22:], v[0, 0, 22:].astype(np.float64))
    assert np.all(cache.v_norms[0, 0, 22:] == 0)
    codes, s = oracle.int8_quantize_rows(v[0, 0, :22])
    np.testing.assert_array_equal(vv[:22], oracle.int8_dequantize_rows(codes, s))


@pytest.mark.parametrize("bad", [np.float16(65504.0), np.float16(-65504.0)])
def test_extreme_fp16_values(bad):
    x = _row([bad, 1.0, -1.0, 0.0])
    codes, s = oracle.int8_quantize_rows(x)
    assert abs(int(codes[0, 0])) == 127 and codes[0, 1] == 0
