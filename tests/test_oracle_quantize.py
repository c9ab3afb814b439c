"""Pins of the oracle's quantize / pack / norm / dequantize (CPU only)."""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from bit_kv_cache_10_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_pack_cases():
    cases = []
    with open(os.path.join(GOLDEN, "pack_lsb_first.txt")) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            head, codes, words = (p.strip() for p in line.split("|"))
            bits, d = (int(v) for v in head.split())
            cases.append((bits, d, [int(c) for c in codes.split()], [int(w, 16) for w in words.split()]))
    return cases


@pytest.mark.parametrize("bits,d,codes,words", _golden_pack_cases())
def test_pack_matches_hand_derived_words(bits, d, codes, words):
    got = oracle.pack(np.array([codes], dtype=np.uint8), bits)
    assert [int(w) for w in got[0]] == words
    np.testing.assert_array_equal(oracle.unpack(got, bits, d)[0], codes)


@pytest.mark.parametrize("bits", [1, 2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("d", [32, 128])
def test_pack_roundtrip(bits, d):
    codes = np.random.default_rng(bits * d).integers(0, 1 << bits, size=(300, d)).astype(np.uint8)
    words = oracle.pack(codes, bits)
    assert words.shape == (300, d * bits // 32) and words.dtype == np.uint32
    np.testing.assert_array_equal(oracle.unpack(words, bits, d), codes)


def _exact_norm_fp32(row):
    s = sum((Fraction(float(v)) ** 2 for v in row), Fraction(0))
    # correctly rounded float32 of sqrt(s) by bisection over float32 bit patterns
    lo, hi = 0, 0x7F800000
    while hi - lo > 1:
        mid = (lo + hi) // 2
        f = Fraction(float(np.array(mid, dtype=np.uint32).view(np.float32)))
        if f * f <= s:
            lo = mid
        else:
            hi = mid
    a = Fraction(float(np.array(lo, dtype=np.uint32).view(np.float32)))
    b = Fraction(float(np.array(lo + 1, dtype=np.uint32).view(np.float32)))
    m = (a + b) / 2
    pick = lo if (m * m > s or (m * m == s and lo % 2 == 0)) else lo + 1
    return np.array(pick, dtype=np.uint32).view(np.float32)


def test_norm_is_correctly_rounded_exact_norm():
    x = synth.kv_fp16(3, synth.STREAM_K, 1, 4, 100, 16, scales=synth.channel_scales(3, 4, 4, 16)).reshape(-1, 16)
    got = oracle.norms_fp32(x)
    for r in range(x.shape[0]):
        assert got[r] == _exact_norm_fp32(x[r]), r


def test_norm_exact_cases():
    rows = np.array([[3, 4, 0, 0], [5, 12, 0, 0], [0, 0, 0, 0], [1, 1, 1, 1], [-8, 6, 0, 0],
                     [65504, 65504, 65504, 65504]], dtype=np.float16)
    got = oracle.norms_fp32(rows)
    np.testing.assert_array_equal(got[:5], np.array([5, 13, 0, 2, 10], np.float32))
    assert got[5] == np.float32(131008.0)


def test_norm_fast_path_agrees_with_exact_path():
    x = synth.kv_fp16(9, synth.STREAM_V, 1, 2, 400, 128, scales=synth.channel_scales(9, 5, 2, 128)).reshape(-1, 128)
    fast = oracle.norms_fp32(x)
    ref = np.array([_exact_norm_fp32(r) for r in x[:150]])
    np.testing.assert_array_equal(fast[:150], ref)


def test_zero_vector_codes_are_middle():
    for bits in (2, 3, 4):
        cb = oracle.codebook(128, bits)
        codes, n, y = oracle.quantize_rows(np.zeros((2, 128), np.float16), oracle.rotation(0, 0, 0, 128), cb)
        assert np.all(codes == 1 << (bits - 1)) and np.all(n == 0) and np.all(y == 0)
        xh = oracle.dequantize_rows(codes, n, oracle.rotation(0, 0, 0, 128), cb)
        assert np.all(xh == 0)


def test_quantize_scale_invariance():
    x = synth.kv_fp16(1, 1, 1, 1, 64, 128).reshape(-1, 128)
    rot = oracle.rotation(0, 0, 0, 128)
    cb = oracle.codebook(128, 3)
    c1, n1, _ = oracle.quantize_rows(x, rot, cb)
    c2, n2, _ = oracle.quantize_rows((x.astype(np.float32) * 4).astype(np.float16), rot, cb)
    np.testing.assert_array_equal(c1, c2)
    np.testing.assert_array_equal(n2, n1 * 4)


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_quantize_mse_matches_codebook_distortion(bits):
    d = 128
    x = synth.kv_fp16(11, 1, 1, 1, 20000, d).reshape(-1, d)
    rot = oracle.rotation(0, 0, 0, d)
    cb = oracle.codebook(d, bits)
    codes, n, _ = oracle.quantize_rows(x, rot, cb)
    xh = oracle.dequantize_rows(codes, n, rot, cb)
    xf = x.astype(np.float64)
    rel = np.sum((xf - xh) ** 2) / np.sum(xf ** 2)
    # a random rotation makes every coordinate follow f_d; each vector's
    # relative error is then d * MSE_b on average
    assert rel == pytest.approx(d * cb.mse_per_coord, rel=0.03)


def test_codes_follow_threshold_definition_and_rotation_order():
    d = 16
    x = synth.kv_fp16(2, 2, 1, 1, 50, d, scales=synth.channel_scales(2, 5, 1, d)).reshape(-1, d)
    rot = oracle.rotation(5, 1, 0, d)
    cb = oracle.codebook(d, 4)
    codes, n, y = oracle.quantize_rows(x, rot, cb)
    s = oracle.rotation_signs(5, 1, 0, d).astype(np.float64)
    h = oracle.hadamard(d)
    for r in range(x.shape[0]):
        xr = x[r].astype(np.float64)
        yr = h @ (s * xr / np.linalg.norm(xr)) / math.sqrt(d)
        np.testing.assert_allclose(y[r], yr, atol=1e-15)
        for i in range(d):
            assert codes[r, i] == sum(np.float32(yr[i]) >= t for t in cb.thresholds32)


def test_storage_ratios_quoted_by_the_pages():
    d = 128
    fp16 = 2 * d
    k3, v4 = oracle.split_bits(3.5)
    packed = oracle.bytes_per_token_head(k3, d) + oracle.bytes_per_token_head(v4, d)
    # "approximately 76% memory reduction" at 3.5 bits, "4-5x" reduction
    assert 1 - packed / (2 * fp16) == pytest.approx(0.766, abs=0.01)
    assert 4 <= 2 * fp16 / packed <= 5
    # turbo4-asym "~3.8x V", turbo3-asym "~5x V", turbo4 "~4x K+V"
    assert fp16 / oracle.bytes_per_token_head(4, d) == pytest.approx(3.8, abs=0.05)
    assert fp16 / oracle.bytes_per_token_head(3, d) == pytest.approx(5.0, abs=0.1)
    assert 2 * fp16 / (2 * oracle.bytes_per_token_head(4, d)) == pytest.approx(4.0, abs=0.25)
