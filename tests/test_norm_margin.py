"""The kernels' exact-norm decision near float32 rounding midpoints.

The quantizer decides the correctly rounded float32 norm from a double-float
sum of squares and sends a vector to the exact integer sum only when the float
residual lies within 2^-37 S of a rounding midpoint (S the sum of squares); the
written error bound of the float residual is 2^-39.4 S.  These vectors are
built so that S sits at chosen relative distances from a midpoint's square,
from far inside the exact-sum window to well outside it, and the host build of
the kernels' quantizer must return the oracle's exact norms for all of them.
"""
import math

import numpy as np
import pytest

import oracle
from bit_kv_cache_10_gb300 import native as N


def _units(x) -> int:
    """x^2 in units of 2^-48 (exact: every fp16 times 2^24 is an integer)."""
    v = int(float(x) * 2 ** 24)
    return v * v


def _fp16_floor_sqrt(units: int) -> np.float16:
    """Largest non-negative fp16 x with x^2 <= units * 2^-48."""
    if units <= 0:
        return np.float16(0.0)
    x = np.float16(math.sqrt(units) * 2.0 ** -24)
    while _units(x) > units:
        x = np.nextafter(x, np.float16(0.0))
    while True:
        up = np.nextafter(x, np.float16(np.inf))
        if _units(up) > units:
            return x
        x = up


def _near_midpoint_row(rng, rel):
    """128 fp16 values whose sum of squares is M^2 (1 + rel) to within a few
    2^-48, M = n0 + ulp(n0) / 2 for a random float32 n0 in [1, 2).  Returns the
    row (with random signs) and the achieved relative distance from M^2."""
    k = int(rng.integers(1 << 23, 1 << 24))    # n0 = k 2^-23
    mid2 = (2 * k + 1) ** 2                    # M^2 in units of 2^-48 (M = (2k + 1) 2^-24)
    rem = mid2 + int(round(rel * mid2))
    row = np.zeros(128, np.float16)
    for i in range(128):  # greedy: each square takes what is left, about 2^-10 of it remains
        row[i] = _fp16_floor_sqrt(rem)
        rem -= _units(row[i])
        if rem == 0:
            break
    row = row[rng.permutation(128)]
    s = sum(_units(v) for v in row)
    signs = np.where(rng.random(128) < 0.5, -1.0, 1.0).astype(np.float16)
    return row * signs, (s - mid2) / mid2


def test_norms_near_rounding_midpoints():
    rng = np.random.default_rng(2024)
    rows, dists = [], []
    for e in np.linspace(-46, -30, 33):  # relative distance of S from a midpoint's square
        for sign in (-1.0, 1.0):
            for _ in range(3):
                r, d = _near_midpoint_row(rng, sign * 2.0 ** e)
                rows.append(r)
                dists.append(abs(d))
    rows = np.stack(rows)
    dists = np.array(dists)
    np.testing.assert_array_equal(rows, _rows())
    # the construction reaches both sides of the 2^-37 window and the float-decided zone
    assert dists.min() < 2.0 ** -44 and dists.max() > 2.0 ** -32
    assert np.any((dists > 2.0 ** -39) & (dists < 2.0 ** -36))
    cb = N.tq_build_codebook(128, 3)
    words, norms = N.tq_debug_quantize_rows_host(cb, 0, 0, 0, rows)
    ref = oracle.norms_fp32(rows)
    np.testing.assert_array_equal(norms, ref)


def _rows():
    rng = np.random.default_rng(2024)
    rows = []
    for e in np.linspace(-46, -30, 33):
        for sign in (-1.0, 1.0):
            for _ in range(3):
                rows.append(_near_midpoint_row(rng, sign * 2.0 ** e)[0])
    return np.stack(rows)


@pytest.mark.gpu
def test_kernel_norms_near_rounding_midpoints():
    """The same vectors through the GPU append (bulk and small-append kernels)."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from bit_kv_cache_10_gb300 import build
    from bit_kv_cache_10_gb300.cache import TurboQuantKVCache
    build.build()
    rows = _rows()
    n = rows.shape[0]
    ref = oracle.norms_fp32(rows)
    x = torch.from_numpy(rows.reshape(1, 1, n, 128)).cuda()
    tc = TurboQuantKVCache(1, 1, 1, n, bits=3.5)
    tc.append(x, x, torch.zeros(1, dtype=torch.int32, device="cuda"))  # one bulk append
    assert tc.device_status() == 0
    np.testing.assert_array_equal(tc.k_norms[0, 0].cpu().numpy(), ref)
    np.testing.assert_array_equal(tc.v_norms[0, 0].cpu().numpy(), ref)
    small = TurboQuantKVCache(1, 1, 1, n, bits=3.5)
    for t in range(0, n, 8):  # appends of 8 tokens: the one-warp-per-vector kernel
        m = min(8, n - t)
        small.append(x[:, :, t:t + m], x[:, :, t:t + m], torch.full((1,), t, dtype=torch.int32, device="cuda"))
    assert small.device_status() == 0
    np.testing.assert_array_equal(small.k_norms[0, 0].cpu().numpy(), ref)
