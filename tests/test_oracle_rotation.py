"""Pins of the oracle's rotation against what mathematics and published
definitions fix (CPU only)."""
import math

import numpy as np
import pytest
import scipy.linalg

import oracle


def test_splitmix64_published_outputs():
    # First outputs of SplitMix64 started from state 0, as printed with the
    # generator's reference implementation (Steele, Lea & Flood; Vigna).
    expected = [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F, 0xF88BB8A8724C81EC]
    state, got = 0, []
    for _ in range(4):
        state, z = oracle.splitmix64(state)
        got.append(z)
    assert got == expected


def test_signs_are_balanced_and_seeded():
    s = np.concatenate([oracle.rotation_signs(0, 0, h, 128) for h in range(32)])
    n_neg = int((s < 0).sum())
    # 4096 fair coin flips: 5 sigma band
    assert abs(n_neg - 2048) < 5 * 32
    assert set(np.unique(s)) == {-1, 1}
    a = oracle.rotation_signs(0, 0, 3, 128)
    b = oracle.rotation_signs(1, 0, 3, 128)
    c = oracle.rotation_signs(0, 1, 3, 128)
    assert (a != b).any() and (a != c).any()
    np.testing.assert_array_equal(a, oracle.rotation_signs(0, 0, 3, 128))


def test_sign_counter_layout():
    # the counter for (layer, head, i) is layer<<32 | head<<16 | i added to the seed
    for layer, head, i in [(0, 0, 0), (2, 5, 77), (7, 1, 127)]:
        _, z = oracle.splitmix64((123 + ((layer << 32) | (head << 16) | i)) & oracle.MASK64)
        expect = -1 if z >> 63 else 1
        assert oracle.rotation_signs(123, layer, head, 128)[i] == expect


@pytest.mark.parametrize("d", [1, 2, 4, 8, 16, 32, 64, 128, 256])
def test_hadamard_is_sylvester_and_orthogonal(d):
    h = oracle.hadamard(d)
    np.testing.assert_array_equal(h, scipy.linalg.hadamard(d).astype(np.float64))
    np.testing.assert_array_equal(h @ h.T, d * np.eye(d))


def test_hadamard_rejects_non_power_of_two():
    for d in (3, 80, 96, 100):
        with pytest.raises(ValueError):
            oracle.hadamard(d)


def _fwht_natural(x):
    # in-place butterflies on index bits 0, 1, 2, ... (natural order output)
    x = np.array(x, dtype=np.int64)
    n, h = x.shape[-1], 1
    while h < n:
        for i in range(0, n, 2 * h):
            a = x[..., i:i + h].copy()
            b = x[..., i + h:i + 2 * h].copy()
            x[..., i:i + h] = a + b
            x[..., i + h:i + 2 * h] = a - b
        h *= 2
    return x


def test_butterfly_matches_dense_hadamard_exactly():
    rng = np.random.default_rng(5)
    x = rng.integers(-1000, 1000, size=(50, 128))
    np.testing.assert_array_equal(_fwht_natural(x), (x @ oracle.hadamard(128).T).astype(np.int64))


def test_rotation_is_orthonormal_and_inverts():
    rot = oracle.rotation(0, 0, 2, 128)
    np.testing.assert_allclose(rot.T @ rot, np.eye(128), atol=1e-15)
    x = np.random.default_rng(1).standard_normal((10, 128))
    np.testing.assert_allclose((x @ rot.T) @ rot, x, atol=1e-13)
    # signs applied before the Hadamard: R e_j = s_j H e_j / sqrt(d)
    s = oracle.rotation_signs(0, 0, 2, 128)
    h = oracle.hadamard(128)
    for j in (0, 5, 127):
        np.testing.assert_allclose(rot[:, j], s[j] * h[:, j] / math.sqrt(128), atol=0)
