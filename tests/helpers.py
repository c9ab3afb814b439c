"""Helpers shared by the test files: tolerance checks and oracle <-> device glue."""
from __future__ import annotations

import numpy as np

import oracle

# Tolerances of the attention output (float32 GPU vs float64 oracle).
ATTN_MAX_ABS = 2e-3
ATTN_REL_L2 = 1e-3
# Code exception rule: a code may differ only where the oracle's float32
# rotated coordinate is within 1e-6 of a threshold, and such codes must stay
# below 1e-5 of all codes.
CODE_NEAR = 1e-6
CODE_RATE = 1e-5


def assert_attention_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape
    assert np.all(np.isfinite(got)), what + ": non-finite output"
    diff = np.abs(got - ref)
    max_abs = float(diff.max()) if diff.size else 0.0
    den = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(got - ref) / den) if den > 0 else float(np.linalg.norm(got - ref))
    assert max_abs <= ATTN_MAX_ABS, "%s: max-abs %.3g > %.1g" % (what, max_abs, ATTN_MAX_ABS)
    assert rel <= ATTN_REL_L2, "%s: rel-L2 %.3g > %.1g" % (what, rel, ATTN_REL_L2)
    return max_abs, rel


def assert_code_rate(n_mismatch, n_codes, what=""):
    """The exception rate is defined over all codes compared by a test."""
    assert n_mismatch / max(n_codes, 1) < CODE_RATE, "%s: %d threshold-near mismatches of %d codes" % (
        what, n_mismatch, n_codes)


def compare_packed(got_words, ref_words, ref_y, bits, thresholds32, what="", check_rate=True):
    """Bit-exact word comparison with the counted threshold exception.

    got_words / ref_words: uint32 [N, d*bits/32]; ref_y: the oracle's float64
    rotated coordinates [N, d].  Every mismatching code must sit within 1e-6
    of a threshold; with ``check_rate`` the mismatch rate of this call is also
    checked (tests that compare several samples aggregate and check once).
    Returns (#mismatching codes, #codes)."""
    got_words = np.asarray(got_words).view(np.uint32).reshape(ref_words.shape)
    if np.array_equal(got_words, ref_words):
        return 0, ref_y.size
    d = ref_y.shape[1]
    rows = np.nonzero(np.any(got_words != ref_words, axis=1))[0]
    gc = oracle.unpack(got_words[rows], bits, d)
    rc = oracle.unpack(ref_words[rows], bits, d)
    mism = gc != rc
    y32 = ref_y[rows].astype(np.float32).astype(np.float64)
    gap = np.min(np.abs(y32[..., None] - thresholds32.astype(np.float64)[None, None, :]), axis=-1)
    bad = mism & (gap >= CODE_NEAR)
    assert not bad.any(), "%s: %d codes differ away from any threshold (e.g. gap %.3g)" % (
        what, int(bad.sum()), float(gap[bad].max()))
    n = int(mism.sum())
    if check_rate:
        assert_code_rate(n, ref_y.size, what)
    return n, ref_y.size


class RealBuffers:
    """Real allocations for the argument-validation tests of the launching entry
    points.  With a visible GPU they are device buffers of the sizes the call
    would use, so that a regression in the host-side validation launches on real,
    large-enough memory instead of a made-up address; without a GPU they are host
    arrays (no device exists, so no kernel can be launched at all)."""

    def __init__(self):
        try:
            import torch
            self._torch = torch if torch.cuda.is_available() else None
        except ImportError:
            self._torch = None
        self._keep = []

    def alloc(self, nbytes: int) -> int:
        """Address of a zeroed buffer of at least ``nbytes`` (256-byte aligned)."""
        nbytes = max(int(nbytes), 256)
        if self._torch is not None:
            t = self._torch.zeros((nbytes + 3) // 4, dtype=self._torch.int32, device="cuda")
            self._keep.append(t)
            return t.data_ptr()
        a = np.zeros(nbytes + 256, np.uint8)
        self._keep.append(a)
        return (a.ctypes.data + 255) & ~255

    def cache(self, desc) -> None:
        """Points every cache buffer of ``desc`` at a real allocation of its size."""
        from bit_kv_cache_10_gb300 import native as N
        for name, size in N.tq_cache_buffer_bytes(desc).items():
            if size:
                setattr(desc, name, self.alloc(size))
