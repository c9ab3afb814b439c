"""Seeded synthetic inputs for the packed-KV hot path.

This module only draws random numbers: it holds none of the quantizer's
arithmetic (no rotation, no codebook, no packing).  Both the CPU oracle and
the CUDA library are fed from it, so that a parity test compares the two on
exactly the same bytes.

Every draw comes from numpy's PCG64 generator keyed by ``(seed, stream)``
through a ``SeedSequence``; the stream ids name what is drawn:

========  =====================================================
stream    what
========  =====================================================
1         K token vectors (N(0,1) before channel scaling)
2         V token vectors
3         decode queries
4         per-channel K scales, lognormal(0, 1)
5         per-channel V scales, lognormal(0, 1)
6         per-sequence context lengths
7         codes of a synthetic packed K cache (decode-only tests)
8         codes of a synthetic packed V cache
9         norms of a synthetic packed K cache
10        norms of a synthetic packed V cache
========  =====================================================

The workloads follow the shapes of the TurboQuant pages' measurements: fp16
K/V drawn i.i.d. N(0, 1), optionally multiplied by a per-(head, channel)
lognormal(0, 1) scale (outlier channels), and rounded to fp16 with
round-to-nearest-even.
"""
from __future__ import annotations

import numpy as np

STREAM_K = 1
STREAM_V = 2
STREAM_Q = 3
STREAM_SCALE_K = 4
STREAM_SCALE_V = 5
STREAM_LENGTHS = 6
STREAM_CODES_K = 7
STREAM_CODES_V = 8
STREAM_NORMS_K = 9
STREAM_NORMS_V = 10


def rng(seed: int, stream: int) -> np.random.Generator:
    """PCG64 generator for one (seed, stream) pair."""
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), int(stream)])))


def channel_scales(seed: int, stream: int, num_heads: int, head_dim: int) -> np.ndarray:
    """lognormal(0, 1) scale per (KV head, channel), float64 [num_heads, head_dim]."""
    return np.exp(rng(seed, stream).standard_normal((num_heads, head_dim)))


def kv_fp16(seed: int, stream: int, batch: int, num_heads: int, tokens: int, head_dim: int,
            scales: np.ndarray | None = None) -> np.ndarray:
    """fp16 token vectors [batch, num_heads, tokens, head_dim].

    Values are N(0, 1) (times ``scales[h, i]`` when given), rounded to fp16.
    Large draws are generated in float32 to halve the host memory they need.
    """
    g = rng(seed, stream)
    out = np.empty((batch, num_heads, tokens, head_dim), dtype=np.float16)
    for b in range(batch):
        for h in range(num_heads):
            x = g.standard_normal((tokens, head_dim), dtype=np.float32)
            if scales is not None:
                x *= scales[h].astype(np.float32)[None, :]
            out[b, h] = x.astype(np.float16)
    return out


def queries_fp16(seed: int, batch: int, num_q_heads: int, head_dim: int) -> np.ndarray:
    """Decode queries, fp16 N(0, 1) [batch, num_q_heads, head_dim] (unscaled)."""
    return rng(seed, STREAM_Q).standard_normal((batch, num_q_heads, head_dim)).astype(np.float16)


def seq_lengths(seed: int, batch: int, lo: int, hi: int) -> np.ndarray:
    """Per-sequence context lengths, uniform integers in [lo, hi] inclusive (int32)."""
    return rng(seed, STREAM_LENGTHS).integers(lo, hi, size=batch, endpoint=True).astype(np.int32)


def random_codes(seed: int, stream: int, shape: tuple, bits: int) -> np.ndarray:
    """Uniform random integer codes in [0, 2**bits), uint8 array of ``shape``."""
    return rng(seed, stream).integers(0, 1 << bits, size=shape, dtype=np.uint8)


def random_norms(seed: int, stream: int, shape: tuple, median: float = 30.0,
                 sigma: float = 0.3) -> np.ndarray:
    """Positive float32 norms, lognormal around ``median`` (spread ``sigma``)."""
    g = rng(seed, stream)
    return (median * np.exp(sigma * g.standard_normal(shape))).astype(np.float32)


def row_rng(seed: int, stream: int, b: int, h: int) -> np.random.Generator:
    """PCG64 generator of one (batch, KV head) row of a stream, so that a
    sampled row can be drawn without drawing the whole cache."""
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), int(stream), int(b), int(h)])))


def packed_row(seed: int, stream: int, b: int, h: int, tokens: int, words_per_token: int,
               norm_median: float, norm_sigma: float = 0.3):
    """Random packed words uint32 [tokens, words_per_token] and lognormal
    float32 norms [tokens] of one cache row: every bit pattern is a valid
    packed record, so uniform random words stand in for a filled cache."""
    words = row_rng(seed, stream, b, h).integers(0, 2 ** 32, size=(tokens, words_per_token), dtype=np.uint32)
    g = row_rng(seed, stream + 1000, b, h)  # separate stream: a shorter draw is a prefix of a longer one
    norms = (norm_median * np.exp(norm_sigma * g.standard_normal(tokens))).astype(np.float32)
    return words, norms
