"""Plain fp64 CPU oracle of TurboQuant KV-cache quantization and decode attention.

TEST INFRASTRUCTURE ONLY (see the package docstring): the CUDA library never
imports this module and the two share no code.

Sources (pages, by title and section):

* [MLX-VLM deep-dive] "TurboQuant KV Cache Quantization in MLX-VLM: Low-Bit
  Compression for Efficient Generation":
  - "The TurboQuantKVCache Class": packed uint32 buffers plus per-token norms.
  - "Quantization Codecs and Bit Splitting": K gets floor(bits), V ceil(bits).
  - "How TurboQuant KV Cache Quantization Works": random Hadamard rotation
    before scalar quantization; Beta-PDF Lloyd-Max codebook; MSE decoding;
    scores computed from the compressed form.
  - "Manual Cache Operations": each uint32 word encodes several low-bit codes.
  - FAQ "Where is the dequantization logic implemented?": dequantize uses the
    stored rotation and codebook and returns float32.
* [MLX-VLM CLI guide] "How to Use TurboQuant with the MLX-VLM CLI":
  - "What Is TurboQuant?": rotation helpers, codebook generator, ~76% memory
    reduction at 3.5 bits; scoring kernels with query-head repeat.
  - "Activation Logic and CLI Integration": when the TurboQuant scheme is on.
* [mlxcel doc] "TurboQuant KV cache":
  - "Available modes": fp16 K + 4-bit V (asym), 4-bit K and V (sym), hot fp16
    V window + packed cold tail (delegated).
  - "WHT head-dimension constraint": power-of-two head_dim only.
  - "Available modes" and the "Measured speed and the memory trade-off" table:
    the int8 mode, per-token INT8 absmax quantization of K and V (~2x), whose
    dequantization is a scale-and-add with no rotation and no codebook.

Where the pages leave a step open this file takes the plainest reading; every
such reading is listed in the design notes and repeated at the function.

Everything is float64 unless a step is defined on stored float32/fp16 values:
the stored norm is the correctly rounded float32 of the exact Euclidean norm,
the codebook is stored as float32, and the code decision compares the float32
rounding of the rotated coordinate with the float32 thresholds.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from fractions import Fraction

import numpy as np
from scipy import special

MASK64 = (1 << 64) - 1
SPLITMIX_GAMMA = 0x9E3779B97F4A7C15
LOG2E = 1.0 / math.log(2.0)

# --------------------------------------------------------------------------
# Rotation: seeded random signs, then a Hadamard transform scaled by 1/sqrt(d)
# --------------------------------------------------------------------------


def splitmix64(state: int) -> tuple[int, int]:
    """One step of SplitMix64 (Steele, Lea & Flood, OOPSLA 2014).

    Returns ``(new_state, output)``: the state advances by the golden-ratio
    increment and the output is the state passed through the two
    xor-shift-multiply rounds and a final xor-shift of that generator.
    """
    state = (state + SPLITMIX_GAMMA) & MASK64
    z = state
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return state, z ^ (z >> 31)


def rotation_signs(seed: int, layer: int, head: int, d: int) -> np.ndarray:
    """The per-head +-1 sign diagonal of the random Hadamard rotation.

    [MLX-VLM deep-dive, "How TurboQuant KV Cache Quantization Works"] names a
    deterministic random rotation; the pages give no generator.  Reading: the
    sign of coordinate i of KV head h in layer ``layer`` is -1 when bit 63 of
    the first SplitMix64 output from state ``seed + (layer<<32 | h<<16 | i)``
    is set, else +1.  K and V of one head share the signs.
    """
    seed, layer, head, d = int(seed), int(layer), int(head), int(d)  # plain Python integers (no numpy overflow)
    if not (0 <= head < 1 << 16 and 0 <= d <= 1 << 16 and 0 <= layer < 1 << 31):
        raise ValueError("head, d or layer out of range")
    out = np.empty(d, dtype=np.int8)
    base = (int(seed) + ((layer << 32) | (head << 16))) & MASK64
    for i in range(d):
        _, z = splitmix64((base + i) & MASK64)
        out[i] = -1 if (z >> 63) & 1 else 1
    return out


def hadamard(d: int) -> np.ndarray:
    """Dense Sylvester Hadamard matrix, H[i, j] = (-1)^popcount(i & j), float64.

    The rotation of [mlxcel doc, "WHT head-dimension constraint"] is a
    Walsh-Hadamard transform, which needs d to be a power of two.
    """
    if d < 1 or d & (d - 1):
        raise ValueError("Hadamard size must be a power of two (head_dim %d)" % d)
    i = np.arange(d)
    parity = np.zeros((d, d), dtype=np.int64)
    x = i[:, None] & i[None, :]
    while np.any(x):
        parity ^= x & 1
        x = x >> 1
    return np.where(parity == 1, -1.0, 1.0)


def rotation(seed: int, layer: int, head: int, d: int) -> np.ndarray:
    """R_h = (1/sqrt(d)) * H * diag(s_h): signs first, then the Hadamard, then the scale."""
    return hadamard(d) * rotation_signs(seed, layer, head, d)[None, :].astype(np.float64) / math.sqrt(d)


# --------------------------------------------------------------------------
# Lloyd-Max codebook for the post-rotation coordinate density
# --------------------------------------------------------------------------


def _density_norm(d: int) -> float:
    """C_d with C_d * integral_{-1}^{1} (1-x^2)^((d-3)/2) dx = 1."""
    return math.exp(math.lgamma(d / 2.0) - 0.5 * math.log(math.pi) - math.lgamma((d - 1) / 2.0))


def _mass(lo, hi, d):
    """P(lo < x < hi) for f_d: x = 2u - 1 with u ~ Beta((d-1)/2, (d-1)/2)."""
    a = (d - 1) / 2.0
    lo = np.asarray(lo, dtype=np.float64)
    hi = np.asarray(hi, dtype=np.float64)
    # use the upper tail where it keeps more digits
    lower = special.betainc(a, a, (hi + 1) / 2) - special.betainc(a, a, (lo + 1) / 2)
    upper = special.betaincc(a, a, (lo + 1) / 2) - special.betaincc(a, a, (hi + 1) / 2)
    return np.where(lo + hi > 0, upper, lower)


def _first_moment(lo, hi, d):
    """integral_lo^hi x f_d(x) dx = C_d [(1-lo^2)^((d-1)/2) - (1-hi^2)^((d-1)/2)] / (d-1)."""
    e = (d - 1) / 2.0
    lo = np.asarray(lo, dtype=np.float64)
    hi = np.asarray(hi, dtype=np.float64)
    return _density_norm(d) * ((1 - lo * lo) ** e - (1 - hi * hi) ** e) / (d - 1)


def _second_moment(lo, hi, d):
    """integral_lo^hi x^2 f_d(x) dx, by parts against the d+2 density.

    With g(x) = -(1-x^2)^((d-1)/2)/(d-1), g' = x (1-x^2)^((d-3)/2), so
    int x^2 f = C_d ([x g]_lo^hi + (1/(d-1)) int (1-x^2)^((d-1)/2) dx) and the
    last integral is the d+2 mass divided by C_{d+2}.
    """
    e = (d - 1) / 2.0
    lo = np.asarray(lo, dtype=np.float64)
    hi = np.asarray(hi, dtype=np.float64)
    xg = lambda x: -x * (1 - x * x) ** e / (d - 1)  # noqa: E731
    rest = _mass(lo, hi, d + 2) / (_density_norm(d + 2) * (d - 1))
    return _density_norm(d) * (xg(hi) - xg(lo) + rest)


@dataclass
class Codebook:
    head_dim: int
    bits: int
    centroids: np.ndarray       # float64 [2^b], ascending
    thresholds: np.ndarray      # float64 [2^b - 1], midpoints
    centroids32: np.ndarray     # float32 rounding of centroids
    thresholds32: np.ndarray    # float32 rounding of thresholds
    mse_per_coord: float        # E[(x - c(x))^2] under f_d, float64
    iterations: int


def lloyd_max(d: int, bits: int, tol: float = 1e-15, max_iter: int = 100000) -> Codebook:
    """MSE-optimal scalar codebook for f_d(x) = C_d (1-x^2)^((d-3)/2) on [-1, 1].

    [MLX-VLM deep-dive, "How TurboQuant KV Cache Quantization Works"]: a
    Beta-PDF-based Lloyd-Max quantizer; f_d is the density of one coordinate
    of a uniformly random unit vector in R^d, the Beta((d-1)/2, (d-1)/2)
    law moved to [-1, 1].  Lloyd's two conditions are iterated: thresholds
    are midpoints of neighbouring centroids, centroids are the conditional
    means of their cells (exact cell integrals from the incomplete beta
    function and the closed-form first moment).  Start: conditional means of
    the 2^b equiprobable cells.  The density is even, so each iterate is made
    exactly antisymmetric.  Stop when no centroid moves by more than ``tol``.
    """
    if d < 2 or not 1 <= bits <= 8:
        raise ValueError("need d >= 2 and 1 <= bits <= 8")
    k = 1 << bits
    a = (d - 1) / 2.0
    edges = 2 * special.betaincinv(a, a, np.arange(k + 1) / k) - 1
    edges[0], edges[-1] = -1.0, 1.0
    c = _first_moment(edges[:-1], edges[1:], d) / _mass(edges[:-1], edges[1:], d)
    c = (c - c[::-1]) / 2
    it = 0
    for it in range(1, max_iter + 1):
        t = (c[:-1] + c[1:]) / 2
        e = np.concatenate([[-1.0], t, [1.0]])
        cn = _first_moment(e[:-1], e[1:], d) / _mass(e[:-1], e[1:], d)
        cn = (cn - cn[::-1]) / 2
        step = float(np.max(np.abs(cn - c)))
        c = cn
        if step < tol:
            break
    t = (c[:-1] + c[1:]) / 2
    e = np.concatenate([[-1.0], t, [1.0]])
    lo, hi = e[:-1], e[1:]
    mse = float(np.sum(_second_moment(lo, hi, d) - 2 * c * _first_moment(lo, hi, d) + c * c * _mass(lo, hi, d)))
    return Codebook(d, bits, c, t, c.astype(np.float32), t.astype(np.float32), mse, it)


_CB_CACHE: dict = {}


def codebook(d: int, bits: int) -> Codebook:
    """Memoised ``lloyd_max(d, bits)``."""
    key = (d, bits)
    if key not in _CB_CACHE:
        _CB_CACHE[key] = lloyd_max(d, bits)
    return _CB_CACHE[key]


# --------------------------------------------------------------------------
# Bit budget helpers
# --------------------------------------------------------------------------


def split_bits(bits: float) -> tuple[int, int]:
    """[MLX-VLM deep-dive, "Quantization Codecs and Bit Splitting"]: K gets floor, V gets ceil."""
    return int(math.floor(bits)), int(math.ceil(bits))


def turboquant_enabled(bits, scheme=None) -> bool:
    """[MLX-VLM CLI guide, "Activation Logic and CLI Integration"], in words:
    no bit width means off; the explicit "turboquant" scheme means on; else on
    exactly when the bit width is not within 1e-6 of an integer."""
    if bits is None:
        return False
    if scheme == "turboquant":
        return True
    b = float(bits)
    return abs(b - round(b)) > 1e-6


def bytes_per_token_head(bits: int, d: int) -> int:
    """Stored bytes of one packed token vector: d*bits/8 of codes plus a float32 norm."""
    return d * bits // 8 + 4


# --------------------------------------------------------------------------
# Quantize / pack / dequantize
# --------------------------------------------------------------------------


def _exact_sum_squares(row16: np.ndarray) -> Fraction:
    return sum((Fraction(float(v)) ** 2 for v in row16), Fraction(0))


def norms_fp32(x16: np.ndarray) -> np.ndarray:
    """Correctly rounded float32 of the exact Euclidean norm of each fp16 row.

    [MLX-VLM deep-dive, "The TurboQuantKVCache Class"]: each token keeps its
    norm.  The float64 sum of squares is within ~1e-14 relative of the exact
    one, so its square root rounds to the right float32 unless the exact norm
    is very close to a float32 rounding midpoint; those rows are redone in
    exact rational arithmetic (ties to even).
    """
    x = np.ascontiguousarray(x16).reshape(-1, x16.shape[-1])
    xf = x.astype(np.float64)
    s = np.einsum("ij,ij->i", xf, xf)
    n32 = np.sqrt(s).astype(np.float32)
    up = np.nextafter(n32, np.float32(np.inf))
    dn = np.nextafter(n32, np.float32(0))
    mid_up = (n32.astype(np.float64) + up.astype(np.float64)) / 2
    mid_dn = (n32.astype(np.float64) + dn.astype(np.float64)) / 2
    near = (np.abs(s - mid_up * mid_up) <= 1e-12 * s) | ((n32 > 0) & (np.abs(s - mid_dn * mid_dn) <= 1e-12 * s))
    for r in np.nonzero(near)[0]:
        exact = _exact_sum_squares(x[r])
        cand = n32[r]
        mu = Fraction(float(mid_up[r])) ** 2
        md = Fraction(float(mid_dn[r])) ** 2
        if exact > mu or (exact == mu and (int(up[r].view(np.uint32)) & 1) == 0):
            cand = up[r]
        elif n32[r] > 0 and (exact < md or (exact == md and (int(dn[r].view(np.uint32)) & 1) == 0)):
            cand = dn[r]
        n32[r] = cand
    return n32.reshape(x16.shape[:-1])


def quantize_rows(x16: np.ndarray, rot: np.ndarray, cb: Codebook):
    """Quantize fp16 rows [N, d] with one rotation.

    Steps of [MLX-VLM deep-dive, "How TurboQuant KV Cache Quantization Works"]:
    1. n = ||x|| (stored as the correctly rounded float32, ``norms_fp32``);
    2. y = R (x / n) with R = H diag(s) / sqrt(d) (a zero row gives y = 0);
    3. code_i = #{k : fp32(y_i) >= t_k}, t the float32 thresholds: the index
       of the nearest float32 centroid, ties going up.
    Returns (codes uint8 [N, d], norms float32 [N], y float64 [N, d]).
    """
    x = x16.astype(np.float64)
    n32 = norms_fp32(x16)
    n64 = np.sqrt(np.einsum("ij,ij->i", x, x))
    safe = np.where(n64 > 0, n64, 1.0)
    u = np.where((n64 > 0)[:, None], x / safe[:, None], 0.0)
    y = u @ rot.T
    y32 = y.astype(np.float32)
    codes = (y32[:, :, None] >= cb.thresholds32[None, None, :]).sum(axis=2).astype(np.uint8)
    return codes, n32, y


def pack(codes: np.ndarray, bits: int) -> np.ndarray:
    """Pack codes [N, d] into uint32 words [N, d*bits/32], LSB-first bitstream.

    [MLX-VLM deep-dive, "Manual Cache Operations"] only says that each uint32
    word holds several low-bit codes.  Reading: code i occupies bits
    [i*bits, i*bits + bits) of the token's bitstream, bit j of the stream is
    bit (j mod 32) of word j // 32, and a code may straddle two words.
    """
    n, d = codes.shape
    if (d * bits) % 32:
        raise ValueError("d*bits must be a multiple of 32")
    words = np.zeros((n, d * bits // 32), dtype=np.uint64)
    c = codes.astype(np.uint64)
    for i in range(d):
        pos = i * bits
        w, off = divmod(pos, 32)
        v = c[:, i] << np.uint64(off)
        words[:, w] |= v & np.uint64(0xFFFFFFFF)
        if off + bits > 32:
            words[:, w + 1] |= v >> np.uint64(32)
    return words.astype(np.uint32)


def unpack(words: np.ndarray, bits: int, d: int) -> np.ndarray:
    """Inverse of ``pack``: codes uint8 [N, d]."""
    w64 = words.astype(np.uint64)
    n = w64.shape[0]
    codes = np.empty((n, d), dtype=np.uint8)
    mask = np.uint64((1 << bits) - 1)
    for i in range(d):
        pos = i * bits
        w, off = divmod(pos, 32)
        v = w64[:, w] >> np.uint64(off)
        if off + bits > 32:
            v |= w64[:, w + 1] << np.uint64(32 - off)
        codes[:, i] = (v & mask).astype(np.uint8)
    return codes


def dequantize_rows(codes: np.ndarray, norms32: np.ndarray, rot: np.ndarray, cb: Codebook) -> np.ndarray:
    """x_hat = n * R^T c[codes], float64 [N, d].

    [MLX-VLM deep-dive, FAQ on dequantization]: the stored rotation and
    codebook decode the packed words; the stored float32 norm rescales.
    """
    c = cb.centroids32.astype(np.float64)[codes]
    return norms32.astype(np.float64)[:, None] * (c @ rot)


# --------------------------------------------------------------------------
# Per-token INT8 absmax mode
# --------------------------------------------------------------------------

INT8_LEVEL = 127  # largest code magnitude: the absmax maps to +-127


def int8_quantize_rows(x16: np.ndarray):
    """Per-token INT8 absmax quantization of fp16 rows [N, d].

    [mlxcel doc, "Available modes"]: the int8 mode quantizes each token with
    its absolute maximum.  Reading (the pages give no formula): one float32
    scale per (token, KV head) vector, s = fp32(max_i |x_i|) / 127 (float32
    division, correctly rounded), and code_i = the integer nearest to the
    float32 quotient fp32(x_i) / s (float32 division), ties to even, clamped
    to [-127, 127].  A zero vector gets s = 0 and all codes 0.  The quotient
    and the rounding are taken in float32, the precision the kernel decides in.
    Returns (codes int8 [N, d], scales float32 [N]).
    """
    x = np.ascontiguousarray(x16).reshape(-1, x16.shape[-1]).astype(np.float32)
    amax = np.abs(x).max(axis=1) if x.shape[1] else np.zeros(x.shape[0], np.float32)
    s = (amax / np.float32(INT8_LEVEL)).astype(np.float32)
    safe = np.where(s > 0, s, np.float32(1.0)).astype(np.float32)
    quot = (x / safe[:, None]).astype(np.float32)
    codes = np.clip(np.rint(quot), -INT8_LEVEL, INT8_LEVEL)
    codes = np.where((s > 0)[:, None], codes, 0).astype(np.int8)
    return codes.reshape(x16.shape), s.reshape(x16.shape[:-1])


def int8_dequantize_rows(codes: np.ndarray, scales32: np.ndarray) -> np.ndarray:
    """x_hat = s * code, float64 [N, d] (exact: a float32 scale times a code of
    at most 8 bits fits in float64).  [mlxcel doc, "Measured speed and the
    memory trade-off"]: int8 dequantization is a scale-and-add."""
    return scales32.astype(np.float64)[..., None] * codes.astype(np.float64)


def int8_words(codes: np.ndarray) -> np.ndarray:
    """Stored form of int8 codes [N, d]: uint32 words [N, d/4], code i in byte
    i mod 4 (bits 8 (i mod 4) ..) of word i // 4 as two's complement, i.e. the
    LSB-first bitstream of ``pack`` with 8-bit fields."""
    return pack(codes.view(np.uint8), 8)


def int8_codes(words: np.ndarray, d: int) -> np.ndarray:
    """Inverse of ``int8_words``."""
    return unpack(words, 8, d).view(np.int8)


# --------------------------------------------------------------------------
# A packed cache as the oracle sees it, and decode attention over it
# --------------------------------------------------------------------------


@dataclass
class PackedCache:
    """Cache state with the same layout as the library's device buffers.

    k_fp16 is None for packed K; then k_words [B, Hkv, cap, d*kb/32] uint32
    and k_norms [B, Hkv, cap] float32.  v_words / v_norms likewise for V.
    With codec "int8" (k_bits = v_bits = 8) the words hold int8 codes
    (``int8_words``) and the norms the per-token absmax scales.
    With hot_window W > 0, v_hot [B, Hkv, W, d] fp16 holds position p of the
    last min(W, L) positions in slot p mod W and the packed V covers the rest.
    """
    seed: int
    layer: int
    head_dim: int
    k_bits: int
    v_bits: int
    k_words: np.ndarray | None
    k_norms: np.ndarray | None
    k_fp16: np.ndarray | None
    v_words: np.ndarray
    v_norms: np.ndarray
    hot_window: int = 0
    v_hot: np.ndarray | None = None
    codec: str = "turbo"  # "int8": K and V words hold int8 codes, the norms hold absmax scales


def cold_end(length: int, hot_window: int) -> int:
    """Number of leading positions of a length-L sequence stored packed."""
    return length - min(hot_window, length) if hot_window > 0 else length


def build_cache(k16: np.ndarray, v16: np.ndarray, lengths, capacity: int, k_bits: int, v_bits: int,
                seed: int = 0, layer: int = 0, k_fp16: bool = False, hot_window: int = 0,
                codec: str = "turbo") -> PackedCache:
    """Quantize full fp16 K/V [B, Hkv, T, d] into the state a cache holds after
    its sequences reached ``lengths`` (positions >= L of a row stay zero).
    codec "int8" stores K and V with ``int8_quantize_rows`` (bits ignored)."""
    b_, hk, t_, d = k16.shape
    lengths = np.asarray(lengths)
    if codec == "int8":
        return _build_int8_cache(k16, v16, lengths, capacity, seed, layer, hot_window)
    wk = d * k_bits // 32
    wv = d * v_bits // 32
    cb_k = None if k_fp16 else codebook(d, k_bits)
    cb_v = codebook(d, v_bits)
    k_words = None if k_fp16 else np.zeros((b_, hk, capacity, wk), np.uint32)
    k_norms = None if k_fp16 else np.zeros((b_, hk, capacity), np.float32)
    k_store = np.zeros((b_, hk, capacity, d), np.float16) if k_fp16 else None
    v_words = np.zeros((b_, hk, capacity, wv), np.uint32)
    v_norms = np.zeros((b_, hk, capacity), np.float32)
    v_hot = np.zeros((b_, hk, hot_window, d), np.float16) if hot_window > 0 else None
    for h in range(hk):
        rot = rotation(seed, layer, h, d)
        for b in range(b_):
            length = int(lengths[b])
            if k_fp16:
                k_store[b, h, :length] = k16[b, h, :length]
            else:
                codes, nrm, _ = quantize_rows(k16[b, h, :length], rot, cb_k)
                k_words[b, h, :length] = pack(codes, k_bits)
                k_norms[b, h, :length] = nrm
            ce = cold_end(length, hot_window)
            codes, nrm, _ = quantize_rows(v16[b, h, :ce], rot, cb_v)
            v_words[b, h, :ce] = pack(codes, v_bits)
            v_norms[b, h, :ce] = nrm
            for p in range(ce, length):
                v_hot[b, h, p % hot_window] = v16[b, h, p]
    return PackedCache(seed, layer, d, k_bits, v_bits, k_words, k_norms, k_store, v_words, v_norms,
                       hot_window, v_hot)


def _build_int8_cache(k16, v16, lengths, capacity, seed, layer, hot_window) -> PackedCache:
    b_, hk, _, d = k16.shape
    k_words = np.zeros((b_, hk, capacity, d // 4), np.uint32)
    k_norms = np.zeros((b_, hk, capacity), np.float32)
    v_words = np.zeros((b_, hk, capacity, d // 4), np.uint32)
    v_norms = np.zeros((b_, hk, capacity), np.float32)
    v_hot = np.zeros((b_, hk, hot_window, d), np.float16) if hot_window > 0 else None
    for b in range(b_):
        length = int(lengths[b])
        ce = cold_end(length, hot_window)
        for h in range(hk):
            codes, s = int8_quantize_rows(k16[b, h, :length])
            k_words[b, h, :length] = int8_words(codes)
            k_norms[b, h, :length] = s
            codes, s = int8_quantize_rows(v16[b, h, :ce])
            v_words[b, h, :ce] = int8_words(codes)
            v_norms[b, h, :ce] = s
            for p in range(ce, length):
                v_hot[b, h, p % hot_window] = v16[b, h, p]
    return PackedCache(seed, layer, d, 8, 8, k_words, k_norms, None, v_words, v_norms, hot_window, v_hot, "int8")


def dequantized_kv(cache: PackedCache, b: int, h: int, length: int):
    """Float64 K and V of positions [0, length) of one (batch, KV head) row."""
    d = cache.head_dim
    if cache.codec == "int8":
        k = int8_dequantize_rows(int8_codes(cache.k_words[b, h, :length], d), cache.k_norms[b, h, :length])
        ce = cold_end(length, cache.hot_window)
        v = np.empty((length, d), np.float64)
        v[:ce] = int8_dequantize_rows(int8_codes(cache.v_words[b, h, :ce], d), cache.v_norms[b, h, :ce])
        for p in range(ce, length):
            v[p] = cache.v_hot[b, h, p % cache.hot_window].astype(np.float64)
        return k, v
    rot = rotation(cache.seed, cache.layer, h, d)
    if cache.k_fp16 is not None:
        k = cache.k_fp16[b, h, :length].astype(np.float64)
    else:
        codes = unpack(cache.k_words[b, h, :length], cache.k_bits, d)
        k = dequantize_rows(codes, cache.k_norms[b, h, :length], rot, codebook(d, cache.k_bits))
    ce = cold_end(length, cache.hot_window)
    v = np.empty((length, d), np.float64)
    codes = unpack(cache.v_words[b, h, :ce], cache.v_bits, d)
    v[:ce] = dequantize_rows(codes, cache.v_norms[b, h, :ce], rot, codebook(d, cache.v_bits))
    for p in range(ce, length):
        v[p] = cache.v_hot[b, h, p % cache.hot_window].astype(np.float64)
    return k, v


def attention_one(q: np.ndarray, k: np.ndarray, v: np.ndarray) -> np.ndarray:
    """softmax(k q / sqrt(d)) v for one query vector, max-subtracted; zeros if L = 0."""
    if k.shape[0] == 0:
        return np.zeros(q.shape[-1])
    s = k @ q / math.sqrt(q.shape[-1])
    p = np.exp(s - s.max())
    return (p @ v) / p.sum()


def decode_attention(cache: PackedCache, q16: np.ndarray, lengths, pairs=None) -> np.ndarray:
    """Decode attention of fp16 queries [B, Hq, d] over the cache.

    Query head hq reads KV head hq // (Hq / Hkv) (contiguous GQA groups, the
    head repeat of [MLX-VLM CLI guide, "What Is TurboQuant?"]); scale 1/sqrt(d).
    ``pairs`` optionally restricts the work to a list of (b, hq); the other
    outputs are left NaN.  Returns float64 [B, Hq, d].
    """
    bsz, hq_n, d = q16.shape
    hk = cache.v_words.shape[1]
    g = hq_n // hk
    out = np.full((bsz, hq_n, d), np.nan)
    todo = pairs if pairs is not None else [(b, hq) for b in range(bsz) for hq in range(hq_n)]
    kv = {}
    for b, hq in todo:
        h = hq // g
        if (b, h) not in kv:
            kv = {(b, h): dequantized_kv(cache, b, h, int(lengths[b]))}
        k, v = kv[(b, h)]
        out[b, hq] = attention_one(q16[b, hq].astype(np.float64), k, v)
    return out


def multi_query_attention(cache: PackedCache, q16: np.ndarray, lengths, triples=None) -> np.ndarray:
    """Causal attention of the T newest tokens of every sequence, fp16 queries
    [B, T, Hq, d] -> float64 [B, T, Hq, d].

    The multi-token counterpart of ``decode_attention`` (prefill chunks and
    speculative verification; [mlxcel doc, "Measured speed and the memory
    trade-off"] reports prefill for every mode).  Reading: with L_b positions
    stored (the T new ones included), query i sits at position L_b - T + i and
    attends to positions 0 .. L_b - T + i; a query before position 0 gets zeros.
    ``triples`` optionally restricts the work to a list of (b, i, hq); the other
    outputs are left NaN.
    """
    bsz, t_n, hq_n, d = q16.shape
    hk = cache.v_words.shape[1]
    g = hq_n // hk
    out = np.full((bsz, t_n, hq_n, d), np.nan)
    todo = triples if triples is not None else [(b, i, hq) for b in range(bsz) for i in range(t_n)
                                                for hq in range(hq_n)]
    kv = {}
    for b, i, hq in todo:
        h = hq // g
        if (b, h) not in kv:
            kv = {(b, h): dequantized_kv(cache, b, h, int(lengths[b]))}
        k, v = kv[(b, h)]
        n = max(0, int(lengths[b]) - t_n + i + 1)
        out[b, i, hq] = attention_one(q16[b, i, hq].astype(np.float64), k[:n], v[:n])
    return out


def sparse_v_bound(q: np.ndarray, k: np.ndarray, v: np.ndarray, tau: float) -> np.ndarray:
    """Per-coordinate bound on how far a sparse-V decode may move one output.

    Sparse-V ([mlxcel doc] "Environment variables": a threshold setting whose
    zero value turns it off) skips the V rows of tokens whose softmax weight is
    below a threshold tau while their weight still counts in the normalization.  Any
    skipped set A of tokens with normalized weight p_j < tau changes the output
    by sum_{j in A} p_j v_j, so every coordinate moves by at most
    sum_{j: p_j < tau} p_j |v_ji|, which this returns (zeros for tau <= 0).
    """
    d = q.shape[-1]
    if tau <= 0.0 or k.shape[0] == 0:
        return np.zeros(d)
    s = k @ q / math.sqrt(d)
    p = np.exp(s - s.max())
    p = p / p.sum()
    skip = p < tau
    return p[skip] @ np.abs(v[skip])


def decode_sparse_v_bound(cache: PackedCache, q16: np.ndarray, lengths, tau: float, pairs=None) -> np.ndarray:
    """sparse_v_bound for every (b, query head) of a decode step (same layout
    and head grouping as decode_attention)."""
    bsz, hq_n, d = q16.shape
    hk = cache.v_words.shape[1]
    g = hq_n // hk
    out = np.full((bsz, hq_n, d), np.nan)
    todo = pairs if pairs is not None else [(b, hq) for b in range(bsz) for hq in range(hq_n)]
    kv = {}
    for b, hq in todo:
        h = hq // g
        if (b, h) not in kv:
            kv = {(b, h): dequantized_kv(cache, b, h, int(lengths[b]))}
        k, v = kv[(b, h)]
        out[b, hq] = sparse_v_bound(q16[b, hq].astype(np.float64), k, v, tau)
    return out


def decode_attention_rotated(cache: PackedCache, q16: np.ndarray, lengths, b: int, hq: int) -> np.ndarray:
    """Same output as ``decode_attention`` through the rotated-domain identity
    (R q).(R k_hat) = q.k_hat: scores from the rotated query and the raw
    centroids, V summed in the rotated domain and rotated back once.  Packed
    K only.  Used to check the oracle against itself."""
    d = cache.head_dim
    hk = cache.v_words.shape[1]
    g = q16.shape[1] // hk
    h = hq // g
    length = int(lengths[b])
    rot = rotation(cache.seed, cache.layer, h, d)
    qr = rot @ q16[b, hq].astype(np.float64)
    ck = codebook(d, cache.k_bits).centroids32.astype(np.float64)[unpack(cache.k_words[b, h, :length], cache.k_bits, d)]
    s = cache.k_norms[b, h, :length].astype(np.float64) * (ck @ qr) / math.sqrt(d)
    p = np.exp(s - s.max())
    ce = cold_end(length, cache.hot_window)
    cv = codebook(d, cache.v_bits).centroids32.astype(np.float64)[unpack(cache.v_words[b, h, :ce], cache.v_bits, d)]
    acc_rot = (p[:ce] * cache.v_norms[b, h, :ce].astype(np.float64)) @ cv
    out = rot.T @ acc_rot
    for pos in range(ce, length):
        out += p[pos] * cache.v_hot[b, h, pos % cache.hot_window].astype(np.float64)
    return out / p.sum()
