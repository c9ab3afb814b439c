"""GPU parity of the asym mode (fp16 K, packed V) against the oracle.

fp16 K runs the tensor-core kernel (scores from ldmatrix fragments of the staged
fp16 rows against the raw fp16 query) with packed V of 4 bits, or of 3 bits spread
to nibbles.  Cases: empty rows, rows shorter than a tile, partial last tiles,
hot windows longer and shorter than the rows, group sizes 1, 2 and 4, peaked
softmax, and sparse V within the oracle's exact deviation bound.
"""
import numpy as np
import pytest

import oracle
from bit_kv_cache_10_gb300 import native as N
from bit_kv_cache_10_gb300 import synth

from helpers import ATTN_MAX_ABS, assert_attention_close

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


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _asym_pair(seed, lens, hk, hq, vb, hot, qscale):
    from bit_kv_cache_10_gb300.cache import TurboQuantKVCache
    lens = np.asarray(lens, np.int32)
    B, cap = len(lens), int(lens.max())
    k = synth.kv_fp16(seed, 1, B, hk, cap, D, synth.channel_scales(seed, 4, hk, D))
    v = synth.kv_fp16(seed, 2, B, hk, cap, D, synth.channel_scales(seed, 5, hk, D))
    q = (synth.queries_fp16(seed, B, hq, D).astype(np.float32) * qscale).astype(np.float16)
    oc = oracle.build_cache(k, v, lens, cap, 16, vb, hot_window=hot, k_fp16=True)
    tc = TurboQuantKVCache(batch=B, num_kv_heads=hk, num_q_heads=hq, capacity=cap, bits=(4, vb), hot_window=hot,
                           k_fp16=True)
    tc.k_cache.copy_(_dev(oc.k_fp16))
    tc.v_cache.copy_(_dev(oc.v_words.view(np.int32)))
    tc.v_norms.copy_(_dev(oc.v_norms))
    if oc.v_hot is not None:
        tc.v_hot.copy_(_dev(oc.v_hot))
    return tc, oc, q, lens, cap


@pytest.mark.parametrize("vb", [4, 3])
@pytest.mark.parametrize("hq,hot,qscale", [(8, 0, 1.0), (16, 48, 2.5), (4, 300, 1.0)])
def test_asym_edges_against_the_oracle(vb, hq, hot, qscale):
    lens = [0, 1, 15, 16, 17, 33, 1000, 2100]
    tc, oc, q, lens, cap = _asym_pair(50 + hq + hot, lens, 4, hq, vb, hot, qscale)
    got = tc.decode(_dev(q), _dev(lens), cap).cpu().numpy()
    assert tc.device_status() == 0
    ref = oracle.decode_attention(oc, q, lens)
    assert np.all(got[0] == 0)
    assert_attention_close(got[1:], ref[1:], "asym V%d G=%d hot=%d" % (vb, hq // 4, hot))


def test_asym_sparse_v_within_the_oracle_bound():
    tc, oc, q, lens, cap = _asym_pair(57, [3000, 1777], 2, 8, 4, 64, 2.0)
    ql, sl = _dev(q), _dev(lens)
    ref = oracle.decode_attention(oc, q, lens)
    dense = tc.decode(ql, sl, cap).cpu().numpy()
    assert np.abs(dense - ref).max() <= ATTN_MAX_ABS
    for tau in (1e-4, 0.02):
        tc.desc.sparse_v_threshold = tau
        got = tc.decode(ql, sl, cap).cpu().numpy()
        bound = oracle.decode_sparse_v_bound(oc, q, lens, tau)
        excess = np.abs(got - ref) - bound
        assert np.all(np.isfinite(got))
        assert excess.max() <= ATTN_MAX_ABS, "tau %g: deviation beyond the sparse-V bound by %.3g" % (tau, excess.max())
    assert tc.device_status() == 0
