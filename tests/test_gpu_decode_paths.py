"""GPU parity of the two decode paths.

Small work runs one thread-block cluster per (sequence, KV head) row whose CTAs
merge their partials in distributed shared memory; everything else runs the
persistent split-K kernel and the merge kernel.  Each case is decoded through
both (forced with the library's test hook) on the oracle's own packed cache
and compared with the oracle (2e-3 max-abs, 1e-3 relative-L2): packed K of 2,
3 and 4 bits with V of 2, 3 and 4 bits, fp16 K, the int8 mode; ragged and
empty rows, rows shorter than a tile, CTAs of a cluster with no tile, hot
windows longer and shorter than the rows, group sizes 1, 2 and 4, peaked
softmax.
"""
import numpy as np
import pytest

import oracle
from bit_kv_cache_10_gb300 import native as N
from bit_kv_cache_10_gb300 import synth

from helpers import assert_attention_close

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

D = 128

# (batch lengths, KV heads, query heads, K bits (16: fp16 K, 8: int8 mode), V bits,
#  hot window, query scale)
CASES = {
    "llama_b1": ([4096], 8, 32, 3, 4, 0, 1.0),
    "ragged_empty": ([0, 1, 31, 33, 1024, 1025, 2100], 2, 8, 2, 4, 0, 1.0),
    "hot_g2": ([3, 8, 9, 64, 65, 300], 2, 4, 4, 4, 64, 1.0),
    "g1_hot256_peaked": ([700, 5000], 4, 4, 3, 4, 256, 2.5),
    "tiny_rows": ([5, 16, 17], 4, 16, 3, 4, 0, 2.5),
    "k3v3_b1": ([4096], 8, 32, 3, 3, 256, 1.0),
    "k2v2_ragged": ([0, 17, 600, 3000], 2, 8, 2, 2, 32, 2.0),
    "k4v3_g2": ([1, 2048], 4, 8, 4, 3, 0, 1.0),
    "asym_b1": ([4096], 8, 32, 16, 4, 0, 2.0),
    "asym_v3_hot": ([100, 1500], 2, 8, 16, 3, 64, 1.0),
    "int8_b1": ([4096], 8, 32, 8, 8, 0, 1.0),
    "int8_hot_ragged": ([0, 15, 700, 2049], 2, 4, 8, 8, 48, 2.0),
    # one or two long rows: the persistent kernel spreads each row over more than 32
    # CTAs, so the merge takes its general path (partials read in rounds of 32)
    "one_long_row_hot": ([20000], 1, 4, 3, 4, 256, 1.0),
    "two_long_rows_g1": ([9000, 12001], 1, 1, 4, 4, 0, 2.0),
    # a single short row: fewer price units of the weighted split than CTAs, so the
    # merge must skip candidate CTAs that took no tile of the row
    "one_short_row": ([40], 1, 4, 3, 4, 0, 1.0),
    "one_short_row_hot": ([40], 1, 4, 3, 4, 16, 1.0),
}


@pytest.fixture(scope="module", autouse=True)
def gpu_library():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from bit_kv_cache_10_gb300 import build
    build.build()
    N.lib()
    yield
    N.tq_debug_set_decode_path(0)


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.mark.parametrize("path", [1, 2])
@pytest.mark.parametrize("case", sorted(CASES))
def test_decode_path_against_the_oracle(case, path):
    from bit_kv_cache_10_gb300.cache import TurboQuantKVCache
    lens, hk, hq, kb, vb, hot, qscale = CASES[case]
    lens = np.asarray(lens, np.int32)
    B, cap = len(lens), int(lens.max())
    seed = 40 + sorted(CASES).index(case)
    k = synth.kv_fp16(seed, 1, B, hk, cap, D, synth.channel_scales(seed, 4, hk, D))
    v = synth.kv_fp16(seed, 2, B, hk, cap, D, synth.channel_scales(seed, 5, hk, D))
    q = (synth.queries_fp16(seed, B, hq, D).astype(np.float32) * qscale).astype(np.float16)
    if kb == 8:
        oc = oracle.build_cache(k, v, lens, cap, 8, 8, hot_window=hot, codec="int8")
        tc = TurboQuantKVCache(batch=B, num_kv_heads=hk, num_q_heads=hq, capacity=cap, bits="int8", hot_window=hot)
    else:
        oc = oracle.build_cache(k, v, lens, cap, kb, vb, hot_window=hot, k_fp16=kb == 16)
        tc = TurboQuantKVCache(batch=B, num_kv_heads=hk, num_q_heads=hq, capacity=cap,
                               bits=(4 if kb == 16 else kb, vb), hot_window=hot, k_fp16=kb == 16)
    if kb == 16:
        tc.k_cache.copy_(_dev(oc.k_fp16))
    else:
        tc.k_cache.copy_(_dev(oc.k_words.view(np.int32)))
        tc.k_norms.copy_(_dev(oc.k_norms))
    tc.v_cache.copy_(_dev(oc.v_words.view(np.int32)))
    tc.v_norms.copy_(_dev(oc.v_norms))
    if oc.v_hot is not None:
        tc.v_hot.copy_(_dev(oc.v_hot))
    N.tq_debug_set_decode_path(path)
    try:
        got = tc.decode(_dev(q), _dev(lens), cap).cpu().numpy()
    finally:
        N.tq_debug_set_decode_path(0)
    assert tc.device_status() == 0
    ref = oracle.decode_attention(oc, q, lens)
    assert np.all(got[lens == 0] == 0)
    keep = lens > 0
    assert_attention_close(got[keep], ref[keep], "%s path %d" % (case, path))
