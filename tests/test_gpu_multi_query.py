"""GPU parity of multi-token attention (the newest n_query tokens of every
sequence, each causal over its own prefix) through the C ABI against the
oracle's multi_query_attention: outputs within 2e-3 max-abs and 1e-3
relative-L2, zeros for queries before position 0, and n_query = 1 bit-identical
to decode."""
import numpy as np
import pytest

import oracle
from bit_kv_cache_10_gb300 import native as N
from bit_kv_cache_10_gb300 import synth

from helpers import assert_attention_close

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


def _cache(**kw):
    from bit_kv_cache_10_gb300.cache import TurboQuantKVCache
    return TurboQuantKVCache(**kw)


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def upload(tc, oc):
    """Copy an oracle cache state into the device buffers of a cache."""
    if oc.k_fp16 is not None:
        tc.k_cache.copy_(_dev(oc.k_fp16))
    else:
        tc.k_cache.copy_(_dev(oc.k_words.view(np.int32)))
        tc.k_norms.copy_(_dev(oc.k_norms))
    tc.v_cache.copy_(_dev(oc.v_words.view(np.int32)))
    tc.v_norms.copy_(_dev(oc.v_norms))
    if oc.v_hot is not None:
        tc.v_hot.copy_(_dev(oc.v_hot))
    torch.cuda.synchronize()


def _queries(seed, B, NQ, HQ):
    return synth.queries_fp16(seed, B * NQ, HQ, D).reshape(B, NQ, HQ, D)


@pytest.mark.parametrize("bits,hq,hot,nq", [((3, 4), 32, 0, 4), ((4, 4), 8, 48, 7), ("int8", 16, 40, 3),
                                            ((0, 4), 8, 0, 2), ((2, 3), 16, 16, 16)])
def test_multi_query_matches_oracle(bits, hq, hot, nq):
    HK, CAP = 8, 1300
    lens = np.array([1300, 641, 33, 5, 0], np.int32)  # 5 < n_query for some: leading queries are empty
    B = len(lens)
    k = synth.kv_fp16(31, 1, B, HK, CAP, D, synth.channel_scales(31, 4, HK, D))
    v = synth.kv_fp16(31, 2, B, HK, CAP, D, synth.channel_scales(31, 5, HK, D))
    k_fp16 = bits == (0, 4)
    tc = _cache(batch=B, num_kv_heads=HK, num_q_heads=hq, capacity=CAP, bits=bits, hot_window=hot, k_fp16=k_fp16)
    tc.append(_dev(k), _dev(v), _dev(np.zeros(B, np.int32)), _dev(lens))
    assert tc.device_status() == 0
    if bits == "int8":
        oc = oracle.build_cache(k, v, lens, CAP, 8, 8, hot_window=hot, codec="int8")
    else:
        oc = oracle.build_cache(k, v, lens, CAP, 16 if k_fp16 else bits[0], bits[1], hot_window=hot, k_fp16=k_fp16)
        # decode parity is checked on the oracle's own cache (a counted code flip may differ)
        upload(tc, oc)
    q = _queries(31, B, nq, hq)
    got = tc.multi_query(_dev(q), _dev(lens), CAP).cpu().numpy()
    ref = oracle.multi_query_attention(oc, q, lens)
    for b in range(B):
        first = max(0, nq - int(lens[b]))  # queries before position 0
        assert np.all(got[b, :first] == 0)
        if first < nq:
            assert_attention_close(got[b, first:], ref[b, first:], "multi-query b=%d" % b)


def test_one_query_is_decode_bit_for_bit():
    B, HQ, HK, CAP = 3, 32, 8, 3000
    lens = np.array([3000, 1777, 16], np.int32)
    k = synth.kv_fp16(32, 1, B, HK, CAP, D, synth.channel_scales(32, 4, HK, D))
    v = synth.kv_fp16(32, 2, B, HK, CAP, D, synth.channel_scales(32, 5, HK, D))
    tc = _cache(batch=B, num_kv_heads=HK, num_q_heads=HQ, capacity=CAP, bits=3.5, hot_window=256)
    tc.append(_dev(k), _dev(v), _dev(np.zeros(B, np.int32)), _dev(lens))
    q = synth.queries_fp16(32, B, HQ, D)
    dec = tc.decode(_dev(q), _dev(lens), CAP).cpu().numpy()
    one = tc.multi_query(_dev(q[:, None]), _dev(lens), CAP).cpu().numpy()
    np.testing.assert_array_equal(one[:, 0], dec)


def test_speculative_verification_long_context_sampled():
    """Speculative-verification shape on the long-context cache: B4, 32 q / 8 KV
    heads, contexts in [64K, 128K], 256-token fp16 V window, 8 query tokens."""
    B, HQ, HK, CAP, W, NQ = 4, 32, 8, 131072, 256, 8
    lens = synth.seq_lengths(5, B, 65536, 131072)
    rk = synth.rng(33, synth.STREAM_CODES_K)
    rv = synth.rng(33, synth.STREAM_CODES_V)
    k_words = rk.integers(0, 2 ** 32, size=(B, HK, CAP, 12), dtype=np.uint32)
    v_words = rv.integers(0, 2 ** 32, size=(B, HK, CAP, 16), dtype=np.uint32)
    k_norms = synth.random_norms(33, synth.STREAM_NORMS_K, (B, HK, CAP), median=12.0)
    v_norms = synth.random_norms(33, synth.STREAM_NORMS_V, (B, HK, CAP), median=30.0)
    v_hot = synth.kv_fp16(33, synth.STREAM_V, B, HK, W, D, synth.channel_scales(33, synth.STREAM_SCALE_V, HK, D))
    oc = oracle.PackedCache(0, 0, D, 3, 4, k_words, k_norms, None, v_words, v_norms, W, v_hot)
    tc = _cache(batch=B, num_kv_heads=HK, num_q_heads=HQ, capacity=CAP, bits=3.5, hot_window=W)
    upload(tc, oc)
    q = _queries(33, B, NQ, HQ)
    got = tc.multi_query(_dev(q), _dev(lens), CAP).cpu().numpy()
    triples = [(0, 0, 0), (1, 7, 13), (2, 3, 22), (3, 5, 31), (3, 0, 4), (0, 7, 27)]
    ref = oracle.multi_query_attention(oc, q, lens, triples)
    idx = tuple(np.array(triples).T)
    assert_attention_close(got[idx], ref[idx], "speculative verification (sampled)")
    assert tc.device_status() == 0


def test_multi_query_paged_equals_contiguous_and_limits():
    B, HQ, HK, cap, bs, NQ = 2, 8, 2, 512, 32, 6
    lens = np.array([500, 200], np.int32)
    k = synth.kv_fp16(34, 1, B, HK, cap, D)
    v = synth.kv_fp16(34, 2, B, HK, cap, D)
    flat = _cache(batch=B, num_kv_heads=HK, num_q_heads=HQ, capacity=cap, bits=(4, 4), hot_window=24)
    paged = _cache(batch=B, num_kv_heads=HK, num_q_heads=HQ, capacity=cap, bits=(4, 4), hot_window=24,
                   block_size=bs, num_blocks=B * cap // bs + 3)
    perm = np.random.default_rng(4).permutation(B * cap // bs + 3)[:B * cap // bs].astype(np.int32)
    paged.block_table.copy_(_dev(perm.reshape(B, cap // bs)))
    for tc in (flat, paged):
        tc.append(_dev(k), _dev(v), _dev(np.zeros(B, np.int32)), _dev(lens))
    q = _dev(_queries(34, B, NQ, HQ))
    sl = _dev(lens)
    np.testing.assert_array_equal(paged.multi_query(q, sl, cap).cpu().numpy(), flat.multi_query(q, sl, cap).cpu().numpy())
    # B * n_query above 512 is refused before any launch
    big = _dev(np.zeros((B, 257, HQ, D), np.float16))
    with pytest.raises(N.TQError) as e:
        flat.multi_query(big, sl, cap)
    assert e.value.status == N.TQ_ERR_UNSUPPORTED


def test_multi_query_at_the_work_list_limit():
    """B x n_query = 512 work-list sequences (the limit), short ragged contexts."""
    B, HQ, HK, CAP, NQ = 64, 8, 2, 96, 8
    lens = np.random.default_rng(62).integers(0, CAP + 1, size=B).astype(np.int32)
    k = synth.kv_fp16(62, 1, B, HK, CAP, D)
    v = synth.kv_fp16(62, 2, B, HK, CAP, D)
    tc = _cache(batch=B, num_kv_heads=HK, num_q_heads=HQ, capacity=CAP, bits="int8")
    tc.append(_dev(k), _dev(v), _dev(np.zeros(B, np.int32)), _dev(lens))
    oc = oracle.build_cache(k, v, lens, CAP, 8, 8, codec="int8")
    q = _queries(62, B, NQ, HQ)
    got = tc.multi_query(_dev(q), _dev(lens), CAP).cpu().numpy()
    ref = oracle.multi_query_attention(oc, q, lens)
    for b in range(B):
        first = max(0, NQ - int(lens[b]))
        assert np.all(got[b, :first] == 0)
        if first < NQ:
            assert_attention_close(got[b, first:], ref[b, first:], "limit b=%d" % b)
