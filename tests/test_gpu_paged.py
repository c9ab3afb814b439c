"""Paged (block-table) layout on the GPU.  The same appends into a contiguous
cache and into a paged cache whose blocks are scattered over a larger pool
must give bit-identical pools (read through the table), dequantized tokens and
decode outputs: the layout only changes where a row is stored.  A table entry
outside the pool raises TQ_DEV_ERR_BLOCK and is skipped."""
import numpy as np
import pytest

from bit_kv_cache_10_gb300 import synth
from bit_kv_cache_10_gb300 import native as N

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


def _pair(B, HK, HQ, cap, bs, hot, k_fp16, extra_blocks, seed):
    from bit_kv_cache_10_gb300.cache import TurboQuantKVCache
    mb = cap // bs
    kw = dict(bits=(3, 4), hot_window=hot, k_fp16=k_fp16)
    flat = TurboQuantKVCache(B, HK, HQ, cap, **kw)
    paged = TurboQuantKVCache(B, HK, HQ, cap, block_size=bs, num_blocks=B * mb + extra_blocks, **kw)
    perm = np.random.default_rng(seed).permutation(B * mb + extra_blocks)[:B * mb].astype(np.int32)
    paged.block_table.copy_(_dev(perm.reshape(B, mb)))
    return flat, paged, perm.reshape(B, mb)


def _append_both(caches, k, v, lens, n_pre, n_steps):
    """Ragged prefill of n_pre[b] tokens, then n_steps single-token appends."""
    B = k.shape[0]
    P = int(max(n_pre))
    for tc in caches:
        tc.append(_dev(k[:, :, :P]), _dev(v[:, :, :P]), _dev(np.zeros(B, np.int32)), _dev(np.asarray(n_pre, np.int32)))
    pos = np.asarray(n_pre, np.int32).copy()
    for _ in range(n_steps):
        kk = np.stack([k[b, :, pos[b]:pos[b] + 1] for b in range(B)])
        vv = np.stack([v[b, :, pos[b]:pos[b] + 1] for b in range(B)])
        for tc in caches:
            tc.append(_dev(kk), _dev(vv), _dev(pos))
        pos += 1
    return pos


@pytest.mark.parametrize("hot,k_fp16", [(0, False), (48, False), (40, True)])
def test_paged_equals_contiguous(hot, k_fp16):
    B, HQ, HK, cap, bs = 3, 8, 2, 1024, 64
    n_pre = np.array([990, 601, 70], np.int32)
    k = synth.kv_fp16(17, synth.STREAM_K, B, HK, cap, D, synth.channel_scales(17, synth.STREAM_SCALE_K, HK, D))
    v = synth.kv_fp16(17, synth.STREAM_V, B, HK, cap, D, synth.channel_scales(17, synth.STREAM_SCALE_V, HK, D))
    flat, paged, table = _pair(B, HK, HQ, cap, bs, hot, k_fp16, extra_blocks=7, seed=1)
    lens = _append_both((flat, paged), k, v, None, n_pre, n_steps=9)
    assert flat.device_status() == 0 and paged.device_status() == 0
    # pools read through the table equal the contiguous buffers
    for name in ("k_cache", "k_norms", "v_cache", "v_norms"):
        a, p = getattr(flat, name), getattr(paged, name)
        if a is None:
            continue
        a, p = a.cpu().numpy(), p.cpu().numpy()
        for b in range(B):
            t = np.arange(int(lens[b]))
            np.testing.assert_array_equal(p[table[b, t // bs], :, t % bs], a[b][:, t].swapaxes(0, 1), err_msg=name)
    if hot:
        np.testing.assert_array_equal(paged.v_hot.cpu().numpy(), flat.v_hot.cpu().numpy())
    # decode and dequantize
    q = _dev(synth.queries_fp16(17, B, HQ, D))
    sl = _dev(lens)
    # the paged layout always runs the persistent split kernel: the contiguous
    # decode it must equal bit for bit is taken through the same kernel
    N.tq_debug_set_decode_path(1)
    try:
        ref = flat.decode(q, sl, cap).cpu().numpy()
    finally:
        N.tq_debug_set_decode_path(0)
    np.testing.assert_array_equal(paged.decode(q, sl, cap).cpu().numpy(), ref)
    for which in (0, 1):
        for b in range(B):
            L = int(lens[b])
            np.testing.assert_array_equal(paged.dequantize(which, b, L, 0, L).cpu().numpy(),
                                          flat.dequantize(which, b, L, 0, L).cpu().numpy())


def test_block_outside_the_pool_is_flagged_and_skipped():
    B, HQ, HK, cap, bs = 2, 8, 2, 256, 32
    k = synth.kv_fp16(19, synth.STREAM_K, B, HK, cap, D)
    v = synth.kv_fp16(19, synth.STREAM_V, B, HK, cap, D)
    flat, paged, table = _pair(B, HK, HQ, cap, bs, 0, False, extra_blocks=0, seed=2)
    lens = _append_both((flat, paged), k, v, None, np.array([200, 150], np.int32), n_steps=0)
    assert paged.device_status() == 0
    bad = table.copy()
    bad[1, 2] = paged.num_blocks + 5  # positions 64..95 of sequence 1
    paged.block_table.copy_(_dev(bad))
    q = _dev(synth.queries_fp16(19, B, HQ, D))
    out = paged.decode(q, _dev(lens), cap).cpu().numpy()
    assert paged.device_status() & N.TQ_DEV_ERR_BLOCK
    assert np.all(np.isfinite(out))
    N.tq_debug_set_decode_path(1)  # the persistent split kernel, as for the paged layout
    try:
        ref = flat.decode(q, _dev(lens), cap).cpu().numpy()
    finally:
        N.tq_debug_set_decode_path(0)
    np.testing.assert_array_equal(out[0], ref[0])  # sequence 0 does not use the bad block


def _upload_paged(tc, oc, table, lens):
    """Write the oracle cache rows [0, L_b) of every sequence into the pools
    through the block table (row (block, h, t mod bs) of position t)."""
    bs = tc.block_size
    names = [("v_cache", oc.v_words.view(np.int32)), ("v_norms", oc.v_norms)]
    if oc.k_fp16 is not None:
        names.append(("k_cache", oc.k_fp16))
    else:
        names += [("k_cache", oc.k_words.view(np.int32)), ("k_norms", oc.k_norms)]
    for name, src in names:
        pool = getattr(tc, name).cpu().numpy()
        for b in range(len(lens)):
            t = np.arange(int(lens[b]))
            pool[table[b, t // bs], :, t % bs] = src[b][:, t].swapaxes(0, 1)
        getattr(tc, name).copy_(_dev(pool))
    if oc.v_hot is not None:
        tc.v_hot.copy_(_dev(oc.v_hot))
    torch.cuda.synchronize()


@pytest.mark.parametrize("kb,vb,hot,k_fp16", [(3, 4, 0, False), (3, 4, 48, False), (4, 4, 40, False),
                                              (2, 3, 0, False), (16, 4, 40, True)])
def test_paged_against_the_oracle(kb, vb, hot, k_fp16):
    """The paged layout against the oracle itself: words and norms of the pools
    (read through a scattered table) after ragged appends, then decode of every
    output and dequantize on the oracle's own cache written into the pools."""
    import oracle
    from helpers import assert_attention_close, assert_code_rate, compare_packed
    from bit_kv_cache_10_gb300.cache import TurboQuantKVCache
    B, HQ, HK, cap, bs = 3, 8, 2, 1024, 32
    n_pre = np.array([1000, 577, 45], np.int32)
    steps = 5
    k = synth.kv_fp16(23, synth.STREAM_K, B, HK, cap, D, synth.channel_scales(23, synth.STREAM_SCALE_K, HK, D))
    v = synth.kv_fp16(23, synth.STREAM_V, B, HK, cap, D, synth.channel_scales(23, synth.STREAM_SCALE_V, HK, D))
    mb = cap // bs
    nblk = B * mb + 11
    tc = TurboQuantKVCache(B, HK, HQ, cap, bits=(0 if k_fp16 else kb, vb), hot_window=hot, k_fp16=k_fp16,
                           block_size=bs, num_blocks=nblk)
    table = np.random.default_rng(29).permutation(nblk)[:B * mb].astype(np.int32).reshape(B, mb)
    tc.block_table.copy_(_dev(table))
    lens = _append_both((tc,), k, v, None, n_pre, n_steps=steps)
    assert tc.device_status() == 0
    oc = oracle.build_cache(k, v, lens, cap, 16 if k_fp16 else kb, vb, hot_window=hot, k_fp16=k_fp16)
    # stored words and norms, read through the table, against the oracle's quantizer
    mism, n_codes = 0, 0
    for which, bits, x in ((0, kb, k), (1, vb, v)):
        if which == 0 and k_fp16:
            pool = tc.k_cache.cpu().numpy()
            for b in range(B):
                t = np.arange(int(lens[b]))
                np.testing.assert_array_equal(pool[table[b, t // bs], :, t % bs], k[b][:, t].swapaxes(0, 1))
            continue
        words = (tc.k_cache if which == 0 else tc.v_cache).cpu().numpy().view(np.uint32)
        norms = (tc.k_norms if which == 0 else tc.v_norms).cpu().numpy()
        cb = oracle.codebook(D, bits)
        for b in range(B):
            L = int(lens[b]) if which == 0 else oracle.cold_end(int(lens[b]), hot)
            t = np.arange(L)
            for h in range(HK):
                codes, n, y = oracle.quantize_rows(x[b, h, :L], oracle.rotation(0, 0, h, D), cb)
                np.testing.assert_array_equal(norms[table[b, t // bs], h, t % bs], n)
                m, c = compare_packed(words[table[b, t // bs], h, t % bs], oracle.pack(codes, bits), y, bits,
                                      cb.thresholds32, "paged", check_rate=False)
                mism, n_codes = mism + m, n_codes + c
    assert_code_rate(mism, n_codes, "paged")
    if hot:
        np.testing.assert_array_equal(tc.v_hot.cpu().numpy(), oc.v_hot)
    # decode and dequantize on the oracle's cache in the pools
    _upload_paged(tc, oc, table, lens)
    q = synth.queries_fp16(23, B, HQ, D) * np.float16(2.5)  # peaked softmax
    got = tc.decode(_dev(q), _dev(lens), cap).cpu().numpy()
    assert_attention_close(got, oracle.decode_attention(oc, q, lens), "paged decode")
    for which in (0, 1):
        for b in range(B):
            L = int(lens[b])
            out = tc.dequantize(which, b, L, 0, L).cpu().numpy()
            for h in range(HK):
                ref = oracle.dequantized_kv(oc, b, h, L)[which]
                scale = np.maximum(np.linalg.norm(ref, axis=1, keepdims=True), 1e-30)
                assert np.all(np.abs(out[h] - ref) <= 1e-5 * scale), (which, b, h)
    assert tc.device_status() == 0
