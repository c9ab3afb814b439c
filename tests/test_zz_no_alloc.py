"""Decode attention without a workspace argument, for callers that cannot
allocate device memory (plugin hosts that pass only inputs and outputs,
runtimes whose memory pool owns the GPU, serving loops that must not call
cudaMalloc).  tq_decode_attention_no_alloc keeps its split-K scratch in a
fixed device array of the library; its results must match the ordinary
entry point, call after call, since every call reuses that array.

This file is collected last so that a run stopping at the first failure has
run every other test before it; it also passes alone in a fresh process.
"""
import numpy as np
import pytest

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


def _random_cache(B, HK, HQ, cap, lens, hot, seed):
    from bit_kv_cache_10_gb300.cache import TurboQuantKVCache
    tc = TurboQuantKVCache(B, HK, HQ, cap, bits=(3, 4), hot_window=hot)
    for b in range(B):
        for h in range(HK):
            kw, kn = synth.packed_row(seed, synth.STREAM_CODES_K, b, h, int(lens[b]), 12, 12.0)
            vw, vn = synth.packed_row(seed, synth.STREAM_CODES_V, b, h, int(lens[b]), 16, 30.0)
            L = int(lens[b])
            tc.k_cache[b, h, :L].copy_(torch.from_numpy(kw.view(np.int32)))
            tc.k_norms[b, h, :L].copy_(torch.from_numpy(kn))
            tc.v_cache[b, h, :L].copy_(torch.from_numpy(vw.view(np.int32)))
            tc.v_norms[b, h, :L].copy_(torch.from_numpy(vn))
    if hot:
        tc.v_hot.copy_(torch.from_numpy(synth.kv_fp16(seed, synth.STREAM_V, B, HK, hot, D)))
    torch.cuda.synchronize()
    return tc


def _no_alloc(tc, q, lens, max_len):
    out = torch.full((tc.batch, tc.num_q_heads, D), float("nan"), dtype=torch.float32, device="cuda")
    N.tq_decode_attention_no_alloc(tc.desc, q.data_ptr(), lens.data_ptr(), max_len, out.data_ptr(),
                                   torch.cuda.current_stream().cuda_stream)
    return out


def test_no_alloc_decode_matches_workspace_decode_on_consecutive_calls():
    B, HK, HQ, CAP, HOT = 3, 8, 32, 40000, 256
    lens = np.array([39000, 12345, 700], np.int32)
    tc = _random_cache(B, HK, HQ, CAP, lens, HOT, seed=21)
    assert tc.workspace_bytes(CAP) <= N.TQ_NO_ALLOC_WORKSPACE_BYTES
    lens_d = torch.from_numpy(lens).cuda()
    for call in range(2):  # the second call finds the first call's partials in the scratch array
        q = torch.from_numpy(synth.queries_fp16(100 + call, B, HQ, D)).cuda()
        if call == 1:  # shorter sequences on the second call: fewer chunks than the first call wrote
            lens_d = torch.from_numpy(np.array([20000, 3000, 1], np.int32)).cuda()
        ref = tc.decode(q, lens_d, CAP).cpu().numpy()
        got = _no_alloc(tc, q, lens_d, CAP).cpu().numpy()
        assert_attention_close(got, ref, "no-alloc decode, call %d" % call)
    assert tc.device_status() == 0


def test_no_alloc_decode_rejects_requests_beyond_its_scratch():
    # 512 sequences x 8 KV heads need more partial slots than the fixed scratch holds: refused before any launch
    from bit_kv_cache_10_gb300.cache import TurboQuantKVCache
    B, HK, HQ, CAP = 512, 8, 32, 64
    tc = TurboQuantKVCache(B, HK, HQ, CAP, bits=(3, 4))  # real buffers of the request's sizes
    assert tc.workspace_bytes(CAP) > N.TQ_NO_ALLOC_WORKSPACE_BYTES
    q = torch.zeros(B, HQ, D, dtype=torch.float16, device="cuda")
    lens = torch.full((B,), CAP, dtype=torch.int32, device="cuda")
    out = torch.zeros(B, HQ, D, dtype=torch.float32, device="cuda")
    assert N.lib().tq_decode_attention_no_alloc(tc.desc, q.data_ptr(), lens.data_ptr(), CAP, out.data_ptr(),
                                                None) == N.TQ_ERR_WORKSPACE
