"""Decode steps captured as a CUDA graph.

The library's calls only launch kernels on the caller's stream (no allocation,
no synchronisation, no host reads of device data), so a loop of appends and
decodes can be captured and replayed.  Two identical caches take the same
prefill and the same 12 one-token decode steps, one launched call by call and
one replayed from a graph captured over all 12 steps: the caches' words, norms
and rings and every step's output must be bit-identical, and the replay must
leave the status word clear.  Covered for the persistent split path (long rows)
and the cluster path (short rows), with a hot window.
"""
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


@pytest.mark.parametrize("lens", [[9000, 7000], [300, 2000]])
def test_graph_replay_equals_stream(lens):
    from bit_kv_cache_10_gb300.cache import TurboQuantKVCache
    B, HK, HQ, hot, steps = len(lens), 2, 8, 64, 12
    cap = max(lens) + steps + 16
    scales = synth.channel_scales(7, synth.STREAM_SCALE_K, HK, D)
    k = synth.kv_fp16(7, synth.STREAM_K, B, HK, cap, D, scales)
    v = synth.kv_fp16(7, synth.STREAM_V, B, HK, cap, D, scales)
    q = synth.queries_fp16(7, steps * B, HQ, D).reshape(steps, B, HQ, D)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    caches = [TurboQuantKVCache(B, HK, HQ, cap, bits=3.5, hot_window=hot) for _ in range(2)]
    n_pre = np.asarray(lens, np.int32)
    P = int(n_pre.max())
    for tc in caches:
        tc.append(dev(k[:, :, :P]), dev(v[:, :, :P]), dev(np.zeros(B, np.int32)), dev(n_pre))
    # per-step inputs on the device, fixed before the capture
    kk = [dev(np.stack([k[b, :, n_pre[b] + s:n_pre[b] + s + 1] for b in range(B)])) for s in range(steps)]
    vv = [dev(np.stack([v[b, :, n_pre[b] + s:n_pre[b] + s + 1] for b in range(B)])) for s in range(steps)]
    qq = [dev(q[s]) for s in range(steps)]
    starts = [dev(n_pre + s) for s in range(steps)]
    lens_s = [dev(n_pre + s + 1) for s in range(steps)]
    max_len = int(n_pre.max()) + steps
    outs = [[torch.empty(B, HQ, D, dtype=torch.float32, device="cuda") for _ in range(steps)] for _ in range(2)]
    wss = [torch.empty(tc.workspace_bytes(max_len), dtype=torch.uint8, device="cuda") for tc in caches]

    def run(i):
        for s in range(steps):
            caches[i].append(kk[s], vv[s], starts[s])
            caches[i].decode(qq[s], lens_s[s], max_len, out=outs[i][s], workspace=wss[i])

    run(0)  # call by call
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run(1)  # captured: nothing runs yet
    graph.replay()
    torch.cuda.synchronize()
    for tc in caches:
        assert tc.device_status() == 0
    for s in range(steps):
        assert torch.equal(outs[0][s], outs[1][s]), "step %d output" % s
    for name in ("k_cache", "k_norms", "v_cache", "v_norms", "v_hot"):
        assert torch.equal(getattr(caches[0], name), getattr(caches[1], name)), name


def test_stream_handle_follows_the_current_stream():
    """The binding launches on the caller's current stream: the handle it passes
    is torch's current stream of the cache's device, on a side stream too."""
    from bit_kv_cache_10_gb300.cache import _stream_handle
    dev = torch.device("cuda", torch.cuda.current_device())
    assert _stream_handle(dev) == torch.cuda.current_stream(dev).cuda_stream
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        assert _stream_handle(dev) == side.cuda_stream
    assert _stream_handle(dev) == torch.cuda.current_stream(dev).cuda_stream
