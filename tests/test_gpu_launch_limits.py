"""Launch setup done once per kernel and device.

The library raises a kernel's dynamic shared-memory limit on its first launch
and remembers it; the append kernel's shared memory grows with the code widths
(its threshold tables), so a later cache of wider codes needs more than the
first launch set.  That launch is refused, the limit raised, and the launch
repeated.  Each case runs in a fresh process, where no earlier launch has set
any limit: appends of 2-bit, then 4-bit, then 2-bit codes must store exactly
what a process that only appends the 4-bit (or the 2-bit) codes stores, with
the device status clear.
"""
import os
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r"""
import hashlib, sys
import numpy as np, torch
sys.path.insert(0, sys.argv[1])
from bit_kv_cache_10_gb300 import synth
from bit_kv_cache_10_gb300.cache import TurboQuantKVCache
B, HK, T, D = 2, 4, 200, 128
k = torch.from_numpy(synth.kv_fp16(11, synth.STREAM_K, B, HK, T, D)).cuda()
v = torch.from_numpy(synth.kv_fp16(11, synth.STREAM_V, B, HK, T, D)).cuda()
zero = torch.zeros(B, dtype=torch.int32, device="cuda")
for bits in [int(x) for x in sys.argv[2].split(",")]:
    tc = TurboQuantKVCache(B, HK, HK * 4, T, bits=(bits, bits))
    tc.append(k, v, zero)
    torch.cuda.synchronize()
    assert tc.device_status() == 0
    h = hashlib.sha1()
    for t in (tc.k_cache, tc.k_norms, tc.v_cache, tc.v_norms):
        h.update(t.contiguous().view(torch.uint8).cpu().numpy().tobytes())
    print(bits, h.hexdigest())
"""


def _run(widths):
    r = subprocess.run([sys.executable, "-c", SCRIPT, ROOT, widths], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    return [tuple(line.split()) for line in r.stdout.strip().splitlines()]


def test_wider_codes_after_narrower_in_one_process():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from bit_kv_cache_10_gb300 import build
    build.build()
    mixed = _run("2,4,2")
    alone4 = _run("4")
    alone2 = _run("2")
    assert [m[0] for m in mixed] == ["2", "4", "2"]
    assert mixed[1] == alone4[0]
    assert mixed[0] == alone2[0] and mixed[2] == alone2[0]
