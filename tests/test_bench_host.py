"""Host logic of bench.py that its reported numbers rest on (no GPU).

* decode_bytes: the algorithmic bytes of a decode step (the roofline numerator),
  counted here from the stored record sizes of each layout;
* profile_traffic: the ncu traffic figure is reported only while the decode
  sources are the ones the committed capture was taken on;
* ClockSampler.summarize: median SM clock and the throttle reasons seen.
"""
import hashlib
import os
import shutil

import numpy as np

import bench


def test_decode_bytes_counts_every_stored_record():
    # one sequence shorter than the hot window, one longer, one empty
    lens = [100, 1000, 0]
    k_rec = 128 * 3 // 8 + 4   # 3-bit codes of 128 coordinates + float32 norm
    v_rec = 128 * 4 // 8 + 4   # 4-bit codes + norm, cold positions only
    hot_rec = 128 * 2          # fp16 V of the ring
    expect = 0
    for L in lens:
        hot = min(256, L)
        expect += 8 * (L * k_rec + (L - hot) * v_rec + hot * hot_rec)
    expect += len(lens) * 32 * 128 * (2 + 4)   # fp16 queries in, float32 outputs out
    assert bench.decode_bytes(lens) == expect
    # 52 + 68 = 120 bytes per cold token-head, the figure the roofline uses
    assert bench.decode_bytes([10000]) - bench.decode_bytes([9999]) == 8 * (k_rec + v_rec)


def _copy_tree(tmp_path):
    root = tmp_path / "repo"
    (root / "profiles").mkdir(parents=True)
    csrc = root / "bit_kv_cache_10_gb300" / "csrc"
    csrc.mkdir(parents=True)
    shutil.copy(os.path.join(bench.ROOT, "profiles", "decode_long_context.md"), root / "profiles")
    for f in bench.DECODE_SOURCES:
        shutil.copy(os.path.join(bench.ROOT, "bit_kv_cache_10_gb300", "csrc", f), csrc / f)
    return root


def test_traffic_follows_the_source_hash(tmp_path, monkeypatch):
    root = _copy_tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(root))
    text = (root / "profiles" / "decode_long_context.md").read_text()
    csrc = root / "bit_kv_cache_10_gb300" / "csrc"
    src = b"".join((csrc / f).read_bytes() for f in bench.DECODE_SOURCES)
    sha = hashlib.sha256(src).hexdigest()[:16]
    # a summary that names the current hash gives its traffic figure
    stamped = "traffic_bytes_per_step: 123456789\ndecode_source_sha256_16: %s\n" % sha
    (root / "profiles" / "decode_long_context.md").write_text(stamped + text)
    assert bench.profile_traffic() == 123456789
    # any edit of the kernel sources makes the figure stale: no traffic is reported
    with open(csrc / "tq_decode.cu", "ab") as fh:
        fh.write(b"\n")
    assert bench.profile_traffic() is None


def test_traffic_needs_a_summary(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profile_traffic() is None


def test_clock_summary():
    rows = [(2070.0, 2070.0, ["Not Active"] * 4), (1980.0, 2070.0, ["Not Active", "Not Active", "Not Active", "Active"]),
            (2070.0, 2070.0, ["Not Active"] * 4)]
    s = bench.ClockSampler.summarize(rows, "test")
    assert s["sm_mhz"] == float(np.median([2070.0, 1980.0, 2070.0]))
    assert s["sm_max_mhz"] == 2070.0 and s["samples"] == 3
    assert s["reasons"] == ["sw_power_cap"]
    assert bench.ClockSampler.summarize([], "none")["samples"] == 0
