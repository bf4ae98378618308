"""The bench's algorithmic byte model (host logic, no GPU): the index scan counts every valid
token of every distinct page once and every query's index query; the step adds each (sequence,
group)'s distinct selected valid tokens x 144 B plus per query token its Q and bf16 output.
Checked against counts made by hand on small workloads, shared pages included."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads as W  # noqa: E402


def test_index_bytes_counts_each_page_once():
    # 300 tokens (3 pages, last 44 valid), 129 (2 pages, last 1 valid); NVFP4 index: 72 B a token
    w = W.make("bytes", [300, 129], [2, 1], seed=5, identity=True)
    assert bench.index_bytes(w, 0) == (300 + 129) * 72 + 3 * 512
    f = W.make("bytes8", [300, 129], [2, 1], seed=5, identity=True, index_dtype=W.INDEX_FP8)
    assert bench.index_bytes(f, 0) == (300 + 129) * 128 + 3 * 512
    # a sequence with no query tokens is not scanned
    z = W.make("bytes0", [300, 129], [2, 0], seed=5, identity=True)
    assert bench.index_bytes(z, 0) == 300 * 72 + 2 * 512


def test_index_bytes_shared_prefix_pages():
    # two sequences share a 256-token (2-page) prefix: those pages are read once
    w = W.make("share", [256 + 10, 256 + 130], [1, 1], seed=6, prefix_len=256, prefix_seqs=2)
    assert w.block_table[0, 0] == w.block_table[1, 0] and w.block_table[0, 1] == w.block_table[1, 1]
    assert bench.index_bytes(w, 0) == (256 + 10 + 130) * 72 + 2 * 512


def test_step_bytes_distinct_selected_tokens():
    w = W.make("step", [300, 129], [2, 1], seed=7, identity=True)
    T = w.T
    sel = -np.ones((T, 4, 16), np.int32)
    # sequence 0 (tokens 0, 1): group 0 selects blocks {2, 0} and {2, 1}: distinct {0, 1, 2} =
    # 128 + 128 + 44 tokens; group 1 selects block 2 twice (44 tokens); groups 2, 3 nothing
    sel[0, 0, :2] = [2, 0]
    sel[1, 0, :2] = [2, 1]
    sel[0, 1, 0] = 2
    sel[1, 1, 0] = 2
    # sequence 1 (token 2): group 3 selects block 1 (1 valid token) and block 0
    sel[2, 3, :2] = [1, 0]
    kv = ((128 + 128 + 44) + 44 + (1 + 128)) * 144
    assert bench.step_bytes(w, 0, sel) == bench.index_bytes(w, 0) + kv + T * (8192 + 16384)


def test_recorded_traffic_follows_the_kernel_source(tmp_path, monkeypatch):
    """roofline.traffic is the committed DRAM count only while the kernel source it was taken
    from is unchanged (its hash), else None."""
    import hashlib
    import json

    (tmp_path / "profiles").mkdir()
    src = tmp_path / "k.cu"
    src.write_text("kernel v1\n")
    sha = hashlib.sha256(src.read_bytes()).hexdigest()[:16]
    (tmp_path / "profiles" / "traffic.json").write_text(
        json.dumps({"k@w": {"source_sha": sha, "bytes_per_launch": 1234}}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.recorded_traffic("k@w", "k.cu") == 1234
    assert bench.recorded_traffic("other", "k.cu") is None
    src.write_text("kernel v2\n")
    assert bench.recorded_traffic("k@w", "k.cu") is None


def test_clock_sampler_parses_a_fake_nvidia_smi(tmp_path, monkeypatch):
    """The bench's clock record from nvidia-smi's CSV lines: median SM clock, the maximum, every
    throttle reason seen Active, and the samples inside the timed loop's window (a fake
    nvidia-smi on PATH stands in for the real one)."""
    import time

    fake = tmp_path / "nvidia-smi"
    marker = tmp_path / "printed"
    fake.write_text("#!/bin/sh\n"
                    "echo '2026/12/02 10:00:00.100, 2070, 2070, 0x0, Not Active, Not Active, Not Active, Not Active'\n"
                    "echo '2026/12/02 10:00:00.200, 1980, 2070, 0x4, Not Active, Not Active, Not Active, Active'\n"
                    "echo '2026/12/02 10:00:00.300, 2010, 2070, 0x0, Not Active, Not Active, Not Active, Not Active'\n"
                    "echo 'garbage line'\n"
                    f"touch '{marker}'\n"
                    "exec sleep 30\n")
    fake.chmod(0o755)
    monkeypatch.setenv("PATH", str(tmp_path) + os.pathsep + os.environ.get("PATH", ""))
    c = bench.ClockSampler(0)
    t_end = time.time() + 20
    while not marker.exists() and time.time() < t_end:  # the fake has printed its lines
        time.sleep(0.01)
    assert marker.exists()
    t0 = time.mktime(time.strptime("2026/12/02 10:00:00", "%Y/%m/%d %H:%M:%S"))
    rec = c.stop((t0 + 0.15, t0 + 0.25))
    assert rec is not None
    assert rec["sm_mhz"] == 2010.0 and rec["sm_max_mhz"] == 2070.0
    assert rec["reasons"] == ["sw_power_cap"] and rec["samples"] == 3
    assert rec["timed_loop"]["samples"] == 1 and rec["timed_loop"]["sm_mhz"] == 1980.0
    assert rec["timed_loop"]["reasons"] == ["sw_power_cap"]


def test_clock_sampler_window_between_samples():
    """A timed loop shorter than the sampling period: the two samples around it stand for it."""
    import time

    t0 = time.mktime(time.strptime("2026/12/02 10:00:00", "%Y/%m/%d %H:%M:%S"))
    out = "\n".join(f"2026/12/02 10:00:00.{ms:03d}, {mhz}, 2070, 0x0, Not Active, Not Active, Not Active, Not Active"
                    for ms, mhz in ((100, 2070), (200, 1500), (300, 2000), (400, 1000)))
    s = bench.ClockSampler.parse(out)
    assert [x[1] for x in s] == [2070.0, 1500.0, 2000.0, 1000.0]
    assert abs(s[1][0] - (t0 + 0.2)) < 1e-6
