#!/usr/bin/env python3
"""Benchmark of the MSA decode step over a paged NVFP4 cache (one layer-step per step).

Default workload: speculative decode, B=64 sequences of 131,072 tokens (1,024 blocks), 8 query
tokens each, hot blocks planted, random paging (the configuration the headline metric is
quoted on). One step = indexer -> top-k -> sparse attention -> merge over the whole batch
(msa_decode_step), inputs resident in HBM, L2 flushed by a 256 MB write between timed steps.

Prints one JSON line. `value` is microseconds per layer-step (lower is better, max over
ranks); the roofline object reports the dominant kernel (the stage with the longer time:
the sparse attention or the indexer) against the measured HBM peak, `roofline_stages` both;
`e2e` repeats the measurement through host buffers with msa_decode_step_host inside the
timed region (pinned H2D of the step's queries and metadata on two streams, q behind the
indexer, and the attention storing the output into the pinned host buffer);
`e2e.copy_back_us` is the same call with the output copied back on the copy stream instead, and
`e2e.serial_copies_us` the same copies issued one after another around msa_decode_step;
`cpu_baseline` times the oracle on a bounded sample on the host cores; `per_config` repeats the
measurement (fewer steps, stated in each entry) on every other configuration: tiny, decode,
long and the four layers of the ragged serving batch, each with its own sampled oracle time.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config spec] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import atexit
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "MSA decode µs/layer-step & achieved HBM TB/s (indexer+topk+attn), B=64 @128K"
L2_FLUSH_BYTES = 256 << 20


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def fp8_tensor_peak():
    """Dense E4M3 tensor peak (TFLOP/s) for a kernel timed alone: the measured bf16 burst figure
    x 2, the nominal FP8 / BF16 ratio (4.5 / 2.25 PFLOP/s)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        return 2.0 * float(json.load(open(p))["bf16_tflops"]), "measured bf16 burst x 2"
    return 2.0 * 1900.0, "fallback bf16 x 2"


def prefill_live_pairs(w: W.Workload) -> int:
    """(tile of 128 index-query rows, index page) pairs the prefill indexer scores with an MMA:
    the pages each tile's last token reaches."""
    qsl = w.query_start_loc()
    n = 0
    for b in range(w.B):
        L, ql = w.seq_lens[b], w.q_lens[b]
        if ql == 0:
            continue
        nb = (L + 127) // 128
        for i in range((4 * ql + 127) // 128):
            last = L - ql + min(ql - 1, (128 * (i + 1) - 1) // 4)
            n += min(nb, last // 128 + 1)
    return n


def index_bytes(w: W.Workload, layer: int) -> int:
    """Algorithmic bytes of the index scan: every valid token's index key once (shared pages
    once), plus the index queries."""
    per_tok = 72 if w.layers[layer].index_dtype == W.INDEX_NVFP4 else 128
    toks = 0
    seen = set()
    for b in range(w.B):
        if w.q_lens[b] == 0:
            continue
        L = w.seq_lens[b]
        for k in range((L + 127) // 128):
            pg = int(w.block_table[b, k])
            if pg in seen:
                continue
            seen.add(pg)
            toks += min(128, L - 128 * k)
    return toks * per_tok + w.T * 512


def step_bytes(w: W.Workload, layer: int, sel: np.ndarray) -> int:
    """Algorithmic bytes of one layer-step: the index scan, each (sequence, group)'s distinct
    selected valid tokens x 144 B (K and V codes + scales), and per query token its Q (8,192
    B), index query (512 B, counted in index_bytes) and bf16 output (16,384 B)."""
    qsl = w.query_start_loc()
    kv = 0
    for b in range(w.B):
        ql, L = w.q_lens[b], w.seq_lens[b]
        if ql == 0:
            continue
        for g in range(4):
            blocks = set(int(x) for x in sel[qsl[b]:qsl[b] + ql, g].ravel() if x >= 0)
            kv += sum(min(128, L - 128 * k) for k in blocks if 128 * k < L) * 144
    return index_bytes(w, layer) + kv + w.T * (8192 + 16384)


class ClockSampler:
    """nvidia-smi clock and throttle-reason samples every 100 ms, each stamped with the time
    nvidia-smi took it; `stop(window)` summarises every sample and, separately, those inside
    the given (start, end) host-clock window (the timed loop, which can be shorter than one
    sampling period: the samples nearest to it are then the ones reported for it)."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, index: int):
        self.proc = None
        self.index = index
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(index), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
        if self.proc is not None:
            atexit.register(self._end)  # an exception before stop() must not leave it running

    def _end(self):
        if self.proc is not None and self.proc.poll() is None:
            self.proc.kill()
            self.proc.wait()

    @staticmethod
    def _stamp(text: str):
        """nvidia-smi's local-time stamp ("2026/12/02 13:25:00.123") as epoch seconds."""
        try:
            return time.mktime(time.strptime(text.split(".")[0], "%Y/%m/%d %H:%M:%S")) + (
                float("0." + text.split(".")[1]) if "." in text else 0.0)
        except (ValueError, IndexError):
            return None

    @classmethod
    def summarise(cls, samples):
        if not samples:
            return None
        reasons = sorted({n for s in samples for n in s[3]})
        return {"sm_mhz": statistics.median(s[1] for s in samples), "sm_max_mhz": max(s[2] for s in samples),
                "reasons": reasons, "samples": len(samples)}

    @classmethod
    def parse(cls, out: str):
        """(stamp or None, sm MHz, max MHz, active reasons) per well-formed line."""
        samples = []
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 8:
                continue
            try:
                sm, mx = float(f[1]), float(f[2])
            except ValueError:
                continue
            act = {n for n, v in zip(cls.REASONS, f[4:8]) if v.lower() == "active"}
            samples.append((cls._stamp(f[0]), sm, mx, act))
        return samples

    def stop(self, window=None):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        samples = self.parse(out)
        rec = self.summarise(samples)
        if rec is None or window is None:
            return rec
        t0, t1 = window
        stamped = [s for s in samples if s[0] is not None]
        inside = [s for s in stamped if t0 <= s[0] <= t1]
        if not inside and stamped:  # the loop fell between two samples: the two around it
            before = [s for s in stamped if s[0] < t0]
            after = [s for s in stamped if s[0] > t1]
            inside = before[-1:] + after[:1]
        rec["timed_loop"] = self.summarise(inside)
        if rec["timed_loop"] is not None:
            rec["timed_loop"]["loop_s"] = t1 - t0
        return rec


def recorded_traffic(kernel: str, source: str):
    """Per-launch DRAM bytes of `kernel` from the committed ncu summary, or None when the
    kernel source changed since the capture."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(kernel)
    if not d:
        return None
    h = hashlib.sha256(open(os.path.join(ROOT, source), "rb").read()).hexdigest()[:16]
    return d.get("bytes_per_launch") if d.get("source_sha") == h else None


# ---------------------------------------------------------------------------- oracle leg
def oracle_sample(w: W.Workload, layer: int, b: int, device: str):
    """Time the oracle (indexer + selection + attention) on sequence b; the inputs are
    quantised outside the timed region (the caches are resident state)."""
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import oracle
    from parity import OracleSeq

    oracle.build()
    ref = OracleSeq(w, layer, b, device, kv_blocks=None)
    t0 = time.perf_counter()
    s = ref.scores()
    sel = oracle.select_seq(s, ref.L, ref.q_len)
    ref.attention(sel, 1.0 / math.sqrt(128))
    dt = time.perf_counter() - t0
    return dt, oracle.hardware_threads()


def run_reference(args, w: W.Workload, rank: int):
    if rank != 0:
        return
    device = "cuda" if _cuda_ok() else "cpu"
    active = [b for b in range(w.B) if w.q_lens[b] > 0]
    times = []
    cores = 0
    for i in range(args.warmup + args.steps):
        b = active[i % len(active)]
        dt, cores = oracle_sample(w, 0, b, device)
        if i >= args.warmup:
            times.append(dt)
    per_step_s = statistics.mean(times) * len(active)
    v = per_step_s * 1e6
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "us/layer-step", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": v / 1e3, "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "seq_len": max(w.seq_lens), "q_len": max(w.q_lens),
                       "parallelism": "host cores"},
            "cpu_baseline": {"value": v, "unit": "us/layer-step", "cores": cores, "kind": "oracle",
                             "sample": f"each step: one of {len(active)} sequences (all its query tokens, 4 groups,"
                                       f" 64 heads), oracle wall time x {len(active)}"},
            "e2e": {"value": v, "unit": "us/layer-step", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def _cuda_ok():
    try:
        import torch

        return torch.cuda.is_available()
    except Exception:
        return False


# ---------------------------------------------------------------------------- GPU leg
def max_over_ranks(value: float, world: int, device) -> float:
    """The job's time: the slowest rank's (every rank runs its own replica of the batch)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def prefill_selection(w: W.Workload, seed: int) -> np.ndarray:
    """Valid selections [T, 4, 16] shaped like top-16 picks: the token's local block, then 15
    distinct earlier blocks drawn uniformly (a prefill batch has no decode indexer to rank them)."""
    rng = np.random.default_rng(seed)
    qsl = w.query_start_loc()
    sel = np.full((w.T, 4, 16), -1, dtype=np.int32)
    for b in range(w.B):
        L, ql = w.seq_lens[b], w.q_lens[b]
        for i in range(ql):
            local = (L - ql + i) // 128
            k = min(15, local)
            for g in range(4):
                sel[qsl[b] + i, g, 0] = local
                if k:
                    sel[qsl[b] + i, g, 1:1 + k] = rng.choice(local, size=k, replace=False)
    return sel


def time_prefill(msa, steps: int, warmup: int, flush, dev):
    """The block-major prefill attention on one 2,048-token prompt chunk at 16K context."""
    import torch

    from workloads.device import DeviceLayer

    wp = W.make("prefill B=1 L=16384 q_len=2048", [16384], [2048], seed=5)
    dlp = DeviceLayer(wp, 0, device=dev)
    sel_np = prefill_selection(wp, 5)
    sel = torch.from_numpy(sel_np).to(dev)
    out = torch.empty((wp.T, 64, 128), dtype=torch.uint16, device=dev)
    wsp = torch.empty(msa.msa_prefill_workspace_size(wp.B, wp.T, dlp.batch.max_blocks), dtype=torch.uint8, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    for _ in range(warmup):
        msa.msa_prefill_attn(dlp.batch, dlp.cache, dlp.q8, sel, dlp.softmax_scale, out, wsp, st)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for i in range(steps):
        flush.fill_(i & 0xFF)
        ev[i][0].record()
        msa.msa_prefill_attn(dlp.batch, dlp.cache, dlp.q8, sel, dlp.softmax_scale, out, wsp, st)
        ev[i][1].record()
    torch.cuda.synchronize()
    assert msa.status_bits(st) == 0
    us = statistics.mean(a.elapsed_time(b) for a, b in ev) * 1e3
    rows, chunks, entries, _ = wsp[:16].view(torch.int32).cpu().tolist()
    # algorithmic bytes: each (page, group) block's K and V once, the query heads once, the
    # per-selection partials written and read back (4 KB of f16 o + 128 B of (m, l)), the output
    partial = entries * (4096 + 128)
    algo = rows * 18432 + wp.T * 64 * 128 + 2 * partial + wp.T * 64 * 128 * 2
    return {"workload": wp.name, "us_per_call": us, "tokens_per_s": wp.T / us * 1e6,
            "distinct_blocks_read": rows, "kv_dequantisations": chunks, "selections_served": entries,
            "kv_bytes_algorithmic": rows * 18432, "bytes_algorithmic": algo,
            f"hbm_frac_of_{peaks()[1]}": algo / (us * 1e-6) / 1e9 / peaks()[0],
            "selections": "local block + 15 distinct earlier blocks drawn uniformly per (token, group)"}


def time_prefill_path(msa, steps: int, warmup: int, flush, dev):
    """The whole prefill path on the same 2,048-token prompt chunk at 16K context: the prefill
    indexer, the selection and the block-major attention on the selection the indexer makes,
    each stage timed with events between the calls."""
    import torch

    from workloads.device import DeviceLayer

    wp = W.make("prefill B=1 L=16384 q_len=2048", [16384], [2048], seed=5)
    dlp = DeviceLayer(wp, 0, device=dev)
    maxb = dlp.batch.max_blocks
    scores = torch.empty((wp.T, 4, maxb), dtype=torch.float32, device=dev)
    sel = torch.empty((wp.T, 4, 16), dtype=torch.int32, device=dev)
    out = torch.empty((wp.T, 64, 128), dtype=torch.uint16, device=dev)
    wsp = torch.empty(msa.msa_prefill_workspace_size(wp.B, wp.T, maxb), dtype=torch.uint8, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)

    def run(ev=None):
        if ev:
            ev[0].record()
        msa.msa_indexer_prefill(dlp.batch, dlp.cache, dlp.iq8, scores, st)
        if ev:
            ev[1].record()
        msa.msa_topk_prefill(dlp.batch, scores, sel, st)
        if ev:
            ev[2].record()
        msa.msa_prefill_attn(dlp.batch, dlp.cache, dlp.q8, sel, dlp.softmax_scale, out, wsp, st)
        if ev:
            ev[3].record()

    for _ in range(warmup):
        run()
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    for i in range(steps):
        flush.fill_(i & 0xFF)
        run(evs[i])
    torch.cuda.synchronize()
    assert msa.status_bits(st) == 0
    stage = [statistics.mean(e[j].elapsed_time(e[j + 1]) for e in evs) * 1e3 for j in range(3)]
    total = statistics.mean(e[0].elapsed_time(e[3]) for e in evs) * 1e3
    rows, chunks, entries, _ = wsp[:16].view(torch.int32).cpu().tolist()
    pairs = prefill_live_pairs(wp)
    flops = pairs * 2 * 128 * 128 * 128
    peak, kind = fp8_tensor_peak()
    tflops = flops / (stage[0] * 1e-6) / 1e12
    nb = (wp.seq_lens[0] + 127) // 128
    idx_bytes = nb * 9216 + wp.T * 512 + wp.T * 4 * nb * 4  # pages once, index queries, scores
    return {"workload": wp.name, "us_per_call": total, "tokens_per_s": wp.T / total * 1e6,
            "stages_us": {"indexer": stage[0], "topk": stage[1], "attention": stage[2]},
            "indexer_roofline": {"kernel": "k_indexer_prefill (msa_indexer_prefill)", "bound": "tensor",
                                 "achieved": tflops, "peak": peak, "unit": "TFLOP/s", "frac": tflops / peak,
                                 "peak_kind": kind, "mma_pairs": pairs, "flops": flops,
                                 "algorithmic_bytes": idx_bytes},
            "attention_distinct_blocks_read": rows, "attention_kv_dequantisations": chunks,
            "attention_selections_served": entries,
            "selections": "the prefill indexer's own (msa_topk_prefill of its scores)"}


PER_CONFIG_STEPS, PER_CONFIG_WARMUP = 8, 3


def measure_config(msa, w: W.Workload, layer: int, flush, dev, with_cpu: bool):
    """One configuration (one layer of it) the way the headline is measured, with fewer steps:
    the fused step's µs (L2 flushed before each step), the three stages timed one by one,
    algorithmic bytes from the step's own selection, and the oracle on one sequence x B."""
    import torch

    from workloads.device import DeviceLayer

    dl = DeviceLayer(w, layer, device=dev)
    o = dl.outputs()
    ws = dl.workspace()
    stream = torch.cuda.current_stream()

    def step():
        msa.msa_decode_step(dl.batch, dl.cache, dl.q8, dl.iq8, dl.softmax_scale, ws, o["out"], o["scores"], o["sel"])

    for _ in range(PER_CONFIG_WARMUP):
        step()
    torch.cuda.synchronize()
    if msa.msa_read_device_status(ws) != msa.MSA_OK:
        raise RuntimeError(f"{w.name} layer {layer}: device status not OK")
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(PER_CONFIG_STEPS)]
    for i in range(PER_CONFIG_STEPS):
        flush.fill_(i & 0xFF)
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    step_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    sel = o["sel"].cpu().numpy()
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    aws = torch.empty(max(msa.msa_attn_workspace_size(w.B, w.T, 0), 256), dtype=torch.uint8, device=dev)
    st_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(PER_CONFIG_STEPS)]
    for i in range(PER_CONFIG_STEPS):
        flush.fill_(i & 0xFF)
        e = st_ev[i]
        e[0].record(stream)
        msa.msa_indexer_decode(dl.batch, dl.cache, dl.iq8, o["scores"], status)
        e[1].record(stream)
        msa.msa_topk_blocks(dl.batch, o["scores"], o["sel"], status)
        e[2].record(stream)
        msa.msa_sparse_attn_decode(dl.batch, dl.cache, dl.q8, o["sel"], dl.softmax_scale, o["out"], 0, aws, status)
        e[3].record(stream)
    torch.cuda.synchronize()
    if msa.status_bits(status) != 0:
        raise RuntimeError(f"{w.name} layer {layer}: stage status not OK")
    stage_ms = [statistics.mean(st_ev[i][j].elapsed_time(st_ev[i][j + 1]) for i in range(PER_CONFIG_STEPS))
                for j in range(3)]
    peak_gbs, peak_kind = peaks()
    idx_bytes = index_bytes(w, layer)
    total = step_bytes(w, layer, sel)
    attn_bytes = total - idx_bytes
    stage_frac = {"indexer": idx_bytes / (stage_ms[0] * 1e-3) / 1e9 / peak_gbs,
                  "attention": attn_bytes / (stage_ms[2] * 1e-3) / 1e9 / peak_gbs}
    dominant = "attention" if stage_ms[2] >= stage_ms[0] else "indexer"
    rec = {"workload": w.name, "layer": layer,
           "index_dtype": "nvfp4" if w.layers[layer].index_dtype == W.INDEX_NVFP4 else "fp8",
           "B": w.B, "T": w.T, "steps": PER_CONFIG_STEPS, "warmup": PER_CONFIG_WARMUP,
           "us_per_layer_step": step_ms * 1e3,
           "stages_us": {"indexer": stage_ms[0] * 1e3, "topk": stage_ms[1] * 1e3, "attention": stage_ms[2] * 1e3},
           "step_bytes": total, "achieved_tbps": total / (step_ms * 1e-3) / 1e12,
           "step_frac_of_hbm_peak": total / (step_ms * 1e-3) / 1e9 / peak_gbs,
           "stage_frac_of_hbm_peak": stage_frac, "dominant_stage": dominant,
           "dominant_frac": stage_frac[dominant], "peak_kind": f"{peak_kind} hbm_gbs"}
    if with_cpu:
        active = [b for b in range(w.B) if w.q_lens[b] > 0]
        b0 = active[0]
        dt, cores = oracle_sample(w, layer, b0, dev)
        rec["cpu_baseline"] = {"value": dt * len(active) * 1e6, "unit": "us/layer-step", "cores": cores,
                               "kind": "oracle",
                               "sample": f"sequence {b0} ({w.seq_lens[b0]} tokens, {w.q_lens[b0]} query tokens, 4 "
                                         f"groups, 64 heads): oracle indexer+selection+attention wall time x "
                                         f"{len(active)}"}
    del dl, o, ws, aws
    torch.cuda.empty_cache()
    return rec


def per_config_lines(msa, flush, dev, with_cpu: bool):
    """Every configuration besides the headline one: tiny, decode, long and the four ragged layers."""
    out = []
    for name in ("tiny", "decode", "long"):
        out.append(measure_config(msa, W.CONFIGS[name](), 0, flush, dev, with_cpu))
    rw = W.CONFIGS["ragged"]()
    for layer in range(len(rw.layers)):
        out.append(measure_config(msa, rw, layer, flush, dev, with_cpu))
    return out


def run_ours(args, w: W.Workload, rank: int, world: int, local_rank: int):
    import torch
    import torch.distributed as dist

    import nvfp4_kv_cache_gb300 as msa
    from workloads.device import DeviceLayer

    torch.cuda.set_device(local_rank)
    dev = f"cuda:{local_rank}"
    dl = DeviceLayer(w, 0, device=dev)
    o = dl.outputs()
    ws = dl.workspace()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    B, T = w.B, w.T

    def step():
        msa.msa_decode_step(dl.batch, dl.cache, dl.q8, dl.iq8, dl.softmax_scale, ws, o["out"])

    def barrier():
        if world > 1:
            dist.barrier()

    # ---- warm-up
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if msa.msa_read_device_status(ws) != msa.MSA_OK:
        raise RuntimeError("device status not OK after warm-up")

    # ---- headline: K timed steps of the fused call, L2 flushed between them
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    clocks = ClockSampler(local_rank) if rank == 0 else None
    barrier()
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    t_epoch = time.time()
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    barrier()
    wall = time.perf_counter() - t_wall
    step_ms = [a.elapsed_time(b) for a, b in ev]
    ms_max = max_over_ranks(statistics.mean(step_ms), world, dev)

    # ---- per-stage breakdown: the same three calls with events between them
    o2 = dl.outputs()
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    aws_n = msa.msa_attn_workspace_size(B, T, 0)
    aws = torch.empty(max(aws_n, 256), dtype=torch.uint8, device=dev)
    st_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        e = st_ev[i]
        e[0].record(stream)
        msa.msa_indexer_decode(dl.batch, dl.cache, dl.iq8, o2["scores"], status)
        e[1].record(stream)
        msa.msa_topk_blocks(dl.batch, o2["scores"], o2["sel"], status)
        e[2].record(stream)
        msa.msa_sparse_attn_decode(dl.batch, dl.cache, dl.q8, o2["sel"], dl.softmax_scale, o2["out"], 0, aws, status)
        e[3].record(stream)
    torch.cuda.synchronize()
    stage_ms = [statistics.mean(st_ev[i][j].elapsed_time(st_ev[i][j + 1]) for i in range(args.steps))
                for j in range(3)]
    assert msa.status_bits(status) == 0
    sel = o2["sel"].cpu().numpy()

    # ---- the exact-score indexer variant (NVFP4 keys scored exactly), timed alone the same way
    exact_ms = None
    if w.layers[0].index_dtype == W.INDEX_NVFP4:
        ex = torch.empty_like(o2["scores"])
        ex_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        for i in range(args.steps):
            flush.fill_(i & 0xFF)
            ex_ev[i][0].record(stream)
            msa.msa_indexer_decode_exact(dl.batch, dl.cache, dl.iq8, ex, status)
            ex_ev[i][1].record(stream)
        torch.cuda.synchronize()
        exact_ms = statistics.mean(a.elapsed_time(b) for a, b in ex_ev)
        assert msa.status_bits(status) == 0

    # ---- the prefill (many-query) attention path, rank 0 alone, on its own synthetic prompt
    prefill = time_prefill(msa, args.steps, args.warmup, flush, dev) if rank == 0 and args.config == "spec" else None
    prefill_path = (time_prefill_path(msa, args.steps, args.warmup, flush, dev)
                    if rank == 0 and args.config == "spec" else None)

    # ---- end to end through host buffers: the library's host-buffer step (pinned H2D of the
    # step's inputs and D2H of its output on a copy stream, overlapped with the kernels), and
    # for comparison the same copies issued one after another around msa_decode_step
    q_h = dl.q8.cpu().pin_memory()
    iq_h = dl.iq8.cpu().pin_memory()
    meta = [dl.batch.query_start_loc, dl.batch.seq_lens, dl.batch.block_table]
    meta_h = [m.cpu().pin_memory() for m in meta]
    out_h = torch.empty(o["out"].shape, dtype=o["out"].dtype).pin_memory()
    h2d = q_h.numel() + iq_h.numel() + sum(m.numel() * m.element_size() for m in meta_h)
    d2h = out_h.numel() * out_h.element_size()
    copy_stream = torch.cuda.Stream()

    def host_step():
        msa.msa_decode_step_host(dl.batch, dl.cache, meta_h[0], meta_h[1], meta_h[2], q_h, iq_h, out_h, dl.q8, dl.iq8,
                                 dl.softmax_scale, ws, None, copy_stream, direct_out=True)

    def host_step_copy_back():
        msa.msa_decode_step_host(dl.batch, dl.cache, meta_h[0], meta_h[1], meta_h[2], q_h, iq_h, out_h, dl.q8, dl.iq8,
                                 dl.softmax_scale, ws, o["out"], copy_stream)

    def serial_step():
        dl.q8.copy_(q_h, non_blocking=True)
        dl.iq8.copy_(iq_h, non_blocking=True)
        for m, mh in zip(meta, meta_h):
            m.copy_(mh, non_blocking=True)
        step()
        out_h.copy_(o["out"], non_blocking=True)

    def time_e2e(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        barrier()
        torch.cuda.synchronize()
        for i in range(args.steps):
            flush.fill_(i & 0xFF)
            evs[i][0].record(stream)
            fn()
            evs[i][1].record(stream)
            evs[i][1].synchronize()
        barrier()
        return max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in evs), world, dev)

    e2e_ms = time_e2e(host_step)
    if msa.msa_read_device_status(ws) != msa.MSA_OK:
        raise RuntimeError("device status not OK after the host-buffer steps")
    e2e_copy_back_ms = time_e2e(host_step_copy_back)
    e2e_serial_ms = time_e2e(serial_step)

    # every other configuration, one line each (rank 0, one GPU, the default headline run only)
    per_config = None
    if rank == 0 and world == 1 and args.config == "spec" and not args.no_per_config:
        del q_h, iq_h, meta_h, out_h
        per_config = per_config_lines(msa, flush, dev, not args.no_cpu_baseline)

    # clocks sampled from the start of the timed loop through the stage, exact-indexer, prefill and
    # end-to-end loops that follow it (the timed loop alone is shorter than the sampling period)
    clk = clocks.stop((t_epoch, t_epoch + wall)) if clocks else None
    if clk is not None:
        clk["window"] = ("all samples: the timed loop through the end-to-end loops; timed_loop: the samples "
                         "inside the timed loop, or the two around it when it fell between samples")
    if rank != 0:
        return
    peak_gbs, peak_kind = peaks()
    idx_bytes = index_bytes(w, 0)
    total_bytes = step_bytes(w, 0, sel)
    idx_gbs = idx_bytes / (stage_ms[0] * 1e-3) / 1e9
    attn_bytes = total_bytes - idx_bytes  # distinct selected K/V + Q + output
    attn_gbs = attn_bytes / (stage_ms[2] * 1e-3) / 1e9
    attn_kernel = "tc::k_attn_tc" if 4 * T > 2 * 152 else "k_attn"
    roof = {
        "indexer": {"kernel": "k_indexer (msa_indexer_decode)", "bound": "hbm", "achieved": idx_gbs,
                    "peak": peak_gbs, "unit": "GB/s", "frac": idx_gbs / peak_gbs,
                    "peak_kind": f"{peak_kind} hbm_gbs", "algorithmic_bytes": idx_bytes,
                    "launch_us": stage_ms[0] * 1e3,
                    "traffic": recorded_traffic("k_indexer", "nvfp4_kv_cache_gb300/csrc/msa_indexer.cu")},
        "attention": {"kernel": f"{attn_kernel} (msa_sparse_attn_decode)", "bound": "hbm", "achieved": attn_gbs,
                      "peak": peak_gbs, "unit": "GB/s", "frac": attn_gbs / peak_gbs,
                      "peak_kind": f"{peak_kind} hbm_gbs", "algorithmic_bytes": attn_bytes,
                      "launch_us": stage_ms[2] * 1e3,
                      "traffic": recorded_traffic(attn_kernel + "@" + w.name, "nvfp4_kv_cache_gb300/csrc/msa_attn.cu")},
    }
    dominant = "attention" if stage_ms[2] >= stage_ms[0] else "indexer"
    launches_per_step = 3 + (1 if aws_n > 0 else 0)
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        dt, cores = oracle_sample(w, 0, 0, dev)
        active = sum(1 for q in w.q_lens if q > 0)
        cpu = {"value": dt * active * 1e6, "unit": "us/layer-step", "cores": cores, "kind": "oracle",
               "sample": f"sequence 0 of {active} (all {w.q_lens[0]} query tokens, 4 groups, 64 heads): oracle "
                         f"indexer+selection+attention wall time x {active}"}
    line = {
        "metric": METRIC, "value": ms_max * 1e3, "unit": "us/layer-step", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3 MMA, fp32 accumulate/softmax, e4m3 PV (P as hi + lo E4M3 parts)", "data": "synthetic",
        "config": {"workload": w.name, "B": B, "seq_len": max(w.seq_lens), "q_len": max(w.q_lens), "T": T,
                   "index_dtype": "nvfp4" if w.layers[0].index_dtype == 0 else "fp8", "layers": 1,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "flushed by a 256 MB write before every timed step"},
        "achieved_tbps": total_bytes / (ms_max * 1e-3) / 1e12,
        "step_bytes": total_bytes, "step_frac_of_hbm_peak": total_bytes / (ms_max * 1e-3) / 1e9 / peak_gbs,
        "stages_us": {"indexer": stage_ms[0] * 1e3, "topk": stage_ms[1] * 1e3, "attention": stage_ms[2] * 1e3},
        "indexer_exact_us": None if exact_ms is None else exact_ms * 1e3,
        "prefill_attn": prefill,
        "prefill_path": prefill_path,
        "roofline": roof[dominant],
        "roofline_stages": roof,
        "e2e": {"value": e2e_ms * 1e3, "unit": "us/layer-step", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h),
                "api": "msa_decode_step_host, MSA_HOST_STEP_DIRECT_OUT: input copies on two streams, q behind "
                       "the indexer, the attention storing the bf16 output into the pinned host buffer",
                "copy_back_us": e2e_copy_back_ms * 1e3, "serial_copies_us": e2e_serial_ms * 1e3},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
        "cpu_baseline": cpu,
        "per_config": per_config,
        "wall_s_timed_region": wall,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="spec", choices=sorted(W.CONFIGS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true", help="skip the lines of the other configurations")
    ap.add_argument("--prefill-only", action="store_true",
                    help="time the prefill attention (its 2,048-token prompt) and the prefill path "
                         "(indexer, selection, attention) and print their records")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.prefill_only:
        import torch

        import nvfp4_kv_cache_gb300 as msa

        dev = torch.device("cuda", local_rank)
        torch.cuda.set_device(dev)
        flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        print(json.dumps({"prefill_attn": time_prefill(msa, args.steps, args.warmup, flush, dev),
                          "prefill_path": time_prefill_path(msa, args.steps, args.warmup, flush, dev)}), flush=True)
        return
    w = W.CONFIGS[args.config]()
    if args.impl == "reference":
        run_reference(args, w, rank)
        return
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", init_method="env://")
    try:
        run_ours(args, w, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()


if __name__ == "__main__":
    main()
