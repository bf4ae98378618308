"""Helpers of the parity tests: oracle-side inputs and the acceptance checks.

The oracle side draws the same fp32 sources as the GPU side (``workloads``), copies them to
the host and quantises them with the oracle's own codec; nothing it uses comes from the CUDA
library. The acceptance checks are the ones the method's correctness criteria fix:
  * quantised bytes and selected block sets: bit-exact;
  * block scores: |gpu - oracle| <= 1e-3 * max(|oracle|, 1);
  * attention (bf16 output): max abs error <= 2e-2 and relative L2 error <= 1e-2, against the
    oracle's attention run on the GPU's own selected set.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads as W

SCORE_RTOL = 1e-3
ATTN_MAX_ABS = 2e-2
ATTN_REL_L2 = 1e-2


def seq_sources(w: W.Workload, layer: int, b: int, device, blocks=None):
    """Host fp32 sources of sequence b. blocks: logical blocks of K/V to draw (None = all)."""
    L = w.seq_lens[b]
    q = w.q_f32(layer, b, device).cpu().numpy()
    iq = w.iq_f32(layer, b, device).cpu().numpy()
    ik = np.concatenate([w.ik_f32(layer, b, t0, min(L, t0 + W.CHUNK), device).cpu().numpy()
                         for t0 in range(0, L, W.CHUNK)]) if L else np.zeros((0, 128), np.float32)
    k = np.zeros((L, 4, 128), np.float32)
    v = np.zeros((L, 4, 128), np.float32)
    want = range((L + 127) // 128) if blocks is None else sorted(set(int(x) for x in blocks if 0 <= x < (L + 127) // 128))
    # group contiguous blocks into ranges to keep generator calls few
    ranges = []
    for blk in want:
        if ranges and ranges[-1][1] == blk:
            ranges[-1][1] = blk + 1
        else:
            ranges.append([blk, blk + 1])
    for b0, b1 in ranges:
        t0, t1 = b0 * 128, min(L, b1 * 128)
        for c0 in range(t0, t1, W.CHUNK):
            c1 = min(t1, c0 + W.CHUNK)
            kk, vv = w.kv_f32(layer, b, c0, c1, device)
            k[c0:c1] = kk.cpu().numpy()
            v[c0:c1] = vv.cpu().numpy()
    return q, iq, ik, k, v


class OracleSeq:
    """The oracle's own quantised inputs of one sequence."""

    def __init__(self, w: W.Workload, layer: int, b: int, device, kv_blocks=None):
        self.L, self.q_len = w.seq_lens[b], w.q_lens[b]
        self.index_dtype = w.layers[layer].index_dtype
        q, iq, ik, k, v = seq_sources(w, layer, b, device, kv_blocks)
        self.q8 = oracle.quantize_fp8(q)
        self.iq8 = oracle.quantize_fp8(iq)
        if self.index_dtype == oracle.INDEX_NVFP4:
            self.ik = oracle.quantize_nvfp4(ik)
        else:
            self.ik = (oracle.quantize_fp8(ik), None)
        kv_, ks_ = oracle.quantize_nvfp4(k)
        vv_, vs_ = oracle.quantize_nvfp4(v)
        self.kv = (kv_, ks_, vv_, vs_)

    def scores(self):
        return oracle.indexer_seq(self.L, self.q_len, self.iq8, self.index_dtype, self.ik[0], self.ik[1])

    def scores_exact(self):
        """Block scores with the NVFP4 index keys taken exactly (no E4M3 re-rounding)."""
        assert self.index_dtype == oracle.INDEX_NVFP4
        return oracle.indexer_seq(self.L, self.q_len, self.iq8, oracle.INDEX_NVFP4_EXACT, self.ik[0], self.ik[1])

    def attention(self, sel, scale):
        return oracle.attention_seq(self.L, self.q_len, self.q8, *self.kv, sel, scale)


def check_scores(gpu: np.ndarray, ref: np.ndarray, what=""):
    gpu = np.asarray(gpu, np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    ninf_ref = np.isneginf(ref)
    assert np.array_equal(np.isneginf(gpu), ninf_ref), f"{what}: -inf pattern differs"
    ok = ~ninf_ref
    err = np.abs(gpu[ok] - ref[ok])
    tol = SCORE_RTOL * np.maximum(np.abs(ref[ok]), 1.0)
    bad = err > tol
    assert not bad.any(), f"{what}: {bad.sum()} scores out of tolerance, worst {err.max():.3g}"
    return float(err.max()) if err.size else 0.0


def check_selection(gpu_sel: np.ndarray, gpu_scores: np.ndarray, ref_scores: np.ndarray, L: int, q_len: int, what=""):
    """GPU sel == oracle selection on the GPU's scores (bit-exact), and == the oracle's own
    selection wherever the gap between the 15th and 16th non-local candidates exceeds 1e-3."""
    own = oracle.select_seq(gpu_scores.astype(np.float64), L, q_len)
    assert np.array_equal(gpu_sel, own), f"{what}: selection differs from the oracle's sort of the GPU scores"
    ref_sel = oracle.select_seq(ref_scores, L, q_len)
    compared = 0
    for t in range(q_len):
        local = (L - q_len + t) // 128
        for g in range(4):
            cand = np.sort(ref_scores[t, g, :local])[::-1]
            if len(cand) > 15:
                gap = cand[14] - cand[15]
                if gap <= 1e-3 * max(abs(cand[14]), 1.0):
                    continue
            compared += 1
            assert set(gpu_sel[t, g].tolist()) == set(ref_sel[t, g].tolist()), f"{what}: t={t} g={g}"
    return compared


def check_attention(gpu_bf16: np.ndarray, ref: np.ndarray, what=""):
    gpu = np.asarray(gpu_bf16, np.float64)
    err = np.abs(gpu - ref)
    max_abs = float(err.max()) if err.size else 0.0
    rel = float(np.linalg.norm(gpu - ref) / max(np.linalg.norm(ref), 1e-30)) if err.size else 0.0
    assert max_abs <= ATTN_MAX_ABS, f"{what}: max abs error {max_abs:.3g}"
    assert rel <= ATTN_REL_L2, f"{what}: relative L2 error {rel:.3g}"
    return max_abs, rel
