"""Device-side setup of a workload for the CUDA library (used by GPU tests, smoke and bench).

Draws the fp32 sources of ``workloads`` on the GPU and hands them to the library's own
producers (msa_kv_insert for the paged caches, msa_quantize_fp8 for the queries). The oracle
side never uses anything built here: it quantises the same fp32 sources itself.
"""
from __future__ import annotations

import math
from typing import Dict, List, Optional

import numpy as np
import torch

import nvfp4_kv_cache_gb300 as msa
from . import BLOCK, CHUNK, GROUPS, HEAD_DIM, Q_HEADS, Workload


class DeviceLayer:
    def __init__(self, w: Workload, layer: int, device="cuda", seqs: Optional[List[int]] = None):
        self.w, self.layer, self.device = w, layer, device
        dt = w.layers[layer].index_dtype
        self.index_dtype = dt
        self.cache = msa.Cache.empty(w.num_pages, dt, device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        qsl = w.query_start_loc()
        self.batch = msa.Batch(torch.from_numpy(qsl).to(device), torch.tensor(w.seq_lens, dtype=torch.int32,
                                                                               device=device),
                               torch.from_numpy(np.ascontiguousarray(w.block_table)).to(device), w.max_q_len,
                               T=w.T)
        T = w.T
        self.q8 = torch.empty((max(T, 1), Q_HEADS, HEAD_DIM), dtype=torch.uint8, device=device)
        self.iq8 = torch.empty((max(T, 1), GROUPS, HEAD_DIM), dtype=torch.uint8, device=device)
        self.softmax_scale = 1.0 / math.sqrt(HEAD_DIM)
        todo = range(w.B) if seqs is None else seqs
        for b in todo:
            self._fill_seq(b)
        torch.cuda.synchronize()

    def _fill_seq(self, b: int) -> None:
        w, layer, dev = self.w, self.layer, self.device
        qsl = w.query_start_loc()
        ql = w.q_lens[b]
        if ql > 0:
            qf = w.q_f32(layer, b, dev).contiguous()
            iqf = w.iq_f32(layer, b, dev).contiguous()
            msa.msa_quantize_fp8(qf, self.q8[qsl[b]:qsl[b] + ql])
            msa.msa_quantize_fp8(iqf, self.iq8[qsl[b]:qsl[b] + ql])
        L = w.seq_lens[b]
        # pages of a shared prefix are written once, by sequence 0
        t_start = w.prefix_len if (0 < b < w.prefix_seqs) else 0
        for t0 in range(t_start, L, CHUNK):
            t1 = min(L, t0 + CHUNK)
            k, v = w.kv_f32(layer, b, t0, t1, dev)
            ik = w.ik_f32(layer, b, t0, t1, dev)
            slots = torch.from_numpy(w.slots(b, t0, t1)).to(dev)
            msa.msa_kv_insert(k.contiguous(), v.contiguous(), ik.contiguous(), slots, self.cache, self.status)

    def workspace(self) -> torch.Tensor:
        n = msa.msa_decode_workspace_size(self.batch.B, self.batch.T, self.batch.max_blocks)
        return torch.empty(max(n, 256), dtype=torch.uint8, device=self.device)

    def outputs(self) -> Dict[str, torch.Tensor]:
        T, maxb = max(self.batch.T, 1), self.batch.max_blocks
        return dict(out=torch.empty((T, Q_HEADS, HEAD_DIM), dtype=torch.uint16, device=self.device),
                    scores=torch.empty((T, GROUPS, maxb), dtype=torch.float32, device=self.device),
                    sel=torch.empty((T, GROUPS, 16), dtype=torch.int32, device=self.device))


def bf16_to_f32(x: torch.Tensor) -> torch.Tensor:
    """uint16 bf16 bit patterns -> float32 (bit shift, exact)."""
    return (x.to(torch.int32) << 16).view(torch.float32)
