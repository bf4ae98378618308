"""Seeded synthetic inputs for the MSA decode step (shared by tests, smoke and bench).

This module holds none of the method's arithmetic: it only draws fp32 sources (queries,
index queries, index keys, K, V), sequence lengths, query lengths and paged block tables.
Both the CUDA path and the oracle quantise from the fp32 values drawn here.

Values are N(0, 1) fp32 drawn with torch generators on the requested device, one generator
per (seed, sequence, tensor kind, 8,192-token chunk), so any token range of any sequence can
be regenerated on its own (the parity tests at full size regenerate only sampled sequences).
Small host-side choices (page permutations, hot blocks, outlier channels, ragged lengths)
use numpy ``default_rng``.

Workload structure follows the configurations the method is measured on:
  * "tiny":    B=1, L=4,096, q_len=1, identity block table                       (seed 0)
  * "decode":  B=32, L=32,768, q_len=1, 24 planted hot blocks, random paging      (seed 1)
  * "spec":    B=64, L=131,072, q_len=8, hot blocks, random paging                (seed 2)
  * "long":    B=8, L=524,288, q_len=1, 1% of K and of V channels x8, paging      (seed 3)
  * "ragged":  4 layers, B=128, L log-uniform in [1,024, 262,144], q_len U{1..8},
               NVFP4 index in layers 0-1 and FP8 in layers 2-3, a 16,384-token prefix whose
               pages are shared by sequences 0-31                                 (seeds 4000+l)
Hot blocks ("aligned with index-q"): for each token of a hot block the index key gets
+3.0 * u_b, u_b = normalize(sum over the sequence's query tokens and groups of the fp32
index queries).
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import numpy as np
import torch

HEAD_DIM = 128
GROUPS = 4
Q_HEADS = 64
BLOCK = 128
CHUNK = 8192  # tokens per generator chunk

INDEX_NVFP4 = 0
INDEX_FP8 = 1

_KIND = {"q": 1, "iq": 2, "ik": 3, "k": 4, "v": 5}


def _mix(*xs: int) -> int:
    """Deterministic 63-bit seed from integers (splitmix-style avalanche)."""
    h = 0x9E3779B97F4A7C15
    for x in xs:
        h ^= (int(x) + 0x9E3779B97F4A7C15 + ((h << 6) & (2**64 - 1)) + (h >> 2)) & (2**64 - 1)
        h = (h * 0xBF58476D1CE4E5B9) & (2**64 - 1)
        h ^= h >> 31
    return h & (2**63 - 1)


def _randn(shape, seed: int, device) -> torch.Tensor:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32)


@dataclasses.dataclass
class Layer:
    seed: int
    index_dtype: int


@dataclasses.dataclass
class Workload:
    name: str
    seq_lens: List[int]
    q_lens: List[int]
    layers: List[Layer]
    block_table: np.ndarray          # [B, max_blocks] int32 physical page ids, -1 unused
    num_pages: int
    hot_blocks: List[np.ndarray]     # per sequence, logical block ids
    k_outlier: Optional[np.ndarray] = None   # flat channel ids in [0, 512) of K scaled x8
    v_outlier: Optional[np.ndarray] = None
    prefix_len: int = 0              # tokens of the shared prefix
    prefix_seqs: int = 0             # sequences 0 .. prefix_seqs-1 share it
    hot_gain: float = 3.0

    @property
    def B(self) -> int:
        return len(self.seq_lens)

    @property
    def T(self) -> int:
        return int(sum(self.q_lens))

    @property
    def max_blocks(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def max_q_len(self) -> int:
        return max(1, max(self.q_lens) if self.q_lens else 1)

    def query_start_loc(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.q_lens)]).astype(np.int32)

    def nblocks(self, b: int) -> int:
        return (self.seq_lens[b] + BLOCK - 1) // BLOCK

    # ---------------------------------------------------------------- fp32 sources
    def _shared(self, b: int, tok: int) -> bool:
        return b < self.prefix_seqs and tok < self.prefix_len

    def q_f32(self, layer: int, b: int, device="cpu") -> torch.Tensor:
        return _randn((self.q_lens[b], Q_HEADS, HEAD_DIM), _mix(self.layers[layer].seed, _KIND["q"], b), device)

    def iq_f32(self, layer: int, b: int, device="cpu") -> torch.Tensor:
        return _randn((self.q_lens[b], GROUPS, HEAD_DIM), _mix(self.layers[layer].seed, _KIND["iq"], b), device)

    def _chunks(self, layer: int, b: int, kind: str, width, t0: int, t1: int, device) -> torch.Tensor:
        """Rows [t0, t1) of the per-token fp32 stream `kind` of sequence b."""
        out = []
        c0, c1 = t0 // CHUNK, (t1 - 1) // CHUNK
        for c in range(c0, c1 + 1):
            a, e = max(t0, c * CHUNK), min(t1, (c + 1) * CHUNK)
            shared = self._shared(b, c * CHUNK)
            owner = -1 if shared else b
            x = _randn((CHUNK,) + tuple(width), _mix(self.layers[layer].seed, _KIND[kind], owner, c), device)
            if shared and (c + 1) * CHUNK > self.prefix_len:
                # a chunk straddling the end of the shared prefix: the tail is the sequence's own
                y = _randn((CHUNK,) + tuple(width), _mix(self.layers[layer].seed, _KIND[kind], b, c), device)
                cut = self.prefix_len - c * CHUNK
                x = torch.cat([x[:cut], y[cut:]], 0)
            out.append(x[a - c * CHUNK:e - c * CHUNK])
        return torch.cat(out, 0) if len(out) > 1 else out[0]

    def ik_f32(self, layer: int, b: int, t0: int, t1: int, device="cpu") -> torch.Tensor:
        x = self._chunks(layer, b, "ik", (HEAD_DIM,), t0, t1, device)
        hot = self.hot_blocks[b] if b < len(self.hot_blocks) else np.zeros(0, np.int64)
        if hot.size:
            iq = self.iq_f32(layer, b, device)
            u = iq.reshape(-1, HEAD_DIM).sum(0)
            u = u / torch.linalg.vector_norm(u)
            mask = torch.from_numpy(np.isin(np.arange(t0, t1) // BLOCK, hot)).to(device)
            x = x + (self.hot_gain * mask.to(torch.float32))[:, None] * u[None, :]
        return x

    def kv_f32(self, layer: int, b: int, t0: int, t1: int, device="cpu"):
        k = self._chunks(layer, b, "k", (GROUPS, HEAD_DIM), t0, t1, device)
        v = self._chunks(layer, b, "v", (GROUPS, HEAD_DIM), t0, t1, device)
        if self.k_outlier is not None:
            sk = torch.ones(GROUPS * HEAD_DIM, device=device)
            sk[torch.from_numpy(self.k_outlier).to(device)] = 8.0
            k = k * sk.view(GROUPS, HEAD_DIM)
        if self.v_outlier is not None:
            sv = torch.ones(GROUPS * HEAD_DIM, device=device)
            sv[torch.from_numpy(self.v_outlier).to(device)] = 8.0
            v = v * sv.view(GROUPS, HEAD_DIM)
        return k, v

    def slots(self, b: int, t0: int, t1: int) -> np.ndarray:
        """Cache slots (physical page * 128 + row) of tokens [t0, t1) of sequence b."""
        tok = np.arange(t0, t1)
        return (self.block_table[b, tok // BLOCK].astype(np.int64) * BLOCK + tok % BLOCK)

    def unique_pages(self) -> int:
        """Physical pages referenced by the batch, shared pages counted once."""
        pages = set()
        for b in range(self.B):
            pages.update(self.block_table[b, :self.nblocks(b)].tolist())
        return len(pages)


# ---------------------------------------------------------------------- construction
def _paging(nblocks: List[int], rng, identity: bool, prefix_blocks: int = 0, prefix_seqs: int = 0):
    B = len(nblocks)
    maxb = max(max(nblocks), 1)
    owned = [nb - (prefix_blocks if b < prefix_seqs else 0) for b, nb in enumerate(nblocks)]
    total = prefix_blocks + sum(owned)
    perm = np.arange(total) if identity else rng.permutation(total)
    table = np.full((B, maxb), -1, dtype=np.int32)
    pos = prefix_blocks
    for b in range(B):
        k0 = 0
        if b < prefix_seqs:
            table[b, :prefix_blocks] = perm[:prefix_blocks]
            k0 = prefix_blocks
        n = nblocks[b] - k0
        table[b, k0:nblocks[b]] = perm[pos:pos + n]
        pos += n
    return table, total


def _hot(nblocks: List[int], q_lens: List[int], seq_lens: List[int], count: int, rng) -> List[np.ndarray]:
    out = []
    for b, nb in enumerate(nblocks):
        first_local = (seq_lens[b] - q_lens[b]) // BLOCK  # non-local for every query token
        pool = np.arange(first_local)
        out.append(np.sort(rng.choice(pool, size=min(count, pool.size), replace=False)))
    return out


def make(name: str, seq_lens, q_lens, seed: int, index_dtype: int = INDEX_NVFP4, hot: int = 0,
         identity: bool = False, outlier_frac: float = 0.0, n_layers: int = 1,
         layer_dtypes=None, layer_seeds=None, prefix_len: int = 0, prefix_seqs: int = 0) -> Workload:
    assert not (hot and prefix_seqs), "hot blocks would break the sharing of prefix pages"
    rng = np.random.default_rng(seed)
    seq_lens = [int(x) for x in seq_lens]
    q_lens = [int(x) for x in q_lens]
    nb = [(L + BLOCK - 1) // BLOCK for L in seq_lens]
    assert prefix_len % BLOCK == 0
    # content choices first, so the block table (identity or permuted) changes nothing else
    hot_blocks = _hot(nb, q_lens, seq_lens, hot, rng) if hot else [np.zeros(0, np.int64)] * len(nb)
    ko = vo = None
    if outlier_frac > 0:
        n = int(round(outlier_frac * GROUPS * HEAD_DIM))
        ko = np.sort(rng.choice(GROUPS * HEAD_DIM, size=n, replace=False))
        vo = np.sort(rng.choice(GROUPS * HEAD_DIM, size=n, replace=False))
    table, total = _paging(nb, rng, identity, prefix_len // BLOCK, prefix_seqs)
    dtypes = layer_dtypes or [index_dtype] * n_layers
    seeds = layer_seeds or [seed + 1000 * l for l in range(n_layers)]
    layers = [Layer(seed=int(s), index_dtype=int(d)) for s, d in zip(seeds, dtypes)]
    return Workload(name, seq_lens, q_lens, layers, table, total, hot_blocks, ko, vo,
                    prefix_len, prefix_seqs)


def tiny() -> Workload:
    return make("tiny B=1 L=4096 q_len=1", [4096], [1], seed=0, identity=True)


def decode() -> Workload:
    return make("decode B=32 L=32768 q_len=1 hot=24", [32768] * 32, [1] * 32, seed=1, hot=24)


def spec() -> Workload:
    return make("spec-decode B=64 L=131072 q_len=8 hot=24", [131072] * 64, [8] * 64, seed=2, hot=24)


def spec_16k() -> Workload:
    """The spec-decode structure at 16K context (a profiling size: ~0.7 GB resident)."""
    return make("spec-decode B=64 L=16384 q_len=8 hot=24", [16384] * 64, [8] * 64, seed=2, hot=24)


def long_context() -> Workload:
    return make("long B=8 L=524288 q_len=1 outliers=1%", [524288] * 8, [1] * 8, seed=3, outlier_frac=0.01)


def ragged() -> Workload:
    rng = np.random.default_rng(4)
    B, prefix, nshare = 128, 16384, 32
    lo, hi = math.log(1024), math.log(262144)
    L = np.floor(np.exp(rng.uniform(lo, hi, size=B))).astype(np.int64)
    L[:nshare] = np.floor(np.exp(rng.uniform(math.log(prefix + 1), hi, size=nshare))).astype(np.int64)
    q = rng.integers(1, 9, size=B)
    L = np.maximum(L, q)
    return make("ragged B=128 L=logU[1024,262144] q_len=U{1..8} 4 layers", L.tolist(), q.tolist(), seed=4,
                n_layers=4, layer_dtypes=[INDEX_NVFP4, INDEX_NVFP4, INDEX_FP8, INDEX_FP8],
                layer_seeds=[4000, 4001, 4002, 4003], prefix_len=prefix, prefix_seqs=nshare)


CONFIGS = {"tiny": tiny, "decode": decode, "spec": spec, "spec_16k": spec_16k, "long": long_context,
           "ragged": ragged}


def small(name: str, seq_lens, q_lens, seed: int, **kw) -> Workload:
    """A small case of the same structure, for parity tests the oracle finishes in seconds."""
    return make(name, seq_lens, q_lens, seed, **kw)
