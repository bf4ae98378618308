"""Context-sharded selection ("Indexador NVFP4 DCP"): the host candidate / merge functions of the
library against the oracle's selection, across shard counts, and the one exchange step run as
two gloo ranks on the CPU (each rank keeps its own blocks' candidates, one all-gather brings
them to the owner, which merges).

The library is only loaded, never asked to touch a GPU: the host functions are plain C++.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _scores(rng, rows: int, nb: int, kind: str) -> np.ndarray:
    """Block scores with the structures that stress an order: ties, NaN, -0/+0, -inf."""
    if kind == "ties":
        s = rng.integers(-3, 4, size=(rows, nb)).astype(np.float32) * 0.5
    else:
        s = rng.standard_normal((rows, nb)).astype(np.float32)
    if kind == "special":
        m = rng.random((rows, nb))
        s[m < 0.05] = np.nan
        s[(m >= 0.05) & (m < 0.10)] = -np.inf
        s[(m >= 0.10) & (m < 0.15)] = -0.0
        s[(m >= 0.15) & (m < 0.20)] = 0.0
    return s


def _shards(nb: int, n: int):
    """n block ranges that partition [0, nb), uneven, one of them possibly empty."""
    cuts = sorted({0, nb, *np.linspace(0, nb, n + 1).astype(int)[1:-1].tolist()})
    while len(cuts) < n + 1:
        cuts.insert(1, cuts[0])  # empty shards keep the count
    return list(zip(cuts[:-1], cuts[1:]))


@pytest.fixture(scope="module")
def msa():
    import nvfp4_kv_cache_gb300 as m

    return m


@pytest.mark.parametrize("kind", ["normal", "ties", "special"])
@pytest.mark.parametrize("n_shards", [1, 2, 3, 5, 8])
def test_host_shards_merge_to_the_oracle_selection(msa, orc, kind, n_shards):
    rng = np.random.default_rng(100 + n_shards)
    rows, nb = 96, 300
    s = _scores(rng, rows, nb, kind)
    local = rng.integers(0, nb, size=rows).astype(np.int32)
    local[:4] = [0, 1, 15, 16]  # fewer candidates than slots, exactly 15, 16
    cand = np.stack([msa.msa_topk_candidates_host(s, local, a, b) for a, b in _shards(nb, n_shards)])
    sel = msa.msa_topk_merge_host(cand, local)
    for r in range(rows):
        ref = orc.select_row(s[r].astype(np.float64), int(local[r]))
        assert np.array_equal(sel[r], ref), (r, sel[r], ref)


def test_host_candidates_are_sorted_keys_of_the_shard(msa):
    rng = np.random.default_rng(7)
    s = _scores(rng, 8, 64, "ties")
    local = np.full(8, 50, dtype=np.int32)
    cand = msa.msa_topk_candidates_host(s, local, 20, 40)
    for r in range(8):
        keys = cand[r][cand[r] != 0]
        ids = (0xFFFFFFFF - (keys & 0xFFFFFFFF)).astype(np.int64)
        assert len(keys) == 15 and np.all(keys[:-1] > keys[1:])  # unique, descending (as integers)
        assert np.all((ids >= 20) & (ids < 40))
    # a shard past the local block has no candidates; a skipped row (local < 0) none either
    assert not msa.msa_topk_candidates_host(s, local, 50, 64).any()
    assert not msa.msa_topk_candidates_host(s, np.full(8, -1, np.int32), 0, 64).any()


def _free_port() -> int:
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def _rank(rank: int, world: int, port: int, seed: int, q: "mp.Queue") -> None:
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import nvfp4_kv_cache_gb300 as m

        rng = np.random.default_rng(seed)  # every rank draws the same batch of rows
        rows, nb = 64, 257
        s = _scores(rng, rows, nb, "ties")
        local = rng.integers(0, nb, size=rows).astype(np.int32)
        a, b = _shards(nb, world)[rank]
        mine = torch.from_numpy(m.msa_topk_candidates_host(s, local, a, b).view(np.int64))
        got = [torch.empty_like(mine) for _ in range(world)]
        dist.all_gather(got, mine)  # the one exchange: world x 15 keys per row
        if rank == 0:
            cand = np.stack([g.numpy().view(np.uint64) for g in got])
            q.put((m.msa_topk_merge_host(cand, local), s, local))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_gloo_two_ranks_exchange_and_merge(orc):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, 11, q)) for r in range(2)]
    for p in procs:
        p.start()
    sel, s, local = q.get(timeout=120)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(s.shape[0]):
        assert np.array_equal(sel[r], orc.select_row(s[r].astype(np.float64), int(local[r])))


# ---- the K/V side: each rank packs the selected pages it holds; the owner assembles them ---
def _gather_case(seed: int):
    """A small batch with its own page pool (random bytes), a permuted block table and a valid
    selection (local block first, then distinct earlier blocks, -1 padded)."""
    rng = np.random.default_rng(seed)
    seq_lens = np.array([1500, 700, 128 * 9 + 5, 300], dtype=np.int32)
    q_lens = np.array([3, 1, 8, 2], dtype=np.int32)
    qsl = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    maxb = int(((seq_lens + 127) // 128).max())
    B, T = len(seq_lens), int(qsl[-1])
    num_pages = B * maxb
    bt = rng.permutation(num_pages).astype(np.int32).reshape(B, maxb)
    kv = rng.integers(0, 256, size=(num_pages, 73728), dtype=np.uint8)
    sel = np.full((T, 4, 16), -1, dtype=np.int32)
    for b in range(B):
        for i in range(q_lens[b]):
            local = (seq_lens[b] - q_lens[b] + i) // 128
            for g in range(4):
                sel[qsl[b] + i, g, 0] = local
                k = min(15, local)
                if k:
                    sel[qsl[b] + i, g, 1:1 + k] = rng.choice(local, size=k, replace=False)
    return qsl, seq_lens, bt, kv, num_pages, sel, maxb


def test_host_gather_map_numbers_the_selected_blocks(msa):
    qsl, seq_lens, bt, kv, num_pages, sel, maxb = _gather_case(3)
    mp, mk, n = msa.msa_kv_gather_map_host(qsl, seq_lens, maxb, sel)
    want = np.zeros_like(mk)
    for b in range(len(seq_lens)):
        for t in range(qsl[b], qsl[b + 1]):
            for g in range(4):
                for v in sel[t, g]:
                    if v >= 0:
                        want[b, v] |= 1 << g
    assert np.array_equal(mk, want)
    on = want.reshape(-1) != 0
    assert n == on.sum() and np.array_equal(mp.reshape(-1)[on], np.arange(n))
    assert np.all(mp.reshape(-1)[~on] == -1)
    bad = sel.copy()
    bad[0, 0, 1] = 99  # past sequence 0's blocks
    with pytest.raises(msa.MsaError):
        msa.msa_kv_gather_map_host(qsl, seq_lens, maxb, bad)


def _gather_rank(rank: int, world: int, port: int, q: "mp.Queue") -> None:
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import nvfp4_kv_cache_gb300 as m

        qsl, seq_lens, bt, kv, num_pages, sel, maxb = _gather_case(3)  # the same on every rank
        mp, mk, n = m.msa_kv_gather_map_host(qsl, seq_lens, maxb, sel)
        a, b = _shards(maxb, world)[rank]
        # this rank holds only the pages of blocks [a, b): its own pool, its own block table
        held = np.unique(bt[:, a:b])
        mine_kv = kv[held]
        local_bt = np.full_like(bt, -1)
        local_bt[:, a:b] = np.searchsorted(held, bt[:, a:b])
        pool = np.zeros((max(n, 1), 73728), dtype=np.uint8)
        m.msa_kv_gather_pages_host(local_bt, mine_kv, len(held), mp, mk, a, b, pool)
        mine = mp[:, a:b][mp[:, a:b] >= 0]  # the gathered pages this rank filled
        got = [None] * world
        dist.all_gather_object(got, (mine, pool[mine]))  # the exchange: only the filled pages move
        if rank == 0:
            owner = np.zeros_like(pool)
            for idx, pages in got:
                owner[idx] = pages
            full = np.zeros_like(pool)
            m.msa_kv_gather_pages_host(bt, kv, num_pages, mp, mk, 0, maxb, full)
            q.put((owner, full, mp, mk, bt, kv))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_gloo_two_ranks_gather_the_selected_pages():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_gather_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    owner, full, gmap, masks, bt, kv = q.get(timeout=120)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # the owner's pool equals the unsharded gather, and every selected region is the source page's
    assert np.array_equal(owner, full)
    B, maxb = gmap.shape
    for b in range(B):
        for blk in range(maxb):
            for g in range(4):
                if masks[b, blk] & (1 << g):
                    r = slice(g * 18432, (g + 1) * 18432)
                    assert np.array_equal(owner[gmap[b, blk], r], kv[bt[b, blk], r])
