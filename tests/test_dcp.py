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
