"""GPU parity of the context-sharded indexer ("Indexador NVFP4 DCP") run as N logical shards on
one GPU: every shard scans only its block range (msa_indexer_decode_range) and keeps its 15 best
non-local blocks per (token, group) as 64-bit keys (msa_topk_candidates); the owner merges the
N lists behind the local block (msa_topk_merge). The shards' block scores must equal the
unsharded indexer's bit for bit, and the merged selection must equal msa_topk_blocks on the
unsharded scores bit for bit (and so the oracle's selection on them, which test_gpu_decode
checks)."""
import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

CASES = {
    "ragged": dict(seq_lens=[1000, 4096 + 77, 300], q_lens=[1, 8, 3], seed=31),
    "hot": dict(seq_lens=[6000, 9000 + 5], q_lens=[8, 2], seed=32, hot=12),
    "fp8_index": dict(seq_lens=[3000, 5000, 129], q_lens=[4, 1, 2], seed=33, index_dtype=1),
    "padded": dict(seq_lens=[4000, 0, 2500, 700, 1], q_lens=[2, 0, 0, 1, 1], seed=34),
}


@pytest.fixture(scope="module")
def msa():
    import nvfp4_kv_cache_gb300 as m

    return m


def shard_ranges(maxb: int, n: int):
    """n uneven block ranges that partition [0, maxb) (the first is the shortest)."""
    cuts = [0] + [int(round(maxb * (i / n) ** 1.3)) for i in range(1, n)] + [maxb]
    return list(zip(cuts[:-1], cuts[1:]))


@pytest.mark.parametrize("case", sorted(CASES))
@pytest.mark.parametrize("n_shards", [2, 3, 5])
def test_sharded_indexer_and_merge_match_unsharded(msa, case, n_shards):
    from workloads.device import DeviceLayer

    w = W.small(case, **CASES[case])
    dl = DeviceLayer(w, 0)
    T, maxb = dl.batch.T, dl.batch.max_blocks
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    full = torch.full((T, 4, maxb), float("nan"), dtype=torch.float32, device="cuda")
    msa.msa_indexer_decode(dl.batch, dl.cache, dl.iq8, full, st)
    sel_full = torch.empty((T, 4, 16), dtype=torch.int32, device="cuda")
    msa.msa_topk_blocks(dl.batch, full, sel_full, st)

    shard = torch.full_like(full, float("nan"))
    cand = torch.empty((n_shards, T, 4, 15), dtype=torch.int64, device="cuda")
    for r, (a, b) in enumerate(shard_ranges(maxb, n_shards)):
        msa.msa_indexer_decode_range(dl.batch, dl.cache, dl.iq8, a, b, shard, st)
        msa.msa_topk_candidates(dl.batch, shard, a, b, cand[r], st)
    sel = torch.empty_like(sel_full)
    msa.msa_topk_merge(dl.batch, cand, n_shards, sel, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0

    # block scores: identical wherever the unsharded indexer wrote one
    f, s = full.cpu().numpy(), shard.cpu().numpy()
    qsl = w.query_start_loc()
    for b in range(w.B):
        ql, L = w.q_lens[b], w.seq_lens[b]
        if ql == 0:
            continue
        nb = (L + 127) // 128
        rows = slice(qsl[b], qsl[b] + ql)
        assert np.array_equal(f[rows, :, :nb].view(np.uint32), s[rows, :, :nb].view(np.uint32)), f"seq {b}"
    assert torch.equal(sel, sel_full)


def test_range_outside_every_sequence_writes_nothing(msa):
    from workloads.device import DeviceLayer

    w = W.small("tiny_range", seq_lens=[700, 300], q_lens=[2, 1], seed=35)
    dl = DeviceLayer(w, 0)
    T, maxb = dl.batch.T, dl.batch.max_blocks
    sc = torch.full((T, 4, maxb), 7.0, dtype=torch.float32, device="cuda")
    msa.msa_indexer_decode_range(dl.batch, dl.cache, dl.iq8, 6, 100, sc)  # both sequences end before block 6
    torch.cuda.synchronize()
    assert bool((sc == 7.0).all())
    with pytest.raises(msa.MsaError):
        msa.msa_indexer_decode_range(dl.batch, dl.cache, dl.iq8, 3, 2, sc)
