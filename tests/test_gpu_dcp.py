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


# ---- the K/V side: the selected blocks' pages gathered on the owner ------------------------
GATHER_CASES = {
    "few_tokens": dict(seq_lens=[6000, 9000 + 5, 300], q_lens=[8, 2, 3], seed=36, hot=12),
    # more than 76 tokens: the owner's attention runs the persistent tensor-core kernel
    "many_tokens": dict(seq_lens=[1500 + 301 * k for k in range(12)], q_lens=[8] * 10 + [3, 5], seed=37, hot=4),
    "padded": dict(seq_lens=[4000, 0, 2500, 700, 1], q_lens=[2, 0, 0, 1, 1], seed=38),
}


def shard_pool(dl, a: int, b: int):
    """The page pool and block table of a rank that holds blocks [a, b) of every sequence: its
    own pages (renumbered from the tail, so no id matches the unsharded one), -1 elsewhere."""
    import nvfp4_kv_cache_gb300 as m

    bt = dl.batch.block_table
    held = bt[:, a:b]
    ids = torch.unique(held[held >= 0])
    local = torch.full_like(bt, -1)
    remap = torch.full((dl.cache.num_pages,), -1, dtype=torch.int32, device=bt.device)
    remap[ids.long()] = torch.arange(len(ids) - 1, -1, -1, dtype=torch.int32, device=bt.device)
    local[:, a:b] = torch.where(held >= 0, remap[held.clamp(min=0).long()], held)
    kv = dl.cache.kv_pages.view(-1, m.KV_PAGE_BYTES)
    pool = torch.zeros((max(len(ids), 1), m.KV_PAGE_BYTES), dtype=torch.uint8, device=bt.device)
    if len(ids):
        pool[remap[ids.long()].long()] = kv[ids.long()]
    cache = m.Cache(pool.view(-1), dl.cache.index_pages, dl.cache.index_dtype, len(ids))
    batch = m.Batch(dl.batch.query_start_loc, dl.batch.seq_lens, local, dl.batch.max_q_len, T=dl.batch.T)
    return batch, cache


@pytest.mark.parametrize("case", sorted(GATHER_CASES))
@pytest.mark.parametrize("n_shards", [1, 2, 3])
def test_gathered_pages_give_the_unsharded_attention(msa, case, n_shards):
    """Every shard copies its selected blocks' K/V into the owner's gathered pool; the owner's
    attention over that pool (block table = the gather map) equals the unsharded attention bit
    for bit, and every gathered (page, group) region equals the source page's."""
    from workloads.device import DeviceLayer

    w = W.small(case, **GATHER_CASES[case])
    dl = DeviceLayer(w, 0)
    T, B, maxb = dl.batch.T, dl.batch.B, dl.batch.max_blocks
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    o = dl.outputs()
    ws = dl.workspace()
    msa.msa_decode_step(dl.batch, dl.cache, dl.q8, dl.iq8, dl.softmax_scale, ws, o["out"], o["scores"], o["sel"])
    sel = o["sel"]
    ref = o["out"]

    gmap = torch.empty((B, maxb), dtype=torch.int32, device="cuda")
    masks = torch.empty((B, maxb), dtype=torch.uint8, device="cuda")
    ng = torch.empty(1, dtype=torch.int32, device="cuda")
    msa.msa_kv_gather_map(dl.batch, sel, gmap, masks, ng, st)
    torch.cuda.synchronize()
    n = int(ng.item())
    # the numbering: the distinct selected (sequence, block) pairs, in order
    s_h, q_h = sel.cpu().numpy(), w.query_start_loc()
    want = np.zeros((B, maxb), dtype=np.uint8)
    for b in range(B):
        for t in range(q_h[b], q_h[b + 1]):
            for g in range(4):
                for v in s_h[t, g]:
                    if v >= 0:
                        want[b, v] |= 1 << g
    assert np.array_equal(masks.cpu().numpy(), want)
    flat = want.reshape(-1) != 0
    assert n == int(flat.sum())
    assert np.array_equal(gmap.cpu().numpy().reshape(-1)[flat], np.arange(n))
    assert np.all(gmap.cpu().numpy().reshape(-1)[~flat] == -1)

    pool = torch.zeros((max(n, 1), msa.KV_PAGE_BYTES), dtype=torch.uint8, device="cuda")
    for a, b in shard_ranges(maxb, n_shards):
        sb, sc = shard_pool(dl, a, b)
        msa.msa_kv_gather_pages(sb, sc, gmap, masks, a, b, pool, n, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    # every gathered region is the source page's region
    kv = dl.cache.kv_pages.view(-1, msa.KV_PAGE_BYTES).cpu().numpy()
    bt, gm, pl = dl.batch.block_table.cpu().numpy(), gmap.cpu().numpy(), pool.cpu().numpy()
    for b in range(B):
        for blk in range(maxb):
            for g in range(4):
                if want[b, blk] & (1 << g):
                    r = slice(g * 18432, (g + 1) * 18432)
                    assert np.array_equal(pl[gm[b, blk], r], kv[bt[b, blk], r]), (b, blk, g)

    # the owner: its block table is the map, its cache the gathered pool
    owner_batch = msa.Batch(dl.batch.query_start_loc, dl.batch.seq_lens, gmap, dl.batch.max_q_len, T=T)
    owner_cache = msa.Cache(pool.view(-1), dl.cache.index_pages, dl.cache.index_dtype, n)
    out = torch.full_like(ref, 0x7FC0)
    aws = torch.empty(max(msa.msa_attn_workspace_size(B, T, 0), 256), dtype=torch.uint8, device="cuda")
    msa.msa_sparse_attn_decode(owner_batch, owner_cache, dl.q8, sel, dl.softmax_scale, out, 0, aws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(out, ref)


def test_gather_rejects_and_flags(msa):
    from workloads.device import DeviceLayer

    w = W.small("gather_bad", seq_lens=[700, 300], q_lens=[2, 1], seed=39)
    dl = DeviceLayer(w, 0)
    T, B, maxb = dl.batch.T, dl.batch.B, dl.batch.max_blocks
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    sel = torch.full((T, 4, 16), -1, dtype=torch.int32, device="cuda")
    sel[0, 0, 0] = 5  # sequence 0 has 6 blocks: fine
    sel[T - 1, 2, 3] = 9  # sequence 1 has 3 blocks: out of range -> flagged and ignored
    gmap = torch.empty((B, maxb), dtype=torch.int32, device="cuda")
    masks = torch.empty((B, maxb), dtype=torch.uint8, device="cuda")
    ng = torch.empty(1, dtype=torch.int32, device="cuda")
    msa.msa_kv_gather_map(dl.batch, sel, gmap, masks, ng, st)
    torch.cuda.synchronize()
    assert int(ng.item()) == 1 and int(gmap[0, 5].item()) == 0 and int(masks[0, 5].item()) == 1
    assert msa.status_bits(st) == 1 << msa.MSA_ERR_DEVICE_FAULT
    pool = torch.zeros((1, msa.KV_PAGE_BYTES), dtype=torch.uint8, device="cuda")
    with pytest.raises(msa.MsaError):
        msa.msa_kv_gather_pages(dl.batch, dl.cache, gmap, masks, 3, 2, pool, 1)
    st.zero_()
    msa.msa_kv_gather_pages(dl.batch, dl.cache, gmap, masks, 0, maxb, pool, 0, st)  # no room: nothing copied
    torch.cuda.synchronize()
    assert int(st.item()) == 0
