"""GPU parity of the block-major prefill attention (msa_prefill_attn: a key-block -> query map,
each selected block dequantised once for all the queries that picked it, log-sum-exp merge of
the per-block partials) against the oracle's attention, for prompts of hundreds of query tokens
per sequence, and against the decode attention where both apply."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from parity import OracleSeq, check_attention

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def msa():
    import nvfp4_kv_cache_gb300 as m

    return m


def random_selection(w: W.Workload, seed: int, dup: bool = False) -> np.ndarray:
    """Valid selections [T, 4, 16]: the token's local block in slot 0, then up to 15 distinct
    earlier blocks, -1 padding (and, with dup, a repeated block in some rows)."""
    rng = np.random.default_rng(seed)
    qsl = w.query_start_loc()
    sel = np.full((w.T, 4, 16), -1, dtype=np.int32)
    for b in range(w.B):
        L, ql = w.seq_lens[b], w.q_lens[b]
        for i in range(ql):
            t = qsl[b] + i
            local = (L - ql + i) // 128
            for g in range(4):
                k = min(15, local)
                others = rng.choice(local, size=k, replace=False) if k else np.zeros(0, np.int64)
                sel[t, g, 0] = local
                sel[t, g, 1:1 + k] = others
                if dup and k >= 2 and (t + g) % 5 == 0:
                    sel[t, g, 2] = sel[t, g, 1]
    return sel


def run_prefill(msa, dl, w, sel_np, status=None, scale=None):
    sel = torch.from_numpy(sel_np).cuda()
    out = torch.full((w.T, 64, 128), 0x7FC0, dtype=torch.uint16, device="cuda")  # NaN fill
    n = msa.msa_prefill_workspace_size(w.B, w.T, dl.batch.max_blocks)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    msa.msa_prefill_attn(dl.batch, dl.cache, dl.q8, sel, dl.softmax_scale if scale is None else scale, out, ws,
                         status)
    torch.cuda.synchronize()
    return out


CASES = {
    "prompts": dict(seq_lens=[3000, 1500 + 33, 700], q_lens=[200, 37, 1], seed=61),
    "long_prompt": dict(seq_lens=[9000 + 5], q_lens=[1100], seed=62),
    "ragged": dict(seq_lens=[129, 4000, 0, 2600], q_lens=[129, 64, 0, 300], seed=63),
    "outliers": dict(seq_lens=[5000, 2000], q_lens=[150, 9], seed=64, outlier_frac=0.01),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_prefill_matches_the_oracle(msa, case):
    from workloads.device import DeviceLayer, bf16_to_f32

    w = W.small(case, **CASES[case])
    dl = DeviceLayer(w, 0)
    sel = random_selection(w, 100 + len(case), dup=True)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = bf16_to_f32(run_prefill(msa, dl, w, sel, st)).cpu().numpy()
    assert msa.status_bits(st) == 0
    qsl = w.query_start_loc()
    for b in range(w.B):
        ql = w.q_lens[b]
        if ql == 0:
            continue
        rows = slice(qsl[b], qsl[b] + ql)
        s = sel[rows]
        ref = OracleSeq(w, 0, b, "cuda", kv_blocks=np.unique(s[s >= 0])).attention(s, dl.softmax_scale)
        check_attention(out[rows], ref, f"{case} seq {b}")


def test_prefill_equals_decode_attention_where_both_apply(msa):
    """q_len <= 8 for every sequence: the prefill path and the decode path attend over the same
    keys (different summation order)."""
    from workloads.device import DeviceLayer, bf16_to_f32

    w = W.small("both", [3000, 5000 + 7, 1300], [8, 3, 1], seed=65)
    dl = DeviceLayer(w, 0)
    sel_np = random_selection(w, 7)
    a = bf16_to_f32(run_prefill(msa, dl, w, sel_np))
    sel = torch.from_numpy(sel_np).cuda()
    b = torch.empty((w.T, 64, 128), dtype=torch.uint16, device="cuda")
    ws = torch.empty(max(msa.msa_attn_workspace_size(w.B, w.T, 0), 256), dtype=torch.uint8, device="cuda")
    msa.msa_sparse_attn_decode(dl.batch, dl.cache, dl.q8, sel, dl.softmax_scale, b, 0, ws)
    torch.cuda.synchronize()
    b = bf16_to_f32(b)
    assert float((a - b).abs().max()) <= 2e-2
    assert float((a - b).norm() / b.norm()) <= 2e-3


def test_prefill_faults_zero_fill_and_report(msa):
    from workloads.device import DeviceLayer, bf16_to_f32

    w = W.small("pfault", [3000, 2000], [100, 20], seed=66)
    dl = DeviceLayer(w, 0)
    sel = random_selection(w, 8)
    good = bf16_to_f32(run_prefill(msa, dl, w, sel))
    bad_sel = sel.copy()
    bad_sel[5, 1, 3] = 10_000  # beyond sequence 0's blocks
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = bf16_to_f32(run_prefill(msa, dl, w, bad_sel, st))
    assert msa.status_bits(st) == 1 << msa.MSA_ERR_DEVICE_FAULT
    assert (out[5, 16:32] == 0).all()
    keep = torch.ones(w.T, 64, dtype=torch.bool)
    keep[5, 16:32] = False
    assert torch.equal(out[keep], good[keep])
    # a bad page id behind a block some tokens selected: those (token, group) rows are zeroed
    bt = dl.batch.block_table.clone()
    victim = int(sel[110, 0, 1])  # a non-local block of a token of sequence 1
    bt[1, victim] = w.num_pages + 3
    batch = msa.Batch(dl.batch.query_start_loc, dl.batch.seq_lens, bt, w.max_q_len, T=w.T)
    st.zero_()
    selt = torch.from_numpy(sel).cuda()
    out2 = torch.empty((w.T, 64, 128), dtype=torch.uint16, device="cuda")
    ws = torch.empty(msa.msa_prefill_workspace_size(w.B, w.T, dl.batch.max_blocks), dtype=torch.uint8, device="cuda")
    msa.msa_prefill_attn(batch, dl.cache, dl.q8, selt, dl.softmax_scale, out2, ws, st)
    torch.cuda.synchronize()
    assert msa.status_bits(st) == 1 << msa.MSA_ERR_DEVICE_FAULT
    out2 = bf16_to_f32(out2)
    hit = (sel[100:120] == victim).any(-1)  # [20, 4] rows of sequence 1 that selected it
    for i in range(20):
        for g in range(4):
            rows = out2[100 + i, 16 * g:16 * (g + 1)]
            if hit[i, g]:
                assert (rows == 0).all()
            else:
                assert torch.equal(rows, good[100 + i, 16 * g:16 * (g + 1)])


def map_counts(w: W.Workload, sel: np.ndarray):
    """The key-block -> query map's counts from the batch alone: the valid first-occurrence
    selections, grouped by (physical page, group) and by (sequence, group, block)."""
    qsl = w.query_start_loc()
    by_page, by_seq = {}, {}
    for b in range(w.B):
        for t in range(qsl[b], qsl[b] + w.q_lens[b]):
            for g in range(4):
                seen = set()
                for v in sel[t, g]:
                    if v < 0 or v in seen:
                        continue
                    seen.add(int(v))
                    ph = int(w.block_table[b, v])
                    by_page[(ph, g)] = by_page.get((ph, g), 0) + 1
                    by_seq[(b, g, int(v))] = by_seq.get((b, g, int(v)), 0) + 1
    return by_page, by_seq


def test_shared_prefix_pages_are_dequantised_once(msa):
    """Four sequences with mixed q_len share the physical pages of a 1,024-token prefix: every
    token selects prefix blocks, and each (page, group) the sequences share is one row of the map,
    dequantised once per 64 selections of all the sequences together, with the oracle's result."""
    from workloads.device import DeviceLayer, bf16_to_f32

    w = W.small("shared_prefix", [3000, 2200 + 5, 1500, 4000 + 77, 900], [90, 3, 1, 8, 17], seed=67,
                prefix_len=1024, prefix_seqs=4)
    assert w.prefix_seqs == 4 and (w.block_table[1:4, :8] == w.block_table[0, :8]).all()
    dl = DeviceLayer(w, 0)
    sel = random_selection(w, 9)
    rng = np.random.default_rng(10)
    qsl = w.query_start_loc()
    for b in range(4):  # slot 1: prefix block 0; slot 2: another prefix block
        for t in range(qsl[b], qsl[b] + w.q_lens[b]):
            sel[t, :, 1] = 0
            sel[t, :, 2] = rng.integers(1, 8, size=4)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    seln = torch.from_numpy(sel).cuda()
    out = torch.full((w.T, 64, 128), 0x7FC0, dtype=torch.uint16, device="cuda")
    ws = torch.empty(msa.msa_prefill_workspace_size(w.B, w.T, dl.batch.max_blocks), dtype=torch.uint8, device="cuda")
    msa.msa_prefill_attn(dl.batch, dl.cache, dl.q8, seln, dl.softmax_scale, out, ws, st)
    torch.cuda.synchronize()
    assert msa.status_bits(st) == 0
    rows, chunks, entries, _ = ws[:16].view(torch.int32).cpu().tolist()
    by_page, by_seq = map_counts(w, sel)
    assert rows == len(by_page)
    assert entries == sum(by_page.values())
    assert chunks == sum((c + 63) // 64 for c in by_page.values())
    shared = {k: c for k, c in by_page.items() if k[0] in set(w.block_table[0, :8].tolist())}
    assert len(shared) == 32 and min(c for (ph, g), c in shared.items() if ph == w.block_table[0, 0]) > 64
    assert rows < len(by_seq)  # keyed by sequence, every sharing sequence would dequantise them again
    got = bf16_to_f32(out).cpu().numpy()
    for b in range(w.B):
        rows_b = slice(qsl[b], qsl[b] + w.q_lens[b])
        s = sel[rows_b]
        ref = OracleSeq(w, 0, b, "cuda", kv_blocks=np.unique(s[s >= 0])).attention(s, dl.softmax_scale)
        check_attention(got[rows_b], ref, f"shared prefix seq {b}")


def test_prefill_large_rows_split_into_chunks(msa):
    """One long prompt whose every token selects the same few blocks: rows of hundreds of
    selections are cut into chunks of 64, each served by its own CTA turn, same result."""
    from workloads.device import DeviceLayer, bf16_to_f32

    w = W.small("hot_rows", [6000 + 3], [700], seed=68)
    dl = DeviceLayer(w, 0)
    sel = random_selection(w, 11)
    sel[:, :, 1:4] = np.array([0, 1, 2], dtype=np.int32)
    sel[:, :, 4:] = np.where(sel[:, :, 4:] <= 2, -1, sel[:, :, 4:])
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    seln = torch.from_numpy(sel).cuda()
    out = torch.empty((w.T, 64, 128), dtype=torch.uint16, device="cuda")
    ws = torch.empty(msa.msa_prefill_workspace_size(w.B, w.T, dl.batch.max_blocks), dtype=torch.uint8, device="cuda")
    msa.msa_prefill_attn(dl.batch, dl.cache, dl.q8, seln, dl.softmax_scale, out, ws, st)
    torch.cuda.synchronize()
    assert msa.status_bits(st) == 0
    rows, chunks, entries, _ = ws[:16].view(torch.int32).cpu().tolist()
    by_page, _ = map_counts(w, sel)
    assert (rows, entries, chunks) == (len(by_page), sum(by_page.values()),
                                       sum((c + 63) // 64 for c in by_page.values()))
    assert max(by_page.values()) >= 600
    ref = OracleSeq(w, 0, 0, "cuda", kv_blocks=np.unique(sel[sel >= 0])).attention(sel, dl.softmax_scale)
    check_attention(bf16_to_f32(out).cpu().numpy(), ref, "hot rows")


def test_prefill_rows_with_no_key(msa):
    """(token, group) rows that list no block, and rows whose only blocks lie after the token's
    position (every key masked): their output is zero, as the oracle's; the other rows of the same
    tokens are unaffected."""
    from workloads.device import DeviceLayer, bf16_to_f32

    w = W.small("no_key", [3000, 1800 + 9], [120, 40], seed=69)
    dl = DeviceLayer(w, 0)
    sel = random_selection(w, 12)
    sel[3, 1, :] = -1            # no block listed
    sel[50, 2, :] = -1
    qsl = w.query_start_loc()
    t_early = int(qsl[0])        # the first prompt token of sequence 0: position 2880, block 22
    sel[t_early, 0, :] = -1
    sel[t_early, 0, 0] = 23      # a later block of the sequence only: all its keys are masked
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = bf16_to_f32(run_prefill(msa, dl, w, sel, st)).cpu().numpy()
    assert msa.status_bits(st) == 0
    for rows_t, g in [(3, 1), (50, 2), (t_early, 0)]:
        assert (out[rows_t, 16 * g:16 * (g + 1)] == 0).all(), (rows_t, g)
    for b in range(w.B):
        rows = slice(qsl[b], qsl[b] + w.q_lens[b])
        s = sel[rows]
        ref = OracleSeq(w, 0, b, "cuda", kv_blocks=np.unique(s[s >= 0])).attention(s, dl.softmax_scale)
        check_attention(out[rows], ref, f"no-key rows, seq {b}")


@pytest.mark.parametrize("sharp", [False, True])
def test_prefill_first_chunk_reference(msa, sharp):
    """The prefill softmax takes each (token, head, block) row's reference maximum from the
    block's first 32 keys and writes the row again from the maximum over all its keys when the
    row sum passes 128. Against the oracle at the default scale and at softmax_scale 1.0 (logits
    about 11x wider); at 1.0 the oracle's own scores must show rows of both kinds (those that
    keep the first-chunk reference and those that cannot), so both paths run."""
    from workloads.device import DeviceLayer, bf16_to_f32

    w = W.small("first_chunk", [3000, 700], [120, 33], seed=65)
    dl = DeviceLayer(w, 0)
    sel = random_selection(w, 166)
    scale = 1.0 if sharp else dl.softmax_scale
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = bf16_to_f32(run_prefill(msa, dl, w, sel, st, scale=scale)).cpu().numpy()
    assert msa.status_bits(st) == 0
    qsl = w.query_start_loc()
    keep = redo = 0
    for b in range(w.B):
        ql, L = w.q_lens[b], w.seq_lens[b]
        rows = slice(qsl[b], qsl[b] + ql)
        s = sel[rows]
        ref = OracleSeq(w, 0, b, "cuda", kv_blocks=np.unique(s[s >= 0]))
        check_attention(out[rows], ref.attention(s, scale), f"seq {b} at scale {scale}")
        if not sharp:
            continue
        q = oracle.e4m3_decode(ref.q8).reshape(ql, 64, 128)
        kvals, kscales = ref.kv[0], ref.kv[1]
        for t in range(ql):
            p_tok = L - ql + t
            for g in range(4):
                for k in dict.fromkeys(int(x) for x in s[t, g] if x >= 0):
                    keys = np.arange(128 * k, min(128 * k + 128, p_tok + 1))
                    kd = oracle.e4m3_decode(oracle.dequant_nvfp4(kvals[keys, g], kscales[keys, g]))
                    z = q[t, 16 * g:16 * g + 16] @ kd.T * scale * np.log2(np.e)
                    lazy = np.exp2(z - z[:, :32].max(axis=1, keepdims=True)).sum(axis=1)
                    redo += int((lazy > 128.0).sum())
                    keep += int((lazy <= 128.0).sum())
    if sharp:
        print(f"scale {scale}: {keep} rows keep the first-chunk reference, {redo} exceed it")
        assert keep > 0 and redo > 0
