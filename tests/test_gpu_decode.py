"""GPU parity of the decode step (indexer -> top-k -> sparse attention) on small cases the
oracle finishes in seconds: ragged lengths with partial last blocks, 1..8 query tokens per
sequence, hot blocks, both index-cache dtypes, padded request rows, and every split count."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from parity import OracleSeq, check_attention, check_scores, check_selection

pytestmark = pytest.mark.gpu

CASES = {
    "ragged": dict(seq_lens=[1000, 4096 + 77, 300], q_lens=[1, 8, 3], seed=21),
    "hot": dict(seq_lens=[6000, 9000 + 5], q_lens=[8, 2], seed=22, hot=12),
    "fp8_index": dict(seq_lens=[3000, 5000, 129], q_lens=[4, 1, 2], seed=23, index_dtype=1),
    "dense": dict(seq_lens=[2048, 1500, 130], q_lens=[1, 5, 2], seed=24),
    "padded": dict(seq_lens=[4000, 0, 2500, 700, 1], q_lens=[2, 0, 0, 1, 1], seed=25),
    "many": dict(seq_lens=[129 * k + 17 for k in range(1, 20)], q_lens=[(k % 8) + 1 for k in range(19)], seed=26),
    # one query token per sequence: the single-token-batch attention kernel
    "decode1": dict(seq_lens=[1000, 4096 + 77, 300, 9000 + 5, 129, 1, 2048], q_lens=[1] * 7, seed=27, hot=6),
    "decode1_fp8": dict(seq_lens=[3000, 5000, 129], q_lens=[1, 1, 1], seed=28, index_dtype=1),
    "decode1_padded": dict(seq_lens=[4000, 0, 2500, 700], q_lens=[1, 0, 1, 1], seed=29),
    # more than 76 tokens: the attention kernel that packs a (token, group) into one CTA
    "many_tokens": dict(seq_lens=[1500 + 301 * k for k in range(12)], q_lens=[8] * 10 + [3, 5], seed=30, hot=4),
}


@pytest.fixture(scope="module")
def msa():
    import nvfp4_kv_cache_gb300 as m

    return m


def run_step(msa, dl, num_splits=None):
    o = dl.outputs()
    ws = dl.workspace()
    msa.msa_decode_step(dl.batch, dl.cache, dl.q8, dl.iq8, dl.softmax_scale, ws, o["out"], o["scores"], o["sel"])
    st = msa.msa_read_device_status(ws)
    return o, st


def compare_case(w, dl, o, device="cuda", seqs=None):
    from workloads.device import bf16_to_f32

    qsl = w.query_start_loc()
    scores = o["scores"].cpu().numpy()
    sel = o["sel"].cpu().numpy()
    out = bf16_to_f32(o["out"]).cpu().numpy()
    stats = []
    for b in (range(w.B) if seqs is None else seqs):
        ql, L = w.q_lens[b], w.seq_lens[b]
        if ql == 0:
            continue
        nb = (L + 127) // 128
        rows = slice(qsl[b], qsl[b] + ql)
        gsel = sel[rows]
        ref = OracleSeq(w, 0, b, device, kv_blocks=np.unique(gsel[gsel >= 0]))
        rs = ref.scores()
        gs = scores[rows, :, :nb]
        check_scores(gs, rs, f"seq {b}")
        check_selection(gsel, gs, rs, L, ql, f"seq {b}")
        ro = ref.attention(gsel, 1.0 / np.sqrt(128.0))
        stats.append(check_attention(out[rows], ro, f"seq {b}"))
    return stats


@pytest.mark.parametrize("case", sorted(CASES))
def test_decode_step_matches_oracle(msa, case):
    from workloads.device import DeviceLayer

    w = W.small(case, **CASES[case])
    dl = DeviceLayer(w, 0)
    o, st = run_step(msa, dl)
    assert st == msa.MSA_OK
    compare_case(w, dl, o)


@pytest.mark.parametrize("case", ["ragged", "decode1", "many_tokens"])
@pytest.mark.parametrize("splits", [1, 2, 3, 7, 16])
def test_standalone_stages_and_splits(msa, splits, case):
    """indexer, top-k and attention called one by one (any split count) == the fused step."""
    from workloads.device import DeviceLayer, bf16_to_f32

    w = W.small(case, **CASES[case])
    dl = DeviceLayer(w, 0)
    o, st = run_step(msa, dl)
    assert st == msa.MSA_OK
    T = w.T
    scores = torch.full((T, 4, dl.batch.max_blocks), float("nan"), device="cuda")
    sel = torch.empty((T, 4, 16), dtype=torch.int32, device="cuda")
    out = torch.empty((T, 64, 128), dtype=torch.uint16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    msa.msa_indexer_decode(dl.batch, dl.cache, dl.iq8, scores, status)
    msa.msa_topk_blocks(dl.batch, scores, sel, status)
    nbytes = msa.msa_attn_workspace_size(w.B, T, splits)
    ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device="cuda")
    msa.msa_sparse_attn_decode(dl.batch, dl.cache, dl.q8, sel, dl.softmax_scale, out, splits, ws, status)
    torch.cuda.synchronize()
    assert msa.status_bits(status) == 0
    qsl = w.query_start_loc()
    for b in range(w.B):
        nb = (w.seq_lens[b] + 127) // 128
        r = slice(qsl[b], qsl[b + 1])
        assert torch.equal(scores[r, :, :nb], o["scores"][r, :, :nb])
    assert torch.equal(sel, o["sel"])
    a, b_ = bf16_to_f32(out), bf16_to_f32(o["out"])
    rel = (a - b_).norm() / b_.norm()
    assert rel < 2e-3, float(rel)  # splits change only the summation order (and bf16 rounding)
    compare_case(w, dl, dict(out=out, scores=o["scores"], sel=sel))


@pytest.mark.parametrize("case", ["decode1", "many_tokens"])
def test_sharp_softmax(msa, case):
    """softmax_scale 1.0 instead of 1/sqrt(128): logits about 11x wider, so later blocks exceed
    the first block's maximum by far more than 2^8 (in exp2 units) and the many-token kernel's
    lazily moved reference must rescale its accumulators (checked on the oracle's scores
    below); both attention kernels against the oracle at the same scale."""
    from workloads.device import DeviceLayer, bf16_to_f32

    w = W.small(case, **CASES[case])
    dl = DeviceLayer(w, 0)
    o = dl.outputs()
    ws = dl.workspace()
    scale = 1.0
    msa.msa_decode_step(dl.batch, dl.cache, dl.q8, dl.iq8, scale, ws, o["out"], o["scores"], o["sel"])
    assert msa.msa_read_device_status(ws) == msa.MSA_OK
    qsl = w.query_start_loc()
    sel = o["sel"].cpu().numpy()
    out = bf16_to_f32(o["out"]).cpu().numpy()
    moves = 0
    for b in range(w.B):
        ql, L = w.q_lens[b], w.seq_lens[b]
        if ql == 0:
            continue
        rows = slice(int(qsl[b]), int(qsl[b]) + ql)
        gsel = sel[rows]
        ref = OracleSeq(w, 0, b, "cuda", kv_blocks=np.unique(gsel[gsel >= 0]))
        check_attention(out[rows], ref.attention(gsel, scale), f"seq {b}")
        # the reference moves: per (token, head), block maxima of s * scale * log2(e) in slot
        # order, a later block more than 8 above the running reference
        q = oracle.e4m3_decode(ref.q8).reshape(ql, 64, 128)
        kvals, kscales = ref.kv[0], ref.kv[1]
        for t in range(ql):
            p_tok = L - ql + t
            for g in range(4):
                blocks = list(dict.fromkeys(int(x) for x in gsel[t, g] if x >= 0))  # distinct, slot order
                per_block = [np.arange(128 * k, min(128 * k + 128, L, p_tok + 1)) for k in blocks]
                keys = np.concatenate(per_block)
                kd = oracle.e4m3_decode(oracle.dequant_nvfp4(kvals[keys, g], kscales[keys, g]))
                z = q[t, 16 * g:16 * g + 16] @ kd.T * scale * np.log2(np.e)
                first = z[:, : len(per_block[0])].max(axis=1)
                moves += int((z.max(axis=1) > first + 8.0).sum())
    if case == "many_tokens":
        assert moves > 0, "the case does not exercise the reference move"


@pytest.mark.parametrize("pad", [0, 80])
def test_topk_on_crafted_scores(msa, pad):
    """Ties, NaN, -inf, -0/+0, fewer than 15 candidates: GPU == the oracle's stable sort. With
    few rows (pad = 0) the rows longer than a warp holds take a CTA each; 80 more sequences push
    the batch past that threshold, so the same rows run one warp each."""
    rng = np.random.default_rng(5)
    # rows of 1,024 and 1,025 candidates sit on the boundary of the in-register path
    seq_lens = [128 * 700 + 3, 128 * 3 + 1, 128 * 16, 5, 128 * 4096, 128 * 1024 + 1, 128 * 1025 + 1] + [128 * 2000 + 7] * pad
    q_lens = [3, 1, 2, 1, 1, 1, 1] + [1] * pad
    B = len(seq_lens)
    maxb = 4096
    qsl = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    T = int(qsl[-1])
    scores = rng.integers(-4, 5, size=(T, 4, maxb)).astype(np.float32)
    scores[0, 0, rng.integers(0, 700, 50)] = np.nan
    scores[0, 1, rng.integers(0, 700, 50)] = -np.inf
    scores[1, 2, :] = 0.0
    scores[1, 2, ::2] = -0.0
    scores[2, 3, :] = rng.standard_normal(maxb)
    scores[5:, :, :] = rng.standard_normal((T - 5, 4, maxb))
    scores[7, 0, :] = 7.0  # all equal over 4,095 candidates
    bt = torch.zeros((B, maxb), dtype=torch.int32, device="cuda")
    batch = msa.Batch(torch.from_numpy(qsl).cuda(), torch.tensor(seq_lens, dtype=torch.int32, device="cuda"), bt,
                      max_q_len=8)
    sd = torch.from_numpy(scores).cuda()
    sel = torch.empty((T, 4, 16), dtype=torch.int32, device="cuda")
    msa.msa_topk_blocks(batch, sd, sel)
    got = sel.cpu().numpy()
    for b in range(B):
        L, ql = seq_lens[b], q_lens[b]
        for i in range(ql):
            t = qsl[b] + i
            local = (L - ql + i) // 128
            for g in range(4):
                want = oracle.select_row(scores[t, g].astype(np.float64), local)
                assert np.array_equal(got[t, g], want), (b, i, g)


@pytest.mark.parametrize("maxb", [128, 129, 256, 257, 512, 513])
@pytest.mark.parametrize("prefill", [False, True])
def test_topk_short_rows(msa, maxb, prefill):
    """The selection kernel holds 4, 8, 16 or 32 keys a lane in registers, by the longest row the
    batch allows (max_blocks_per_seq <= 128, 256, 512, else): the same crafted rows (ties, NaN,
    -inf, -0/+0, 5 to maxb - 1 candidates) on both sides of each threshold, through the decode
    entry point and through the prefill one with more than 8 query tokens a sequence, equal the
    oracle's stable sort."""
    rng = np.random.default_rng(6 + maxb + prefill)
    seq_lens = [128 * maxb, 128 * 100 + 5, 128 * 65 + 1, 128 * 64 + 1, 128 * 6, 700]
    q_lens = [12 if prefill else 8, 3, 1, 1, 2, 1]
    B = len(seq_lens)
    qsl = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    T = int(qsl[-1])
    scores = rng.standard_normal((T, 4, maxb)).astype(np.float32)
    scores[0, 0, rng.integers(0, 127, 20)] = np.nan
    scores[0, 1, rng.integers(0, 127, 20)] = -np.inf
    scores[1, 2, :] = 0.0
    scores[1, 2, ::2] = -0.0
    scores[2, 3, :] = rng.integers(-2, 3, maxb).astype(np.float32)  # heavy ties
    scores[3, 0, :] = 3.0  # all equal
    bt = torch.zeros((B, maxb), dtype=torch.int32, device="cuda")
    batch = msa.Batch(torch.from_numpy(qsl).cuda(), torch.tensor(seq_lens, dtype=torch.int32, device="cuda"), bt,
                      max_q_len=max(q_lens))
    sd = torch.from_numpy(scores).cuda()
    sel = torch.empty((T, 4, 16), dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    (msa.msa_topk_prefill if prefill else msa.msa_topk_blocks)(batch, sd, sel, st)
    got = sel.cpu().numpy()
    assert msa.status_bits(st) == 0
    for b in range(B):
        L, ql = seq_lens[b], q_lens[b]
        for i in range(ql):
            t = qsl[b] + i
            local = (L - ql + i) // 128
            for g in range(4):
                want = oracle.select_row(scores[t, g].astype(np.float64), local)
                assert np.array_equal(got[t, g], want), (b, i, g)


def test_paging_invariance(msa):
    """Identity vs permuted block tables: bit-identical scores, selection and output."""
    from workloads.device import DeviceLayer

    kw = dict(seq_lens=[5000, 3000 + 11, 777], q_lens=[4, 8, 1], seed=31, hot=8)
    outs = []
    for identity in (True, False):
        w = W.small("paging", identity=identity, **kw)
        dl = DeviceLayer(w, 0)
        o, st = run_step(msa, dl)
        assert st == msa.MSA_OK
        outs.append(o)
    for key in ("sel", "out"):
        assert torch.equal(outs[0][key], outs[1][key]), key


def test_shared_prefix_pages(msa):
    """Sequences sharing the physical pages of a prefix read the same bytes."""
    from workloads.device import DeviceLayer

    w = W.small("prefix", [16384 + 1000, 16384 + 5, 20000], [3, 1, 2], seed=32, prefix_len=16384, prefix_seqs=2)
    dl = DeviceLayer(w, 0)
    o, st = run_step(msa, dl)
    assert st == msa.MSA_OK
    compare_case(w, dl, o)


def test_cuda_graph_replay(msa):
    """The decode step captured once replays with new device contents."""
    from workloads.device import DeviceLayer

    w = W.small("graph", [3000, 4100], [2, 5], seed=33)
    dl = DeviceLayer(w, 0)
    o = dl.outputs()
    ws = dl.workspace()
    msa.msa_decode_step(dl.batch, dl.cache, dl.q8, dl.iq8, dl.softmax_scale, ws, o["out"], o["scores"], o["sel"])
    torch.cuda.synchronize()
    eager = o["out"].clone()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            msa.msa_decode_step(dl.batch, dl.cache, dl.q8, dl.iq8, dl.softmax_scale, ws, o["out"], o["scores"],
                                o["sel"])
    torch.cuda.current_stream().wait_stream(s)
    o["out"].zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(o["out"], eager)
    # new query contents, same graph
    dl.q8.copy_(torch.roll(dl.q8, 1, dims=1))
    g.replay()
    torch.cuda.synchronize()
    o2 = dl.outputs()
    msa.msa_decode_step(dl.batch, dl.cache, dl.q8, dl.iq8, dl.softmax_scale, dl.workspace(), o2["out"])
    torch.cuda.synchronize()
    assert torch.equal(o["out"], o2["out"])
