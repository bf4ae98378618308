"""GPU parity of the prefill indexer (msa_indexer_prefill: block-major, each index page
dequantised once for up to 128 query tokens of its sequence) and of the prefill selection
(msa_topk_prefill) against the oracle's indexer and selection, for prompts of one to thousands
of query tokens per sequence; against the decode indexer where both apply; and the whole prefill
path (indexer -> selection -> block-major attention) against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from parity import OracleSeq, check_attention, check_scores, check_selection

pytestmark = pytest.mark.gpu

SENTINEL = 12345.0  # written before the call: entries past a sequence's block count must keep it


@pytest.fixture(scope="module")
def msa():
    import nvfp4_kv_cache_gb300 as m

    return m


def run_indexer(msa, dl, w, status=None, decode=False):
    scores = torch.full((max(w.T, 1), 4, dl.batch.max_blocks), SENTINEL, dtype=torch.float32, device="cuda")
    if decode:
        msa.msa_indexer_decode(dl.batch, dl.cache, dl.iq8, scores, status)
    else:
        msa.msa_indexer_prefill(dl.batch, dl.cache, dl.iq8, scores, status)
    torch.cuda.synchronize()
    return scores.cpu().numpy().astype(np.float64)


def check_against_oracle(w, dl, scores, what, oracle_threads=0):
    qsl = w.query_start_loc()
    for b in range(w.B):
        ql, L = w.q_lens[b], w.seq_lens[b]
        if ql == 0:
            continue
        nb = (L + 127) // 128
        rows = slice(qsl[b], qsl[b] + ql)
        o = OracleSeq(w, 0, b, "cuda", kv_blocks=[])
        ref = oracle.indexer_seq(L, ql, o.iq8, o.index_dtype, o.ik[0], o.ik[1], nthreads=oracle_threads)
        check_scores(scores[rows, :, :nb], ref, f"{what} seq {b}")
        assert np.all(scores[rows, :, nb:] == SENTINEL), f"{what} seq {b}: entries past the block count written"


CASES = {
    "prompts": dict(seq_lens=[3000, 1500 + 33, 700], q_lens=[200, 37, 1], seed=71),
    "long_prompt": dict(seq_lens=[9000 + 5], q_lens=[1100], seed=72),
    "ragged": dict(seq_lens=[129, 4000, 0, 2600], q_lens=[129, 64, 0, 300], seed=73),
    # a fresh prompt: every token of the sequence is a query, so early tokens see few blocks
    "whole_prompt": dict(seq_lens=[777, 2100], q_lens=[777, 2100], seed=74),
    "fp8_index": dict(seq_lens=[2500, 900], q_lens=[150, 40], seed=75, index_dtype=W.INDEX_FP8),
    "shared_prefix": dict(seq_lens=[2000, 1800, 3000], q_lens=[300, 100, 50], seed=76, prefix_len=1024,
                          prefix_seqs=3),
    "outliers": dict(seq_lens=[5000, 2000], q_lens=[150, 9], seed=77, outlier_frac=0.01),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_prefill_indexer_matches_the_oracle(msa, case):
    from workloads.device import DeviceLayer

    w = W.small(case, **CASES[case])
    dl = DeviceLayer(w, 0)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    scores = run_indexer(msa, dl, w, st)
    assert msa.status_bits(st) == 0
    check_against_oracle(w, dl, scores, case)


def test_prefill_indexer_agrees_with_the_decode_indexer(msa):
    """Batches of at most 8 query tokens a sequence go through both indexers: the same scores
    (within the score tolerance: the two MMAs order their products differently) and the same
    -inf pattern."""
    from workloads.device import DeviceLayer

    w = W.small("short", [3000, 5000, 2000, 129], [8, 3, 1, 8], seed=78)
    dl = DeviceLayer(w, 0)
    a = run_indexer(msa, dl, w)
    b = run_indexer(msa, dl, w, decode=True)
    qsl = w.query_start_loc()
    for s in range(w.B):
        nb = (w.seq_lens[s] + 127) // 128
        rows = slice(qsl[s], qsl[s] + w.q_lens[s])
        check_scores(a[rows, :, :nb], b[rows, :, :nb], f"seq {s}")


def test_prefill_path_matches_the_oracle(msa):
    """Indexer -> selection -> block-major attention for prompts, each stage against the oracle:
    the selection bit-exact against the oracle's sort of the GPU scores (and against the oracle's
    own wherever the 15th and 16th candidates are more than 1e-3 apart), the attention on the GPU's
    selection against the oracle's."""
    from workloads.device import DeviceLayer, bf16_to_f32

    w = W.small("path", [6000, 2500], [400, 90], seed=79)
    dl = DeviceLayer(w, 0)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    scores = torch.empty((w.T, 4, dl.batch.max_blocks), dtype=torch.float32, device="cuda")
    sel = torch.empty((w.T, 4, 16), dtype=torch.int32, device="cuda")
    out = torch.empty((w.T, 64, 128), dtype=torch.uint16, device="cuda")
    ws = torch.empty(msa.msa_prefill_workspace_size(w.B, w.T, dl.batch.max_blocks), dtype=torch.uint8,
                     device="cuda")
    msa.msa_indexer_prefill(dl.batch, dl.cache, dl.iq8, scores, st)
    msa.msa_topk_prefill(dl.batch, scores, sel, st)
    msa.msa_prefill_attn(dl.batch, dl.cache, dl.q8, sel, dl.softmax_scale, out, ws, st)
    torch.cuda.synchronize()
    assert msa.status_bits(st) == 0
    scores_np = scores.cpu().numpy()
    sel_np = sel.cpu().numpy()
    out_np = bf16_to_f32(out).cpu().numpy()
    qsl = w.query_start_loc()
    compared = total = 0
    for b in range(w.B):
        L, ql = w.seq_lens[b], w.q_lens[b]
        nb = (L + 127) // 128
        rows = slice(qsl[b], qsl[b] + ql)
        o = OracleSeq(w, 0, b, "cuda")
        ref_scores = o.scores()
        check_scores(scores_np[rows, :, :nb], ref_scores, f"seq {b} scores")
        compared += check_selection(sel_np[rows], scores_np[rows, :, :nb], ref_scores, L, ql, f"seq {b}")
        total += 4 * ql
        check_attention(out_np[rows], o.attention(sel_np[rows], dl.softmax_scale), f"seq {b} attention")
    print(f"prefill path: {compared} of {total} (token, group) selections compared with the oracle's own")
    assert compared >= total // 2


def test_prefill_indexer_bad_page_and_bad_batch(msa):
    """A block-table entry outside the cache: that block scores -inf for every row of its
    sequence and MSA_ERR_DEVICE_FAULT is raised, the other blocks are scored as usual. An
    inconsistent batch (a sequence shorter than its query count) raises MSA_ERR_INVALID_ARG."""
    from workloads.device import DeviceLayer

    w = W.small("badpage", [2000, 1000], [150, 20], seed=80)
    dl = DeviceLayer(w, 0)
    qsl = w.query_start_loc()
    bt = dl.batch.block_table
    bad_k = 5
    good = int(bt[0, bad_k])
    bt[0, bad_k] = w.num_pages + 7
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    scores = run_indexer(msa, dl, w, st)
    bt[0, bad_k] = good
    assert msa.status_bits(st) == 1 << msa.MSA_ERR_DEVICE_FAULT
    o = OracleSeq(w, 0, 0, "cuda", kv_blocks=[])
    ref = o.scores()
    ref[:, :, bad_k] = -np.inf
    rows = slice(qsl[0], qsl[0] + w.q_lens[0])
    check_scores(scores[rows, :, :ref.shape[2]], ref, "seq 0 with a bad page")
    o1 = OracleSeq(w, 0, 1, "cuda", kv_blocks=[])
    rows1 = slice(qsl[1], qsl[1] + w.q_lens[1])
    check_scores(scores[rows1, :, :o1.scores().shape[2]], o1.scores(), "seq 1")

    sl = dl.batch.seq_lens
    keep = int(sl[1])
    sl[1] = w.q_lens[1] - 1
    st.zero_()
    run_indexer(msa, dl, w, st)
    sl[1] = keep
    assert msa.status_bits(st) & (1 << msa.MSA_ERR_INVALID_ARG)


def test_prefill_indexer_full_size(msa):
    """The bench's prefill workload (one 2,048-token prompt chunk at 16K context): every row
    against the oracle."""
    from workloads.device import DeviceLayer

    w = W.make("prefill B=1 L=16384 q_len=2048", [16384], [2048], seed=5)
    dl = DeviceLayer(w, 0)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    scores = run_indexer(msa, dl, w, st)
    assert msa.status_bits(st) == 0
    check_against_oracle(w, dl, scores, "prefill 2048 @ 16K")
