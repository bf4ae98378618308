"""The allocation-free attention entry point (for callers that cannot allocate device
memory, such as a host runtime with a fixed memory plan and no allocator to pass down, or
code running inside another library's callback where cudaMalloc would synchronise the
device) gives the same results as the workspace entry point, call after call.

Both calls run the same kernel with the same split count on the same inputs, so the outputs
must be identical bit for bit: a stale or partly written partial in the shared device array
would show up as a difference. The output is also checked against the oracle directly.

Collected last on purpose, so a run that stops at the first failure has run everything
else first. It must pass alone in a fresh process and after the other tests."""
import numpy as np
import pytest
import torch

import workloads as W
from parity import OracleSeq, check_attention

pytestmark = pytest.mark.gpu


def _select(msa, dl, T):
    scores = torch.empty((T, 4, dl.batch.max_blocks), device="cuda")
    sel = torch.empty((T, 4, 16), dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    msa.msa_indexer_decode(dl.batch, dl.cache, dl.iq8, scores, status)
    msa.msa_topk_blocks(dl.batch, scores, sel, status)
    return sel, status


def _check_twice(msa, w, dl, sel, num_splits, status, oracle_seqs):
    """noalloc == workspace entry point (same split count), on two calls in a row; the output
    of the last call against the oracle's attention on the same selection."""
    from workloads.device import bf16_to_f32

    T = w.T
    need = msa.msa_attn_workspace_size(w.B, T, num_splits)
    assert 0 < need <= msa.msa_noalloc_scratch_bytes(), "the case must use the split partials and fit the array"
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    ref = torch.empty((T, 64, 128), dtype=torch.uint16, device="cuda")
    msa.msa_sparse_attn_decode(dl.batch, dl.cache, dl.q8, sel, dl.softmax_scale, ref, num_splits, ws, status)
    for call in range(2):
        out = torch.full((T, 64, 128), 0x7FC0, dtype=torch.uint16, device="cuda")  # NaN fill
        msa.msa_sparse_attn_decode_noalloc(dl.batch, dl.cache, dl.q8, sel, dl.softmax_scale, out, num_splits, status)
        torch.cuda.synchronize()
        assert torch.equal(out, ref), f"call {call}: differs from the workspace entry point"
    assert msa.status_bits(status) == 0
    qsl = w.query_start_loc()
    got = bf16_to_f32(out).cpu().numpy()
    sel_h = sel.cpu().numpy()
    for b in oracle_seqs:
        rows = slice(int(qsl[b]), int(qsl[b]) + w.q_lens[b])
        gsel = sel_h[rows]
        orc = OracleSeq(w, 0, b, "cuda", kv_blocks=np.unique(gsel[gsel >= 0]))
        check_attention(got[rows], orc.attention(gsel, dl.softmax_scale), f"noalloc seq {b}")


def test_noalloc_small_batch_kernel_twice():
    """Few tokens (the one-unit-per-CTA kernel): automatic splits (> 1) and 3 splits."""
    import nvfp4_kv_cache_gb300 as msa
    from workloads.device import DeviceLayer

    w = W.small("noalloc", [5000 + 33, 3000], [8, 3], seed=77, hot=6)
    dl = DeviceLayer(w, 0)
    sel, status = _select(msa, dl, w.T)
    _check_twice(msa, w, dl, sel, 0, status, oracle_seqs=[0, 1])
    _check_twice(msa, w, dl, sel, 3, status, oracle_seqs=[1])


def test_noalloc_many_token_kernel_twice():
    """More than 76 tokens (the persistent tensor-core kernel) with 2 splits: its partials go
    through the shared array and the merge (88 tokens: 5.8 MB of partials)."""
    import nvfp4_kv_cache_gb300 as msa
    from workloads.device import DeviceLayer

    w = W.small("noalloc-many", [1200 + 211 * k for k in range(11)], [8] * 11, seed=79, hot=4)
    assert w.T == 88
    dl = DeviceLayer(w, 0)
    sel, status = _select(msa, dl, w.T)
    _check_twice(msa, w, dl, sel, 2, status, oracle_seqs=[0, 10])


def test_noalloc_rejects_oversized_requests():
    import nvfp4_kv_cache_gb300 as msa
    from workloads.device import DeviceLayer

    w = W.small("noalloc-big", [2000], [1], seed=78)
    dl = DeviceLayer(w, 0)
    limit = msa.msa_noalloc_scratch_bytes()
    # a batch description claiming many tokens with 16 splits needs more than the array holds
    T = 8 * 512
    assert 16 * T * 64 * 129 * 4 > limit
    big = msa.Batch(dl.batch.query_start_loc, dl.batch.seq_lens, dl.batch.block_table, 8, T=T)
    big.c.B = 512
    out = torch.empty((1, 64, 128), dtype=torch.uint16, device="cuda")
    sel = torch.zeros((1, 4, 16), dtype=torch.int32, device="cuda")
    with pytest.raises(msa.MsaError) as e:
        msa.msa_sparse_attn_decode_noalloc(big, dl.cache, dl.q8, sel, dl.softmax_scale, out, 16)
    assert e.value.code == msa.MSA_ERR_INVALID_ARG
