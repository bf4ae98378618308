"""The allocation-free attention entry point (for callers that cannot allocate device
memory, such as a host runtime with a fixed memory plan and no allocator to pass down, or
code running inside another library's callback where cudaMalloc would synchronise the
device) gives the same results as the workspace entry point, call after call.

Collected last on purpose, so a run that stops at the first failure has run everything
else first. It must pass alone in a fresh process and after the other tests."""
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

REL_L2 = 1e-2     # the attention tolerance of the parity tests
MAX_ABS = 2e-2


def test_noalloc_matches_workspace_entry_point_twice():
    import nvfp4_kv_cache_gb300 as msa
    from workloads.device import DeviceLayer, bf16_to_f32

    # B=2 makes the automatic split count > 1, so the scratch array is really used
    w = W.small("noalloc", [5000 + 33, 3000], [8, 3], seed=77, hot=6)
    dl = DeviceLayer(w, 0)
    T = w.T
    scores = torch.empty((T, 4, dl.batch.max_blocks), device="cuda")
    sel = torch.empty((T, 4, 16), dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    msa.msa_indexer_decode(dl.batch, dl.cache, dl.iq8, scores, status)
    msa.msa_topk_blocks(dl.batch, scores, sel, status)
    assert msa.msa_attn_workspace_size(w.B, T, 0) > 0, "the case must exercise the split partials"
    ws = torch.empty(msa.msa_attn_workspace_size(w.B, T, 0), dtype=torch.uint8, device="cuda")
    ref = torch.empty((T, 64, 128), dtype=torch.uint16, device="cuda")
    msa.msa_sparse_attn_decode(dl.batch, dl.cache, dl.q8, sel, dl.softmax_scale, ref, 0, ws, status)
    refd = bf16_to_f32(ref)
    for call in range(2):
        out = torch.full((T, 64, 128), 0x7FC0, dtype=torch.uint16, device="cuda")  # NaN fill
        msa.msa_sparse_attn_decode_noalloc(dl.batch, dl.cache, dl.q8, sel, dl.softmax_scale, out, 0, status)
        torch.cuda.synchronize()
        got = bf16_to_f32(out)
        assert torch.isfinite(got).all(), f"call {call}: output not fully written"
        diff = (got - refd)
        assert float(diff.abs().max()) <= MAX_ABS, f"call {call}"
        assert float(diff.norm() / refd.norm()) <= REL_L2, f"call {call}"
    assert msa.status_bits(status) == 0


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
