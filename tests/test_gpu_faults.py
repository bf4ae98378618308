"""Device-side fault reporting without faulting the GPU.

Bad page ids, out-of-range selected blocks and inconsistent batch descriptions are found by
the kernels' own checks and reported in the status word; the bounded-wait mechanism is
exercised with a barrier nobody arrives on. Every case here keeps all memory accesses in
bounds: the checks skip the access instead of making it.
"""
import numpy as np
import pytest
import torch

import workloads as W
from parity import OracleSeq, check_attention

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def msa():
    import nvfp4_kv_cache_gb300 as m

    return m


def layer(w):
    from workloads.device import DeviceLayer

    return DeviceLayer(w, 0)


def step(msa, dl, batch=None):
    o = dl.outputs()
    ws = dl.workspace()
    msa.msa_decode_step(batch or dl.batch, dl.cache, dl.q8, dl.iq8, dl.softmax_scale, ws, o["out"], o["scores"],
                        o["sel"])
    return o, msa.msa_read_device_status(ws)


# few tokens run the attention kernel that spreads a (token, group) over an SM; 88 tokens run
# the one that packs a (token, group) into one CTA of eight block-owning warps
MANY = [8, 8] + [8] * 9


@pytest.mark.parametrize("q_lens", [[2, 1], [1, 1], MANY])
def test_bad_page_id_is_reported_and_zero_filled(msa, q_lens):
    from workloads.device import bf16_to_f32

    w = W.small("fault", [3000, 2000] + [1000] * (len(q_lens) - 2), q_lens, seed=41)
    q0 = q_lens[0]
    dl = layer(w)
    good, st = step(msa, dl)
    assert st == msa.MSA_OK
    bt = dl.batch.block_table.clone()
    nb1 = (w.seq_lens[1] + 127) // 128
    bt[1, nb1 - 1] = w.num_pages + 7   # the local block of sequence 1: always selected
    bt[0, 3] = -5                       # a middle block of sequence 0
    batch = msa.Batch(dl.batch.query_start_loc, dl.batch.seq_lens, bt, w.max_q_len, T=w.T)
    o, st = step(msa, dl, batch)
    assert st == msa.MSA_ERR_DEVICE_FAULT
    s = o["scores"].cpu().numpy()
    assert np.isneginf(s[0:q0, :, 3]).all()
    out = bf16_to_f32(o["out"])
    assert (out[q0] == 0).all(), "tokens whose selected page is bad are zero-filled"
    # sequence 0 never selects the -inf block; its other scores are unchanged and its output
    # is the oracle's attention over its (new) selection
    sel0 = o["sel"][0:q0].cpu().numpy()
    assert not (sel0 == 3).any()
    keep = [k for k in range(24) if k != 3]
    assert torch.equal(o["scores"][0:q0, :, keep], good["scores"][0:q0, :, keep])
    ref = OracleSeq(w, 0, 0, "cuda", kv_blocks=np.unique(sel0))
    check_attention(out[0:q0].cpu().numpy(), ref.attention(sel0, dl.softmax_scale), "seq 0")


@pytest.mark.parametrize("q_lens", [[1, 2], [1, 1], MANY])
def test_selected_block_out_of_range(msa, q_lens):
    from workloads.device import bf16_to_f32

    w = W.small("selbad", [1500, 900] + [1000] * (len(q_lens) - 2), q_lens, seed=42)
    dl = layer(w)
    o, st = step(msa, dl)
    sel = o["sel"].clone()
    sel[1, 2, 5] = 99  # beyond sequence 1's 8 blocks
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty_like(o["out"])
    ws = torch.empty(max(msa.msa_attn_workspace_size(w.B, w.T, 0), 256), dtype=torch.uint8, device="cuda")
    msa.msa_sparse_attn_decode(dl.batch, dl.cache, dl.q8, sel, dl.softmax_scale, out, 0, ws, status)
    torch.cuda.synchronize()
    assert msa.status_bits(status) == 1 << msa.MSA_ERR_DEVICE_FAULT
    outf = bf16_to_f32(out)
    assert (outf[1, 32:48] == 0).all()      # group 2 of token 1 zero-filled
    assert torch.equal(out[0], o["out"][0])  # other tokens untouched
    assert torch.equal(out[1, :32], o["out"][1, :32])


def test_inconsistent_batch_is_reported(msa):
    w = W.small("badbatch", [2000, 1000], [2, 2], seed=43)
    dl = layer(w)
    # sequence 1 claims 3 query tokens but the token count says 2, and seq_lens < q_len
    qsl = torch.tensor([0, 2, 5], dtype=torch.int32, device="cuda")
    sl = torch.tensor([2000, 2], dtype=torch.int32, device="cuda")
    batch = msa.Batch(qsl, sl, dl.batch.block_table, 8, T=4)
    o, st = step(msa, dl, batch)
    assert st == msa.MSA_ERR_INVALID_ARG


def test_bounded_wait_times_out_cleanly(msa):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    msa.msa_selftest_wait_timeout(status, 2_000_000)  # 2 ms
    torch.cuda.synchronize()
    assert msa.status_bits(status) == 1 << msa.MSA_ERR_TIMEOUT
    # the context is still healthy: a normal step runs and succeeds
    w = W.small("after", [1000], [1], seed=44)
    dl = layer(w)
    o, st = step(msa, dl)
    assert st == msa.MSA_OK


def test_host_side_errors(msa):
    w = W.small("host", [1000], [1], seed=45)
    dl = layer(w)
    with pytest.raises(msa.MsaError) as e:
        msa.msa_sparse_attn_decode(dl.batch, dl.cache, dl.q8, torch.zeros((1, 4, 16), dtype=torch.int32,
                                                                             device="cuda"), -1.0,
                                   torch.empty((1, 64, 128), dtype=torch.uint16, device="cuda"))
    assert e.value.code == msa.MSA_ERR_INVALID_ARG
    small_ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(msa.MsaError):
        msa.msa_decode_step(dl.batch, dl.cache, dl.q8, dl.iq8, dl.softmax_scale, small_ws,
                            torch.empty((1, 64, 128), dtype=torch.uint16, device="cuda"))
