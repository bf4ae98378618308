"""The decode step from page-locked host buffers (msa_decode_step_host): its output equals
msa_decode_step's bit for bit, copied back (the attention in one launch or split in two) or
stored into host memory by the attention itself, and the host checks reject buffers that are
not page-locked."""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

CASES = {
    # one query token per sequence: the small-batch attention kernel, one launch
    "decode1": dict(seq_lens=[1000, 4096 + 77, 300, 9000 + 5, 129], q_lens=[1] * 5, seed=41),
    # 96 tokens: the many-token kernel, too few rounds to split
    "tc_one_launch": dict(seq_lens=[1500 + 211 * k for k in range(12)], q_lens=[8] * 12, seed=42, hot=3),
    # 211 tokens (ragged query counts): the many-token kernel in two launches, split inside a
    # sequence's tokens
    "tc_split": dict(seq_lens=[1200 + 173 * k for k in range(28)], q_lens=[8] * 25 + [1, 3, 7], seed=43, hot=3),
}


@pytest.fixture(scope="module")
def msa():
    import nvfp4_kv_cache_gb300 as m

    return m


def pinned(t: torch.Tensor) -> torch.Tensor:
    return t.cpu().contiguous().pin_memory()


@pytest.mark.parametrize("direct", [False, True])
@pytest.mark.parametrize("case", sorted(CASES))
def test_host_step_equals_device_step(msa, case, direct):
    from workloads.device import DeviceLayer

    w = W.small(case, **CASES[case])
    dl = DeviceLayer(w, 0)
    o = dl.outputs()
    ws = dl.workspace()
    msa.msa_decode_step(dl.batch, dl.cache, dl.q8, dl.iq8, dl.softmax_scale, ws, o["out"])
    assert msa.msa_read_device_status(ws) == msa.MSA_OK
    ref = o["out"].view(torch.int16).cpu()

    b = dl.batch
    h = [pinned(x) for x in (b.query_start_loc, b.seq_lens, b.block_table, dl.q8, dl.iq8)]
    h_out = torch.full(tuple(o["out"].shape), 7, dtype=o["out"].dtype).pin_memory()
    # fresh device buffers: everything the step reads comes through the copies
    d = [torch.zeros_like(x) for x in (b.query_start_loc, b.seq_lens, b.block_table, dl.q8, dl.iq8)]
    batch2 = msa.Batch(d[0], d[1], d[2], b.max_q_len, T=b.T)
    out2 = None if direct else torch.zeros_like(o["out"])
    ws2 = dl.workspace()
    copy = torch.cuda.Stream()
    for _ in range(2):  # the second call reuses every buffer
        msa.msa_decode_step_host(batch2, dl.cache, h[0], h[1], h[2], h[3], h[4], h_out, d[3], d[4], dl.softmax_scale,
                                 ws2, out2, copy, direct_out=direct)
        torch.cuda.current_stream().synchronize()
        assert msa.msa_read_device_status(ws2) == msa.MSA_OK
        assert torch.equal(h_out.view(torch.int16), ref), case
        h_out.fill_(7)


def test_host_step_rejects_pageable_buffers(msa):
    from workloads.device import DeviceLayer

    w = W.small("pageable", seq_lens=[1000, 300], q_lens=[1, 1], seed=44)
    dl = DeviceLayer(w, 0)
    o = dl.outputs()
    ws = dl.workspace()
    b = dl.batch
    pageable = [x.cpu().contiguous() for x in (b.query_start_loc, b.seq_lens, b.block_table, dl.q8, dl.iq8)]
    out_h = torch.empty(tuple(o["out"].shape), dtype=o["out"].dtype)
    with pytest.raises(ValueError):
        msa.msa_decode_step_host(b, dl.cache, *pageable, out_h, dl.q8, dl.iq8, dl.softmax_scale, ws, o["out"],
                                 torch.cuda.Stream())
    # the library's own check, past the binding's
    io = msa.msa_host_step_io(*(x.data_ptr() for x in pageable), out_h.data_ptr())
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for flags in (0, msa.MSA_HOST_STEP_DIRECT_OUT):
        code = msa._lib.msa_decode_step_host(ctypes.byref(msa.GEOMETRY), ctypes.byref(b.c), ctypes.byref(dl.cache.c),
                                             ctypes.byref(io), msa._ptr(dl.q8), msa._ptr(dl.iq8),
                                             float(dl.softmax_scale), msa._ptr(ws), ws.numel(), msa._ptr(o["out"]),
                                             flags, s, s)
        assert code == msa.MSA_ERR_INVALID_ARG
    # pinned inputs but a pageable output: the direct mode has nowhere to store
    pinned_in = [x.pin_memory() for x in pageable]
    io2 = msa.msa_host_step_io(*(x.data_ptr() for x in pinned_in), out_h.data_ptr())
    code = msa._lib.msa_decode_step_host(ctypes.byref(msa.GEOMETRY), ctypes.byref(b.c), ctypes.byref(dl.cache.c),
                                         ctypes.byref(io2), msa._ptr(dl.q8), msa._ptr(dl.iq8), float(dl.softmax_scale),
                                         msa._ptr(ws), ws.numel(), None, msa.MSA_HOST_STEP_DIRECT_OUT, s, s)
    assert code == msa.MSA_ERR_INVALID_ARG


@pytest.mark.parametrize("direct", [False, True])
def test_host_step_in_a_cuda_graph(msa, direct):
    """msa_decode_step_host captured once (both streams, the copies and the kernels) replays with
    new host contents and equals msa_decode_step on them."""
    from workloads.device import DeviceLayer

    case = "tc_split"
    w = W.small(case, **CASES[case])
    dl = DeviceLayer(w, 0)
    b = dl.batch
    h = [pinned(x) for x in (b.query_start_loc, b.seq_lens, b.block_table, dl.q8, dl.iq8)]
    o = dl.outputs()
    h_out = torch.zeros(tuple(o["out"].shape), dtype=o["out"].dtype).pin_memory()
    d = [torch.zeros_like(x) for x in (b.query_start_loc, b.seq_lens, b.block_table, dl.q8, dl.iq8)]
    batch2 = msa.Batch(d[0], d[1], d[2], b.max_q_len, T=b.T)
    out2 = None if direct else torch.zeros_like(o["out"])
    ws2 = dl.workspace()
    copy = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            msa.msa_decode_step_host(batch2, dl.cache, h[0], h[1], h[2], h[3], h[4], h_out, d[3], d[4],
                                     dl.softmax_scale, ws2, out2, copy, direct_out=direct)
    torch.cuda.current_stream().wait_stream(s)
    for it in range(2):
        if it == 1:  # new query contents on the host, same graph
            h[3].copy_(torch.roll(h[3], 1, dims=1))
            dl.q8.copy_(h[3])
        ws = dl.workspace()
        msa.msa_decode_step(dl.batch, dl.cache, dl.q8, dl.iq8, dl.softmax_scale, ws, o["out"])
        torch.cuda.synchronize()
        ref = o["out"].view(torch.int16).cpu()
        h_out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert msa.msa_read_device_status(ws2) == msa.MSA_OK
        assert torch.equal(h_out.view(torch.int16), ref), it
