"""GPU parity of the exact-score indexer variant (msa_indexer_decode_exact: NVFP4 index keys
converted straight to f16 and scored with an f16 MMA, no E4M3 re-rounding — "vLLM ofrece
soporte en día 0 para MiniMax-M3.1-Flash", "NVIDIA Rubin MSA optimizado") against the oracle's
exact mode, on small ragged cases and sampled sequences of the full-size decode workload."""
import numpy as np
import pytest
import torch

import workloads as W
from parity import OracleSeq, check_scores

pytestmark = pytest.mark.gpu

CASES = {
    "ragged": dict(seq_lens=[1000, 4096 + 77, 300], q_lens=[1, 8, 3], seed=51),
    "hot": dict(seq_lens=[6000, 9000 + 5], q_lens=[8, 2], seed=52, hot=12),
    "padded": dict(seq_lens=[4000, 0, 2500, 700, 1], q_lens=[2, 0, 0, 1, 1], seed=53),
    "outliers": dict(seq_lens=[5000, 129], q_lens=[4, 1], seed=54, outlier_frac=0.01),
}


@pytest.fixture(scope="module")
def msa():
    import nvfp4_kv_cache_gb300 as m

    return m


def _exact(msa, dl):
    T = dl.batch.T
    out = torch.full((T, 4, dl.batch.max_blocks), float("nan"), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    msa.msa_indexer_decode_exact(dl.batch, dl.cache, dl.iq8, out, st)
    torch.cuda.synchronize()
    assert msa.status_bits(st) == 0
    return out.cpu().numpy()


def _compare(w, scores, seqs):
    qsl = w.query_start_loc()
    n = 0
    for b in seqs:
        ql, L = w.q_lens[b], w.seq_lens[b]
        if ql == 0:
            continue
        nb = (L + 127) // 128
        ref = OracleSeq(w, 0, b, "cuda", kv_blocks=np.zeros(0, np.int64)).scores_exact()
        check_scores(scores[qsl[b]:qsl[b] + ql, :, :nb], ref, f"seq {b}")
        n += 1
    return n


@pytest.mark.parametrize("case", sorted(CASES))
def test_exact_scores_match_the_oracle(msa, case):
    from workloads.device import DeviceLayer

    w = W.small(case, **CASES[case])
    dl = DeviceLayer(w, 0)
    assert _compare(w, _exact(msa, dl), range(w.B)) > 0


def test_exact_differs_from_e4m3_scores_and_fp8_cache_is_unchanged(msa):
    from workloads.device import DeviceLayer

    w = W.small("nv", [3000, 2000], [2, 1], seed=55)
    dl = DeviceLayer(w, 0)
    ex = _exact(msa, dl)
    T = dl.batch.T
    rer = torch.empty((T, 4, dl.batch.max_blocks), dtype=torch.float32, device="cuda")
    msa.msa_indexer_decode(dl.batch, dl.cache, dl.iq8, rer, None)
    torch.cuda.synchronize()
    nb0 = (w.seq_lens[0] + 127) // 128
    assert not np.array_equal(ex[:2, :, :nb0], rer.cpu().numpy()[:2, :, :nb0])  # E4M3 re-rounding shows
    # an FP8 index cache has nothing to re-round: both entry points give the same bits
    w8 = W.small("fp8", [3000, 2000], [2, 1], seed=56, index_dtype=1)
    d8 = DeviceLayer(w8, 0)
    a = _exact(msa, d8)
    b = torch.empty((d8.batch.T, 4, d8.batch.max_blocks), dtype=torch.float32, device="cuda")
    msa.msa_indexer_decode(d8.batch, d8.cache, d8.iq8, b, None)
    torch.cuda.synchronize()
    for s, (L, ql) in enumerate(zip(w8.seq_lens, w8.q_lens)):
        r = slice(w8.query_start_loc()[s], w8.query_start_loc()[s] + ql)
        nb = (L + 127) // 128
        assert np.array_equal(a[r, :, :nb].view(np.uint32), b.cpu().numpy()[r, :, :nb].view(np.uint32))


def test_exact_full_size_decode_sampled(msa):
    """B = 32 sequences of 32K tokens (the decode workload), two sequences checked."""
    from workloads.device import DeviceLayer

    w = W.CONFIGS["decode"]()
    dl = DeviceLayer(w, 0)
    assert _compare(w, _exact(msa, dl), [0, 31]) == 2
    del dl
    torch.cuda.empty_cache()
