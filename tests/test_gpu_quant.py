"""GPU parity of the cache producers and the dequantiser: bit-exact against the oracle."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from parity import seq_sources

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def msa():
    import nvfp4_kv_cache_gb300 as m

    return m


def gpu_quant_nvfp4(msa, x: np.ndarray, vstride=None, sstride=None):
    rows, cols = x.shape
    vs = vstride or cols // 2
    ss = sstride or cols // 16
    xd = torch.from_numpy(np.ascontiguousarray(x, np.float32)).cuda()
    vals = torch.full((rows, vs), 0xAB, dtype=torch.uint8, device="cuda")
    scales = torch.full((rows, ss), 0xCD, dtype=torch.uint8, device="cuda")
    msa.msa_quantize_nvfp4(xd, vals, scales, vs, ss)
    torch.cuda.synchronize()
    return vals.cpu().numpy(), scales.cpu().numpy()


def edge_rows(rng):
    rows = [np.zeros(128, np.float32)]
    hand = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "nvfp4_hand_vectors.json")))
    for v in hand["vectors"]:
        rows.append(np.tile(np.array(v["x"], np.float32), 8))
    for scale in (1e-6, 1e-3, 0.05, 1.0, 37.0, 1000.0, 3e4):
        rows.append((rng.standard_normal(128) * scale).astype(np.float32))
    # every E2M1 tie point for several scales, and values just around them
    ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0], np.float32)
    for S in (1.0, 0.5, 2.0 ** -9, 448.0 / 6):
        r = np.concatenate([ties, -ties, np.nextafter(ties, 0), np.nextafter(ties, 10)]).astype(np.float32)
        row = np.tile(r, 4)[:128] * np.float32(S)
        row[::16] = np.float32(6.0 * S)  # pins amax so the scale is S
        rows.append(row.astype(np.float32))
    return np.stack(rows)


@pytest.mark.parametrize("shape", [(1, 16), (37, 128), (1000, 128), (5, 4096), (129, 48)])
def test_quantize_nvfp4_bitexact(msa, shape):
    rng = np.random.default_rng(shape[0] * 7 + shape[1])
    x = rng.standard_normal(shape).astype(np.float32)
    x[:, :: max(1, shape[1] // 5)] *= 8  # outlier channels
    v, s = gpu_quant_nvfp4(msa, x)
    rv, rs = oracle.quantize_nvfp4(x)
    assert np.array_equal(s, rs)
    assert np.array_equal(v, rv)


def test_quantize_nvfp4_edges_and_strides(msa):
    rng = np.random.default_rng(1)
    x = edge_rows(rng)
    v, s = gpu_quant_nvfp4(msa, x, vstride=80, sstride=12)
    rv, rs = oracle.quantize_nvfp4(x)
    assert np.array_equal(s[:, :8], rs)
    assert np.array_equal(v[:, :64], rv)
    assert (v[:, 64:] == 0xAB).all() and (s[:, 8:] == 0xCD).all()  # strides respected


@pytest.mark.parametrize("n,offset", [(1, 0), (4093, 0), (100000, 0), (1001, 1)])
def test_quantize_fp8_bitexact(msa, n, offset):
    rng = np.random.default_rng(n)
    x = (rng.standard_normal(n + offset) * 8).astype(np.float32)
    specials = np.array([0.0, -0.0, 448.0, -448.0, 449.0, 464.0, 1e9, -1e9, 2.0 ** -10, -(2.0 ** -10),
                         1.5 * 2.0 ** -10, 2.0 ** -9, 1e-30, 0.09375, 17.0, 18.0], np.float32)
    x[: min(len(specials), n)] = specials[: min(len(specials), n)]
    xd = torch.from_numpy(x).cuda()[offset:]
    out = torch.empty(n + 1, dtype=torch.uint8, device="cuda")[1:] if offset else torch.empty(n, dtype=torch.uint8,
                                                                                             device="cuda")
    msa.msa_quantize_fp8(xd.contiguous() if not offset else xd, out)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), oracle.quantize_fp8(x[offset:]))


def test_dequant_all_scale_code_pairs(msa):
    """All 4,096 (scale byte, code) pairs against the oracle's table."""
    codes = np.tile(np.arange(16, dtype=np.uint8), (256, 1))  # row s: codes 0..15
    vals = oracle.pack_nvfp4(codes)                          # [256, 8]
    scales = np.arange(256, dtype=np.uint8)[:, None]         # [256, 1]
    out = torch.empty((256, 16), dtype=torch.uint8, device="cuda")
    msa.msa_dequant_nvfp4(torch.from_numpy(vals).cuda(), torch.from_numpy(scales).cuda(), out)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), oracle.dequant_table())


def test_dequant_random_rows(msa):
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((333, 128)) * rng.uniform(0.01, 50, (333, 1))).astype(np.float32)
    vals, scales = oracle.quantize_nvfp4(x)
    out = torch.empty((333, 128), dtype=torch.uint8, device="cuda")
    msa.msa_dequant_nvfp4(torch.from_numpy(vals).cuda(), torch.from_numpy(scales).cuda(), out)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), oracle.dequant_nvfp4(vals, scales))


@pytest.mark.parametrize("index_dtype", [0, 1])
def test_kv_insert_paged_bitexact(msa, index_dtype):
    from workloads.device import DeviceLayer

    w = W.small("insert", [16384 + 300, 16384 + 129, 5000], [2, 1, 3], seed=11, index_dtype=index_dtype,
                prefix_len=16384, prefix_seqs=2)
    dl = DeviceLayer(w, 0)
    assert msa.status_bits(dl.status) == 0
    kv = dl.cache.kv_pages.cpu().numpy()
    ix = dl.cache.index_pages.cpu().numpy()
    for b in range(w.B):
        L = w.seq_lens[b]
        _, _, ik, k, v = seq_sources(w, 0, b, "cuda")
        gv, gs = oracle.gather_index_rows(ix, w.block_table[b], L, index_dtype)
        if index_dtype == 0:
            rv, rs = oracle.quantize_nvfp4(ik)
            assert np.array_equal(gv, rv) and np.array_equal(gs, rs), b
        else:
            assert np.array_equal(gv, oracle.quantize_fp8(ik)), b
        got = oracle.gather_kv_rows(kv, w.block_table[b], L)
        want = oracle.quantize_nvfp4(k) + oracle.quantize_nvfp4(v)
        for g_, w_ in zip(got, want):
            assert np.array_equal(g_, w_), b


def test_kv_insert_skips_and_faults(msa):
    cache = msa.Cache.empty(2, 0)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    n = 4
    k = torch.randn(n, 4, 128, device="cuda")
    v = torch.randn(n, 4, 128, device="cuda")
    ik = torch.randn(n, 128, device="cuda")
    slots = torch.tensor([0, -1, 2 * 128 + 5, 255], dtype=torch.int64, device="cuda")  # ok, skip, bad, ok
    msa.msa_kv_insert(k, v, ik, slots, cache, status)
    torch.cuda.synchronize()
    assert msa.status_bits(status) == (1 << msa.MSA_ERR_DEVICE_FAULT)
    kvp = cache.kv_pages.cpu().numpy()
    kq = oracle.quantize_nvfp4(k.cpu().numpy())
    got = oracle.gather_kv_rows(kvp, [0, 1], 256)
    assert np.array_equal(got[0][0], kq[0][0]) and np.array_equal(got[0][255], kq[0][3])
    assert (got[0][1:255] == 0).all()  # the skipped and the faulting tokens wrote nothing
