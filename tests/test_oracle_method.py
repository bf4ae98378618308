"""Pins of the oracle's method steps (indexer, selection, attention) and byte arithmetic.

Each step is checked against something other than itself:
* indexer: a numpy fp64 matmul over torch-decoded FP8 keys, with the block max-pool and the
  causal / partial-block masks written as index arithmetic over positions;
* selection: rank counting (an O(n^2) brute force, not a sort), the equivalent "top-16 over
  all blocks with the local block forced in" formulation, and permutation invariance;
* attention: a textbook numpy softmax attention over the gathered selected keys, and the
  dense special case (context <= 2,048 tokens: every block selected, so MSA is dense causal
  GQA attention);
* byte arithmetic: the sizes printed on the pages (tests/golden/byte_arithmetic.json).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

D, G, HPG, H, BS = 128, 4, 16, 64, 128


def fp8_values(b):
    t = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return t[np.asarray(b, dtype=np.uint8)]


def rand_fp8(rng, shape, scale=1.0):
    x = (rng.standard_normal(shape) * scale).astype(np.float32)
    return torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def rand_nvfp4(orc, rng, shape):
    x = rng.standard_normal(shape).astype(np.float32)
    return orc.quantize_nvfp4(x)


# ------------------------------------------------------------------------------ indexer
@pytest.mark.parametrize("index_dtype", [0, 1])
@pytest.mark.parametrize("L,q_len", [(700, 3), (128, 1), (129, 2), (1000, 8)])
def test_indexer_matches_numpy(orc, index_dtype, L, q_len):
    rng = np.random.default_rng(L * 10 + q_len + index_dtype)
    iq = rand_fp8(rng, (q_len, G, D))
    if index_dtype == 0:
        vals, scales = rand_nvfp4(orc, rng, (L, D))
        keys = fp8_values(orc.dequant_nvfp4(vals, scales))
    else:
        vals, scales = rand_fp8(rng, (L, D)), None
        keys = fp8_values(vals)
    got = orc.indexer_seq(L, q_len, iq, index_dtype, vals, scales)
    s = fp8_values(iq).reshape(q_len * G, D) @ keys.T  # [q_len*4, L]
    nb = -(-L // BS)
    j = np.arange(L)
    for t in range(q_len):
        p = L - q_len + t
        for g in range(G):
            row = s[t * G + g]
            for k in range(nb):
                m = (j // BS == k) & (j <= p)
                want = row[m].max() if m.any() else -np.inf
                assert got[t, g, k] == pytest.approx(want, rel=1e-12, abs=1e-12), (t, g, k)


# ---------------------------------------------------------------------------- selection
def rank_count_select(scores, local):
    """Brute force: block i is ranked by how many candidates beat it (higher score, or the
    same score and a lower id). NaN ranks as -inf."""
    s = np.where(np.isnan(scores[:local]), -np.inf, scores[:local])
    n = len(s)
    rank = [sum(1 for j in range(n) if s[j] > s[i] or (s[j] == s[i] and j < i)) for i in range(n)]
    order = sorted(range(n), key=lambda i: rank[i])
    picked = [i for i in order if rank[i] < 15]
    return [local] + picked + [-1] * (15 - len(picked))


def forced_local_select(scores, local):
    """Alternative reading: top-16 over blocks 0..local (local scored too), then force local in
    without double counting; returns the set."""
    s = np.where(np.isnan(scores[:local + 1]), -np.inf, scores[:local + 1])
    order = sorted(range(local + 1), key=lambda i: (-s[i], i))
    top = order[:16]
    if local not in top:
        top = top[:15] + [local]
    return set(top)


@pytest.mark.parametrize("seed", range(6))
def test_select_bruteforce(orc, seed):
    rng = np.random.default_rng(seed)
    nb = int(rng.integers(1, 60))
    local = int(rng.integers(0, nb))
    # integer-valued scores force many ties
    scores = rng.integers(-5, 6, size=nb).astype(np.float64)
    if seed % 2:
        scores[rng.integers(0, nb, size=3)] = np.nan
        scores[rng.integers(0, nb, size=2)] = -np.inf
    got = orc.select_row(scores, local).tolist()
    assert got == rank_count_select(scores, local)
    assert set(x for x in got if x >= 0) == forced_local_select(scores, local)


@pytest.mark.parametrize("seed", range(4))
def test_select_alternative_formulation(orc, seed):
    rng = np.random.default_rng(100 + seed)
    nb = 64
    local = 50
    scores = rng.standard_normal(nb)
    scores[local] = 10.0 if seed % 2 else -10.0  # the local block ranks first / last
    got = set(int(x) for x in orc.select_row(scores, local) if x >= 0)
    assert got == forced_local_select(scores, local)
    assert len(got) == 16


def test_select_permutation_and_ties(orc):
    rng = np.random.default_rng(9)
    nb, local = 40, 39
    scores = rng.standard_normal(nb)
    perm = rng.permutation(local)
    sel = orc.select_row(scores, local)
    scores_p = scores.copy()
    scores_p[perm] = scores[:local]  # block i moves to perm[i]
    sel_p = orc.select_row(scores_p, local)
    assert sel_p[0] == local
    assert sel_p[1:].tolist() == [int(perm[i]) for i in sel[1:]]
    # all equal -> lowest ids first
    eq = np.zeros(nb)
    assert orc.select_row(eq, local)[1:].tolist() == list(range(15))
    # fewer than 15 candidates -> all of them, then -1
    assert orc.select_row(scores, 5).tolist()[6:] == [-1] * 10
    assert orc.select_row(scores, 0).tolist() == [0] + [-1] * 15


# ---------------------------------------------------------------------------- attention
def textbook_attention(q8, kd, vd, L, q_len, blocks_per_tg, scale):
    """numpy fp64 softmax attention of every head over its group's gathered keys.
    kd, vd: decoded FP8 values [L, G, D]."""
    out = np.zeros((q_len, H, D))
    for t in range(q_len):
        p = L - q_len + t
        for g in range(G):
            blocks = sorted(set(b for b in blocks_per_tg[t][g] if b >= 0))
            j = np.array([x for b in blocks for x in range(b * BS, min((b + 1) * BS, L)) if x <= p])
            K = kd[j, g]
            V = vd[j, g]
            for hh in range(HPG):
                h = g * HPG + hh
                z = scale * (K @ fp8_values(q8[t, h]))
                w = np.exp(z - z.max())
                out[t, h] = (w[:, None] * V).sum(0) / w.sum()
    return out


def build_kv(orc, rng, L, outliers=False):
    k = rng.standard_normal((L, G, D)).astype(np.float32)
    v = rng.standard_normal((L, G, D)).astype(np.float32)
    if outliers:
        k[:, :, :3] *= 8
    kv_, ks_ = orc.quantize_nvfp4(k)
    vv_, vs_ = orc.quantize_nvfp4(v)
    return kv_, ks_, vv_, vs_


def decoded(orc, vals, scales):
    return fp8_values(orc.dequant_nvfp4(vals, scales))


@pytest.mark.parametrize("L,q_len,seed", [(3000, 1, 0), (2500, 4, 1), (777, 3, 2)])
def test_attention_matches_textbook(orc, L, q_len, seed):
    rng = np.random.default_rng(seed)
    kv = build_kv(orc, rng, L, outliers=seed == 1)
    q8 = rand_fp8(rng, (q_len, H, D))
    nb = -(-L // BS)
    sel = np.full((q_len, G, 16), -1, np.int32)
    for t in range(q_len):
        local = (L - q_len + t) // BS
        for g in range(G):
            others = rng.choice(max(local, 1), size=min(local, int(rng.integers(1, 16))), replace=False) if local else []
            row = [local] + list(others)
            sel[t, g, :len(row)] = row
    kd = decoded(orc, kv[0], kv[1])  # [L, G, D]
    vd = decoded(orc, kv[2], kv[3])
    scale = 1 / math.sqrt(D)
    got = orc.attention_seq(L, q_len, q8, *kv, sel, scale)
    want = textbook_attention(q8, kd, vd, L, q_len, sel.tolist(), scale)
    np.testing.assert_allclose(got, want, rtol=1e-10, atol=1e-12)
    assert nb >= 1


@pytest.mark.parametrize("L,q_len", [(2048, 1), (2048, 8), (1500, 5), (130, 2)])
def test_dense_special_case(orc, L, q_len):
    """Context <= 2,048 tokens: MSA selects every block and equals dense causal GQA."""
    rng = np.random.default_rng(L + q_len)
    iq = rand_fp8(rng, (q_len, G, D))
    ik = rand_nvfp4(orc, rng, (L, D))
    kv = build_kv(orc, rng, L)
    q8 = rand_fp8(rng, (q_len, H, D))
    scale = 1 / math.sqrt(D)
    _, sels, outs = orc.decode_batch([L], [q_len], [iq], [q8], 0, [ik], [kv], scale)
    sel = sels[0]
    for t in range(q_len):
        local = (L - q_len + t) // BS
        for g in range(G):
            assert sorted(x for x in sel[t, g] if x >= 0) == list(range(local + 1))
    kd = decoded(orc, kv[0], kv[1])
    vd = decoded(orc, kv[2], kv[3])
    want = np.zeros((q_len, H, D))
    for t in range(q_len):
        p = L - q_len + t
        for h in range(H):
            g = h // HPG
            z = scale * (kd[:p + 1, g] @ fp8_values(q8[t, h]))
            w = np.exp(z - z.max())
            want[t, h] = (w[:, None] * vd[:p + 1, g]).sum(0) / w.sum()
    np.testing.assert_allclose(outs[0], want, rtol=1e-10, atol=1e-12)


def test_key_cap_2048(orc):
    rng = np.random.default_rng(21)
    L, q_len = 9000, 4
    iq = rand_fp8(rng, (q_len, G, D))
    ik = rand_nvfp4(orc, rng, (L, D))
    s = orc.indexer_seq(L, q_len, iq, 0, *ik)
    sel = orc.select_seq(s, L, q_len)
    for t in range(q_len):
        p = L - q_len + t
        for g in range(G):
            blocks = set(int(b) for b in sel[t, g] if b >= 0)
            keys = sum(1 for b in blocks for j in range(b * BS, min((b + 1) * BS, L)) if j <= p)
            assert len(blocks) == 16 and keys <= 2048
            assert p // BS in blocks


# ----------------------------------------------------------------------- byte arithmetic
def test_byte_arithmetic(orc, golden_dir):
    g = {e["name"]: e["value"] for e in json.load(open(os.path.join(golden_dir, "byte_arithmetic.json")))["entries"]}
    layers = g["layers"]
    kv_nvfp4 = orc.GROUPS * 2 * (orc.ROW_CODE_BYTES + orc.ROW_SCALE_BYTES)   # K and V, 4 heads
    kv_fp8 = orc.GROUPS * 2 * orc.HEAD_DIM
    idx_nvfp4 = orc.ROW_CODE_BYTES + orc.ROW_SCALE_BYTES
    idx_fp8 = orc.INDEX_PAGE_BYTES[orc.INDEX_FP8] // orc.BLOCK
    assert idx_fp8 == g["index_bytes_per_token_per_layer_fp8"]
    assert kv_fp8 == g["dense_fp8_kv_bytes_per_token_per_layer"]
    assert layers * kv_nvfp4 == g["nvfp4_kv_bytes_per_token_all_layers"]
    assert layers * kv_fp8 == g["fp8_kv_bytes_per_token_all_layers"]
    assert 1 - kv_nvfp4 / kv_fp8 == g["kv_saving_fraction"]
    assert idx_fp8 / kv_fp8 == g["index_to_dense_ratio"] == idx_nvfp4 / kv_nvfp4
    assert orc.K_SEL * orc.BLOCK == g["keys_per_query_cap"]
    assert idx_nvfp4 * 8 / orc.HEAD_DIM == g["nvfp4_bits_per_element"]
    assert orc.dequant_table()[:, :8].nbytes == g["dequant_table_bytes"]
    # the page sizes the layout implies, and the oracle's codec output sizes
    assert orc.INDEX_PAGE_BYTES[orc.INDEX_NVFP4] == orc.BLOCK * idx_nvfp4 == 9216
    assert orc.KV_PAGE_BYTES == orc.BLOCK * kv_nvfp4 == 73728
    vals, scales = orc.quantize_nvfp4(np.ones((10, 128), np.float32))
    assert vals.nbytes + scales.nbytes == 10 * idx_nvfp4


def test_page_gather_scatter_roundtrip(orc):
    rng = np.random.default_rng(4)
    L = 300
    nb = 3
    table = np.array([5, 1, 3], np.int32)
    vals, scales = rand_nvfp4(orc, rng, (L, D))
    pages = np.zeros(6 * orc.INDEX_PAGE_BYTES[0], np.uint8)
    orc.scatter_index_rows(pages, table, vals, scales, 0)
    v2, s2 = orc.gather_index_rows(pages, table, L, 0)
    assert np.array_equal(v2, vals) and np.array_equal(s2, scales)
    kv = build_kv(orc, rng, L)
    kvp = np.zeros(6 * orc.KV_PAGE_BYTES, np.uint8)
    orc.scatter_kv_rows(kvp, table, *kv)
    for a, b in zip(orc.gather_kv_rows(kvp, table, L), kv):
        assert np.array_equal(a, b)
    # the codes of token 130 (block 1 -> page 1, row 2) of head 2's V sit where the layout says
    off = orc.kv_region_offset(1, 2, 1) + 2 * orc.ROW_CODE_BYTES
    assert np.array_equal(kvp[off:off + 64], kv[2][130, 2])
    assert nb == 3
