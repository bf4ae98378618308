"""Pins of the oracle's number formats and NVFP4 codec against values it does not produce.

* E4M3 decode: torch's float8_e4m3fn conversion table (an independent library routine).
* E4M3 encode: torch's round-to-nearest-even cast where it is defined (|x| <= 448) and a
  brute-force nearest-value search everywhere, plus hand cases for saturation and zero.
* E2M1: the magnitude list of the FP4 format and a brute-force nearest search.
* Dequant-to-FP8 table (256 scales x 16 codes): torch's cast of the exact product.
* NVFP4 quantisation: hand-derived vectors (tests/golden/nvfp4_hand_vectors.json) and the
  half-spacing error bound of round-to-nearest.
"""
import json
import os

import numpy as np
import pytest
import torch

E2M1_MAGS = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def torch_e4m3_table():
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def torch_e4m3_cast(x32: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.asarray(x32, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def representable_e4m3():
    t = torch_e4m3_table()
    codes = np.array([c for c in range(128) if not np.isnan(t[c])])
    return codes, t[codes]


def brute_e4m3(x: float) -> int:
    """Nearest finite E4M3 value, ties to even code, saturating; independent search."""
    codes, vals = representable_e4m3()
    sign = 0x80 if np.signbit(x) else 0
    a = min(abs(x), 448.0)
    err = np.abs(vals - a)
    best = np.flatnonzero(err == err.min())
    c = int(codes[best[0]]) if len(best) == 1 else int(codes[best][codes[best] % 2 == 0][0])
    return sign | c


def test_e4m3_decode_matches_torch(orc):
    ours = orc.e4m3_decode(np.arange(256))
    ref = torch_e4m3_table()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])
    assert np.flatnonzero(np.isnan(ours)).tolist() == [0x7F, 0xFF]
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9 and ours[0x38] == 1.0


def test_e4m3_encode_random_vs_torch_and_bruteforce(orc):
    rng = np.random.default_rng(7)
    mag = np.exp2(rng.uniform(-12, np.log2(448), 4000)).astype(np.float32)
    x = (mag * rng.choice([-1, 1], mag.size)).astype(np.float32)
    ours = orc.e4m3_encode(x.astype(np.float64))
    assert np.array_equal(ours, torch_e4m3_cast(x))
    for v, o in zip(x[:400], ours[:400]):
        assert brute_e4m3(float(v)) == int(o)


def test_e4m3_encode_ties_and_edges(orc):
    codes, vals = representable_e4m3()
    mids = ((vals[1:] + vals[:-1]) / 2).astype(np.float32)  # exact halfway points
    ours = orc.e4m3_encode(mids.astype(np.float64))
    assert np.array_equal(ours, torch_e4m3_cast(mids))
    for m, o in zip(mids, ours):
        assert int(o) % 2 == 0, "a tie must go to the even mantissa"
        assert brute_e4m3(float(m)) == int(o)
    hand = [(448.0, 0x7E), (449.0, 0x7E), (500.0, 0x7E), (1e30, 0x7E), (-500.0, 0xFE),
            (2.0 ** -10, 0x00), (1.5 * 2.0 ** -10, 0x01), (2.0 ** -9, 0x01), (-0.0, 0x80), (0.0, 0x00),
            (-1e-9, 0x80), (1.0, 0x38), (0.0625 * 1.5, 0x1C)]
    for x, want in hand:
        assert int(orc.e4m3_encode([x])[0]) == want, x
    assert int(orc.e4m3_encode([float("nan")])[0]) & 0x7F == 0x7F


def test_e2m1_decode_table(orc):
    ref = E2M1_MAGS + [-m for m in E2M1_MAGS]
    ours = orc.e2m1_decode(np.arange(16))
    assert np.array_equal(ours, np.array(ref))
    assert np.signbit(ours[8])


def test_e2m1_encode_bruteforce(orc):
    rng = np.random.default_rng(3)
    r = np.concatenate([rng.uniform(-7, 7, 3000), [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.5, 100.0, -0.0]])
    r = r.astype(np.float32)
    ours = orc.e2m1_encode(r)
    mags = np.array(E2M1_MAGS)
    for v, o in zip(r, ours):
        a = min(abs(float(v)), 6.0)
        err = np.abs(mags - a)
        cand = np.flatnonzero(err == err.min())
        c = int(cand[0]) if len(cand) == 1 else int([k for k in cand if k % 2 == 0][0])
        want = 0 if c == 0 else ((8 if v < 0 else 0) | c)
        assert int(o) == want, (v, o, want)
    ties = {0.25: 0, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6, -0.25: 0, -5.0: 14, 7.0: 7}
    for v, want in ties.items():
        assert int(orc.e2m1_encode([v])[0]) == want, v


def test_dequant_table_matches_torch_products(orc):
    """E4M3_RNE_sat(E2M1(c) * E4M3(s)) for all 4,096 (scale, code) pairs."""
    tab = orc.dequant_table()
    scales = torch_e4m3_table()
    fp4 = np.array(E2M1_MAGS + [-m for m in E2M1_MAGS])
    fp4[8] = -0.0
    for s in range(256):
        prod = (fp4 * scales[s]).astype(np.float32)  # exact: at most 5 significant bits
        for c in range(16):
            got = int(tab[s, c])
            sign = (c >> 3) ^ (s >> 7)
            if np.isnan(scales[s]):
                assert got == (0x7F | (sign << 7)), (s, c)
            elif abs(prod[c]) > 448:
                assert got == (0x7E | (sign << 7)), (s, c)
            else:
                assert got == int(torch_e4m3_cast(prod[c:c + 1])[0]), (s, c, prod[c])
    # the 2 KB table of pre-rounded FP8 values: 256 scales x 8 magnitudes, sign applied after
    pos = tab[:, :8]
    assert pos.size == 2048
    assert np.array_equal(tab[:128, 8:] & 0x7F, pos[:128] & 0x7F)


def test_nvfp4_hand_vectors(orc, golden_dir):
    g = json.load(open(os.path.join(golden_dir, "nvfp4_hand_vectors.json")))
    for v in g["vectors"]:
        x = np.array(v["x"], dtype=np.float32)[None, :]
        vals, scales = orc.quantize_nvfp4(x)
        assert int(scales[0, 0]) == v["scale"], v["name"]
        assert orc.unpack_nvfp4(vals)[0].tolist() == v["codes"], v["name"]


def test_pack_layout_hand_words(orc, golden_dir):
    g = json.load(open(os.path.join(golden_dir, "nvfp4_hand_vectors.json")))
    for case in g["pack_words"]["cases"]:
        codes = np.array(case["codes"] * 2, dtype=np.uint8)[None, :]  # two words
        vals = orc.pack_nvfp4(codes)
        word = int.from_bytes(bytes(vals[0, :4]), "little")
        assert word == int(case["word"], 16), case
        assert np.array_equal(orc.unpack_nvfp4(vals), codes)


def test_pack_unpack_roundtrip(orc):
    rng = np.random.default_rng(11)
    codes = rng.integers(0, 16, size=(37, 128), dtype=np.uint8)
    assert np.array_equal(orc.unpack_nvfp4(orc.pack_nvfp4(codes)), codes)


@pytest.mark.parametrize("outliers", [False, True])
def test_nvfp4_error_bound(orc, outliers):
    """|x/S - E2M1(code)| <= half the spacing of E2M1 around x/S, unless saturated at 6."""
    rng = np.random.default_rng(5 + outliers)
    x = rng.standard_normal((400, 128)).astype(np.float32)
    if outliers:
        x[:, rng.choice(128, 5, replace=False)] *= 8
    vals, scales = orc.quantize_nvfp4(x)
    codes = orc.unpack_nvfp4(vals)
    S = np.repeat(orc.e4m3_decode(scales), 16, axis=1)
    q = orc.e2m1_decode(codes)
    r = (x / S.astype(np.float32)).astype(np.float64)
    a = np.abs(r)
    half = np.where(a < 2, 0.25, np.where(a < 4, 0.5, 1.0))
    sat = a > 6
    assert np.all(np.abs(r - q)[~sat] <= half[~sat])
    assert np.all(np.abs(q[sat]) == 6.0)
    assert np.all(S > 0)
    # the scale is E4M3(amax/6): the largest element of each group maps near the top code
    amax = np.abs(x).reshape(400, 8, 16).max(-1)
    want = orc.e4m3_encode((amax / np.float32(6)).astype(np.float32).astype(np.float64))
    assert np.array_equal(want.reshape(scales.shape), scales)


def test_quantize_fp8_matches_torch(orc):
    rng = np.random.default_rng(2)
    x = rng.standard_normal(5000).astype(np.float32) * 4
    assert np.array_equal(orc.quantize_fp8(x), torch_e4m3_cast(x))
