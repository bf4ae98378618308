"""Pins of the oracle's exact-score indexer mode (NVFP4 index keys taken as E2M1 x E4M3
exactly, with no re-rounding to E4M3 — "vLLM ofrece soporte en día 0 para
MiniMax-M3.1-Flash", "NVIDIA Rubin MSA optimizado").

* With power-of-two scales every E2M1 x scale product is an E4M3 value, so the exact mode must
  equal the (separately pinned) E4M3 mode bit for bit.
* Hand-worked products where E4M3 must round: 6 x 1.125 = 6.75 is a tie between the E4M3
  neighbours 6.5 and 7, and round-to-nearest-even gives 7; the exact mode keeps 6.75.
* Signs multiply (a negative code times a negative scale is positive); a NaN scale's keys are
  passed over by the block maximum.
"""
import numpy as np

import oracle

E4M3_ONE = 0x38      # 1.0
E4M3_1_125 = 0x39    # 1.125 = (1 + 1/8) x 2^0
E2M1_SIX = 0x7       # magnitude code of 6.0
E2M1_NEG_SIX = 0xF   # sign bit + 6.0


def _one_key(code: int, scale: int, dim: int = 0):
    codes = np.zeros((1, 128), dtype=np.uint8)
    codes[0, dim] = code
    scales = np.zeros((1, 8), dtype=np.uint8)
    scales[0, dim // 16] = scale
    return oracle.pack_nvfp4(codes), scales


def _iq_unit(dim: int = 0):
    iq = np.zeros((1, 4, 128), dtype=np.uint8)
    iq[0, 0, dim] = E4M3_ONE
    return iq


def test_power_of_two_scales_match_the_e4m3_mode_exactly():
    rng = np.random.default_rng(3)
    L, q_len = 300, 2
    codes = rng.integers(0, 16, size=(L, 128)).astype(np.uint8)
    vals = oracle.pack_nvfp4(codes)
    # 2^k for k in [-8, 6]: E2M1 magnitudes (0.5 .. 6) times these stay exact E4M3 values
    exps = rng.integers(-8, 7, size=(L, 8))
    scales = oracle.e4m3_encode(np.ldexp(1.0, exps)).reshape(L, 8)
    assert np.array_equal(oracle.e4m3_decode(scales), np.ldexp(1.0, exps))
    iq = oracle.quantize_fp8(rng.standard_normal((q_len, 4, 128)).astype(np.float32))
    a = oracle.indexer_seq(L, q_len, iq, oracle.INDEX_NVFP4, vals, scales)
    b = oracle.indexer_seq(L, q_len, iq, oracle.INDEX_NVFP4_EXACT, vals, scales)
    assert np.array_equal(a, b)


def test_a_tie_that_e4m3_rounds_is_kept_exactly():
    vals, scales = _one_key(E2M1_SIX, E4M3_1_125, dim=5)
    iq = _iq_unit(dim=5)
    rer = oracle.indexer_seq(1, 1, iq, oracle.INDEX_NVFP4, vals, scales)
    exact = oracle.indexer_seq(1, 1, iq, oracle.INDEX_NVFP4_EXACT, vals, scales)
    assert rer[0, 0, 0] == 7.0     # 6.75 -> RNE to the even-mantissa neighbour 7 (1.75 x 4)
    assert exact[0, 0, 0] == 6.75  # 6 x 1.125
    assert np.all(exact[0, 1:, 0] == 0.0) and np.all(rer[0, 1:, 0] == 0.0)


def test_signs_multiply_and_a_nan_scale_propagates():
    vals, scales = _one_key(E2M1_NEG_SIX, 0x80 | E4M3_1_125)
    iq = _iq_unit()
    assert oracle.indexer_seq(1, 1, iq, oracle.INDEX_NVFP4_EXACT, vals, scales)[0, 0, 0] == 6.75
    vals, scales = _one_key(E2M1_SIX, 0x80 | E4M3_1_125)
    assert oracle.indexer_seq(1, 1, iq, oracle.INDEX_NVFP4_EXACT, vals, scales)[0, 0, 0] == -6.75
    # a NaN scale makes its keys' scores NaN, which the block maximum passes over like fmax
    # does (the same rule as the E4M3 mode): a block of only such keys scores -inf
    vals, scales = _one_key(E2M1_SIX, 0x7F)
    assert np.isneginf(oracle.indexer_seq(1, 1, iq, oracle.INDEX_NVFP4_EXACT, vals, scales)[0, 0, 0])
    v2 = np.concatenate([vals, _one_key(E2M1_SIX, E4M3_ONE)[0]])
    s2 = np.concatenate([scales, _one_key(E2M1_SIX, E4M3_ONE)[1]])
    assert oracle.indexer_seq(2, 1, iq, oracle.INDEX_NVFP4_EXACT, v2, s2)[0, 0, 0] == 6.0


def test_exact_scores_stay_within_the_e4m3_rounding_bound():
    """|exact - re-rounded| <= sum_d |iq_d| * |ik_d| * 2^-4 (half an E4M3 ulp, relative)."""
    rng = np.random.default_rng(4)
    L = 256
    x = rng.standard_normal((L, 128)).astype(np.float32)
    vals, scales = oracle.quantize_nvfp4(x)
    iq = oracle.quantize_fp8(rng.standard_normal((1, 4, 128)).astype(np.float32))
    a = oracle.indexer_seq(L, 1, iq, oracle.INDEX_NVFP4, vals, scales)
    b = oracle.indexer_seq(L, 1, iq, oracle.INDEX_NVFP4_EXACT, vals, scales)
    assert not np.array_equal(a, b)  # the two readings do differ on ordinary data
    codes = oracle.unpack_nvfp4(vals)
    ik = oracle.e2m1_decode(codes) * np.repeat(oracle.e4m3_decode(scales), 16, axis=1)
    q = oracle.e4m3_decode(iq).reshape(4, 128)
    bound_key = (np.abs(q) @ np.abs(ik).T) * 2.0 ** -4  # [4, L]
    bound = np.stack([bound_key[:, 128 * k:128 * (k + 1)].max(1) for k in range(2)], 1)  # per block
    assert np.all(np.abs(a[0] - b[0]) <= bound + 1e-12)
