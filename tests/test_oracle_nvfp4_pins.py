"""Pins for the oracle's NVFP4 weight format (reading R10: E2M1 codes, one E4M3 scale per 16
elements, one fp32 global scale per matrix).  Each test checks the oracle against something
other than itself: the OFP8 table, torch's own float8_e4m3fn conversion, hand-worked blocks,
brute-force nearest-value searches, exact invariants, and the MXFP4 path that a
power-of-two-scaled NVFP4 matrix reduces to.

No test here needs a GPU.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

from conftest import golden_lines
from oracle import oracle as O

E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0])


def torch_e4m3_table():
    """Values of the 256 E4M3 bytes as torch decodes them (float8_e4m3fn is the OCP E4M3)."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


E4M3 = torch_e4m3_table()


def np_nv_unpack(q, s, gs):
    """Independent decode of one NVFP4 matrix: numpy nibbles, torch's E4M3 table, fp64."""
    q = np.asarray(q, dtype=np.uint8)
    codes = np.empty((q.shape[0], q.shape[1] * 2), dtype=np.uint8)
    codes[:, 0::2] = q & 0xF
    codes[:, 1::2] = q >> 4
    return E2M1[codes] * np.repeat(E4M3[np.asarray(s)], 16, axis=1) * float(gs)


# ------------------------------------------------------------------ E4M3

def test_e4m3_table_matches_spec_and_torch():
    for line in golden_lines("e4m3.txt"):
        code, v = line.split()
        got = O.e4m3_value(int(code, 16))
        if v == "nan":
            assert math.isnan(got)
        else:
            assert got == float(v) and math.copysign(1, got) == math.copysign(1, float(v)), code
    for c in range(256):
        got = O.e4m3_value(c)
        if math.isnan(E4M3[c]):
            assert math.isnan(got), c
        else:
            assert got == E4M3[c] and math.copysign(1, got) == math.copysign(1, E4M3[c]), c
    pos = [O.e4m3_value(c) for c in range(0x7F)]
    assert all(a < b for a, b in zip(pos, pos[1:]))  # 127 finite non-negative values, increasing


def test_e4m3_encoder_round_trips_ties_to_even_and_saturates():
    for c in range(0x7F):
        assert O.e4m3_encode(O.e4m3_value(c)) == c
    for c in range(0x7E):
        mid = (O.e4m3_value(c) + O.e4m3_value(c + 1)) / 2
        even = c if c % 2 == 0 else c + 1
        assert O.e4m3_encode(mid) == even, c
        assert O.e4m3_encode(np.nextafter(mid, 0)) == c
        assert O.e4m3_encode(np.nextafter(mid, 1e9)) == c + 1
    for a in (448.0, 460.0, 464.0, 500.0, 1e6, 3e38):
        assert O.e4m3_encode(a) == 0x7E
    assert O.e4m3_encode(2.0 ** -10) == 0            # halfway to the smallest subnormal: even (0)
    assert O.e4m3_encode(np.nextafter(2.0 ** -10, 1)) == 1


def test_e4m3_encoder_matches_torch_conversion():
    # torch's fp32 -> float8_e4m3fn conversion rounds to nearest even; below 464 it never
    # needs saturation, so on [0, 460] the two must agree bit for bit
    rng = np.random.default_rng(3)
    a = np.concatenate([rng.uniform(0, 460, 4000), np.exp(rng.uniform(-14, 6, 4000)),
                        [(E4M3[c] + E4M3[c + 1]) / 2 for c in range(0x7E)]]).astype(np.float32)
    ref = torch.from_numpy(a).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([O.e4m3_encode(float(v)) for v in a])
    np.testing.assert_array_equal(got, ref)


# ------------------------------------------------------------------ block quantiser

def test_nv_block_handworked():
    # gs = 1, block maximum 6: t = 1 -> scale 1.0 (0x38), D = 1; 1.25 and -0.25 are ties
    v = np.zeros(16, np.float32)
    v[:5] = [6.0, 3.0, 1.25, -0.25, -5.5]
    codes, sb = O.nv_block_quantize(v, 1.0)
    assert sb == 0x38
    assert list(codes[:5]) == [0x7, 0x5, 0x2, 0x0, 0xF]  # 6, 3, 1 (even), +0 (never -0), -6
    assert not codes[5:].any()
    # gs = 0.5, maximum 9: t = (9 / 0.5) / 6 = 3 -> 0x44, D = 1.5
    v = np.zeros(16, np.float32)
    v[:4] = [9.0, -4.5, 2.2, 0.7]
    codes, sb = O.nv_block_quantize(v, 0.5)
    assert sb == 0x44 and O.e4m3_value(sb) == 3.0
    assert list(codes[:4]) == [0x7, 0xD, 0x3, 0x1]  # 6, -3, 1.5 (2.2/1.5 = 1.47), 0.5 (0.47)


def test_global_scale_rule():
    assert O.nvfp4_global_scale(0.0) == 1.0
    assert O.nvfp4_global_scale(2688.0) == 1.0
    assert O.nvfp4_global_scale(1.0) == np.float32(1.0) / np.float32(2688.0)
    w = np.random.default_rng(1).standard_normal((3, 8, 64)).astype(np.float32)
    _, s, gs = O.nvfp4_pack(w)
    for m in range(3):
        assert gs[m] == np.float32(np.abs(w[m]).max()) / np.float32(2688.0)
        # the block holding the matrix maximum gets the largest scale, 448
        r, c = np.unravel_index(np.abs(w[m]).argmax(), w[m].shape)
        assert s[m, r, c // 16] == 0x7E


def test_pack_choices_are_nearest_by_brute_force():
    rng = np.random.default_rng(7)
    w = (rng.standard_normal((12, 64)) * np.exp(rng.uniform(-6, 6, size=(12, 1)))).astype(np.float32)
    q, s, gs = O.nvfp4_pack(w)
    gs = np.float32(gs)
    codes = np.empty((12, 64), np.uint8)
    codes[:, 0::2] = q & 0xF
    codes[:, 1::2] = q >> 4
    finite = [c for c in range(0x7F)]
    for r in range(12):
        for b in range(4):
            blk = w[r, 16 * b:16 * b + 16]
            t = (np.float32(np.abs(blk).max()) / gs) / np.float32(6.0)
            sb = int(s[r, b])
            # the scale byte is a nearest E4M3 value to t (exact rational distances)
            dist = [abs(Fraction(float(t)) - Fraction(float(E4M3[c]))) for c in finite]
            assert dist[sb] == min(dist)
            D = np.float32(E4M3[sb]) * gs
            for i in range(16):
                a = np.abs(blk[i]) / D  # fp32 quotient, the quantity the rule rounds
                d = [abs(Fraction(float(a)) - Fraction(float(E2M1[c]))) for c in range(8)]
                mag = int(codes[r, 16 * b + i]) & 7
                assert d[mag] == min(d)
                if mag:
                    assert (codes[r, 16 * b + i] >> 3) == (1 if blk[i] < 0 else 0)
                else:
                    assert codes[r, 16 * b + i] == 0


def test_pack_error_bound():
    rng = np.random.default_rng(5)
    w = (rng.standard_normal((32, 256)) * np.exp(rng.uniform(-3, 3, size=(32, 1)))).astype(np.float32)
    q, s, gs = O.nvfp4_pack(w)
    deq = np_nv_unpack(q, s, gs)
    np.testing.assert_array_equal(deq, O.nvfp4_unpack(q, s, gs))
    D = (E4M3[s] * float(np.float32(gs))).repeat(16, axis=1)
    D32 = (E4M3[s].astype(np.float32) * np.float32(gs)).repeat(16, axis=1).astype(np.float64)
    a = np.abs(w.astype(np.float64)) / D32
    half_gap = np.where(a <= 2, 0.25, np.where(a <= 4, 0.5, 1.0))
    err = np.abs(deq - w)
    inside = a <= 6
    assert np.all(err[inside] <= D[inside] * half_gap[inside] * (1 + 1e-6))
    assert np.all(err[~inside] <= (np.abs(w) - 6 * D)[~inside] * (1 + 1e-6) + 1e-30)
    # the scale of a block is within E4M3 rounding of amax / 6: amax / D lies in [5.5, 6.4]
    amax = np.abs(w.reshape(32, 16, 16)).max(axis=2)
    ratio = amax / (E4M3[s] * float(gs))
    assert np.all((ratio > 5.4) & (ratio < 6.5))


def test_pack_is_invariant_under_powers_of_two():
    rng = np.random.default_rng(9)
    w = rng.standard_normal((2, 16, 64)).astype(np.float32)
    q0, s0, g0 = O.nvfp4_pack(w)
    for n in (-40, -3, 1, 20):
        q1, s1, g1 = O.nvfp4_pack(w * np.float32(2.0 ** n))
        np.testing.assert_array_equal(q1, q0)
        np.testing.assert_array_equal(s1, s0)
        np.testing.assert_array_equal(g1, g0 * np.float32(2.0 ** n))


def test_zero_matrix_and_nan_scale():
    q, s, gs = O.nvfp4_pack(np.zeros((4, 32), np.float32))
    assert not q.any() and not s.any() and gs == 1.0
    with pytest.raises(ValueError):
        O.nvfp4_unpack(np.zeros((1, 8), np.uint8), np.full((1, 1), 0x7F, np.uint8), 1.0)
    with pytest.raises(ValueError):
        O.nvfp4_pack(np.zeros((1, 24), np.float32))


# ------------------------------------------------------------------ expert FFN

POW2_E4M3 = {j: ((j + 7) << 3) if j >= -6 else (1 << (j + 9)) for j in range(-9, 9)}


def _pow2_pair(rng, rows, K):
    """An NVFP4 matrix (global scale 1) whose two 16-element halves of every 32-element block
    share one power-of-two E4M3 scale, and the MXFP4 matrix with the same values."""
    q = rng.integers(0, 256, size=(rows, K // 2), dtype=np.uint8)
    j = rng.integers(-9, 9, size=(rows, K // 32))
    s_nv = np.vectorize(POW2_E4M3.get)(j).astype(np.uint8).repeat(2, axis=1)
    s_mx = (j + 127).astype(np.uint8)
    return (q, s_mx), (q, s_nv, np.float32(1.0))


@pytest.mark.parametrize("act", [O.ACT_BF16, O.ACT_MXFP4])
def test_expert_with_power_of_two_scales_is_the_mxfp4_expert(act):
    rng = np.random.default_rng(21 + act)
    d, I, n = 128, 96, 5
    (gmx, gnv), (umx, unv), (dmx, dnv) = _pow2_pair(rng, I, d), _pow2_pair(rng, I, d), _pow2_pair(rng, d, I)
    np.testing.assert_array_equal(np_nv_unpack(*gnv), np.repeat(2.0 ** (gmx[1].astype(float) - 127), 32, axis=1)
                                  * E2M1[np.stack([gmx[0] & 0xF, gmx[0] >> 4], axis=2).reshape(I, d)])
    xb = O_bits(rng.standard_normal((n, d)))
    a = O.activation_rows(xb, act)
    y_mx = O.expert_ffn(a, gmx, umx, dmx, act)
    y_nv = O.expert_ffn(a, gnv, unv, dnv, act)
    np.testing.assert_array_equal(y_nv, y_mx)


def O_bits(x):
    from bit_expert_ffn_moe_gb300 import inputs as IN
    return IN.to_bf16_bits(np.asarray(x, dtype=np.float32))


def _nv_expert(rng, d, I, std=0.05):
    mats = [O.nvfp4_pack((rng.standard_normal((r, c)) * std).astype(np.float32)) for r, c in ((I, d), (I, d), (d, I))]
    return mats


def test_nvfp4_expert_is_a_dense_swiglu_ffn_on_the_decoded_weights():
    rng = np.random.default_rng(33)
    d, I, n = 256, 128, 6
    wg, wu, wd = _nv_expert(rng, d, I)
    xb = O_bits(rng.standard_normal((n, d)))
    a = O.activation_rows(xb, O.ACT_BF16).astype(np.float64)
    G, U, Dn = (np_nv_unpack(*m) for m in (wg, wu, wd))
    g = (a @ G.T).astype(np.float32).astype(np.float64)
    u = (a @ U.T).astype(np.float32).astype(np.float64)
    h = g / (1 + np.exp(-g)) * u
    h = torch.from_numpy(h.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    ref = torch.from_numpy((h @ Dn.T).astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    y = O.expert_ffn(a.astype(np.float32), wg, wu, wd, O.ACT_BF16)
    # equal up to one bf16 rounding step where the two summation orders straddle a boundary
    assert np.all(np.abs(y - ref) <= np.abs(ref) * 2.0 ** -7 + 1e-30)
    assert np.mean(y == ref) > 0.9


def test_global_scales_scale_the_output_exactly():
    rng = np.random.default_rng(41)
    d, I, n = 128, 64, 4
    wg, wu, wd = _nv_expert(rng, d, I)
    xb = O_bits(rng.standard_normal((n, d)))
    a = O.activation_rows(xb, O.ACT_BF16)
    y0 = O.expert_ffn(a, wg, wu, wd, O.ACT_BF16)
    y_down = O.expert_ffn(a, wg, wu, (wd[0], wd[1], wd[2] * np.float32(2.0)), O.ACT_BF16)
    y_up = O.expert_ffn(a, wg, (wu[0], wu[1], wu[2] * np.float32(0.25)), wd, O.ACT_BF16)
    np.testing.assert_array_equal(y_down, y0 * 2)
    np.testing.assert_array_equal(y_up, y0 * 0.25)
