"""Pins for the oracle's MXFP8 activation format (reading R11: E4M3 elements after OCP OFP8, one
E8M0 scale per 32 elements with the OCP MX shared-exponent rule, X = floor(log2 amax) - 8).  Each
test checks the oracle against something other than itself: numpy's frexp for the scale and
torch's own float8_e4m3fn conversion for the elements, hand-worked ties and saturation,
grid-valued round trips, power-of-two invariance, and a numpy SwiGLU expert on operands
quantised by that independent route.

No test here needs a GPU.
"""
import numpy as np
import pytest
import torch

from bit_expert_ffn_moe_gb300 import inputs as IN
from oracle import oracle as O


def e4m3_table():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


E4M3 = e4m3_table()


def torch_mx8(v):
    """Independent MXFP8 of one block: the scale from numpy's frexp, the elements by torch's
    round-to-nearest-even conversion after clamping at 448 (for |v| / 2^X in (448, 512) the
    nearest-even result with saturation is 448, which is what clamping first gives)."""
    v = np.asarray(v, dtype=np.float64)
    amax = np.abs(v).max()
    if amax == 0:
        return np.zeros(v.shape[0], np.uint8), 0
    X = int(np.clip(np.frexp(amax)[1] - 1 - 8, -127, 127))
    a = np.minimum(np.abs(v) * 2.0 ** -X, 448.0).astype(np.float32)
    codes = torch.from_numpy(a).to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()
    neg = (codes != 0) & (v < 0)
    codes[neg] |= 0x80
    return codes, X + 127


def dequant(codes, sb):
    return E4M3[codes] * 2.0 ** (sb - 127)


def test_scale_rule_and_element_rounding_match_numpy_and_torch():
    rng = np.random.default_rng(12)
    for _ in range(400):
        scale = np.exp(rng.uniform(-60, 60))
        v = (rng.standard_normal(32) * scale).astype(np.float32).astype(np.float64)
        v[rng.integers(0, 32, 3)] = 0.0
        codes, sb = O.mx8_block_quantize(v)
        ref_codes, ref_sb = torch_mx8(v)
        assert sb == ref_sb
        np.testing.assert_array_equal(codes, ref_codes)


def test_ties_saturation_and_signed_zero_handworked():
    # amax 448: X = 8 - 8 = 0, scale byte 127; values need no scaling
    v = np.zeros(32)
    v[:6] = [448.0, 1.0625, 1.1875, -2.0 ** -10, -3.0, 0.013671875]
    codes, sb = O.mx8_block_quantize(v)
    assert sb == 127
    # 448 -> 0x7E; 1.0625 ties 1.0 / 1.125 -> even 0x38; 1.1875 ties 1.125 / 1.25 -> even 0x3A;
    # -2^-10 ties 0 / 2^-9 -> +0 (never -0); -3 -> 0xC4; the largest subnormal -> 0x07
    assert list(codes[:6]) == [0x7E, 0x38, 0x3A, 0x00, 0xC4, 0x07]
    # amax 500: X = 0 as well, and 500 / 470 saturate to 448
    v = np.zeros(32)
    v[:3] = [500.0, -470.0, 300.0]
    codes, sb = O.mx8_block_quantize(v)
    # 300 = 1.17 x 2^8 lies between 288 (1.125 x 2^8, 0x79) and 320 (0x7A): nearer 288
    assert sb == 127 and list(codes[:3]) == [0x7E, 0xFE, 0x79]
    assert E4M3[0x79] == 288.0 and E4M3[0x7A] == 320.0
    z, zs = O.mx8_block_quantize(np.zeros(32))
    assert zs == 0 and not z.any()


def test_grid_valued_blocks_round_trip_exactly():
    rng = np.random.default_rng(4)
    finite = [c for c in range(256) if not np.isnan(E4M3[c])]
    top = [c for c in range(0x78, 0x7F)]  # exponent field 15: 256 .. 448
    for _ in range(200):
        X = int(rng.integers(-100, 100))
        codes = rng.choice(finite, size=32).astype(np.uint8)
        codes[rng.integers(0, 32)] = rng.choice(top)  # the block maximum fixes the scale at X
        codes[(codes & 0x7F) == 0] = 0                # -0 is stored as +0
        v = E4M3[codes] * 2.0 ** X
        got, sb = O.mx8_block_quantize(v)
        assert sb == X + 127
        np.testing.assert_array_equal(got, codes)


def test_power_of_two_invariance():
    rng = np.random.default_rng(8)
    v = rng.standard_normal(32)
    c0, s0 = O.mx8_block_quantize(v)
    for n in (-50, -1, 3, 40):
        c1, s1 = O.mx8_block_quantize(v * 2.0 ** n)
        np.testing.assert_array_equal(c1, c0)
        assert s1 == s0 + n


def test_activation_rows_use_the_block_rule():
    rng = np.random.default_rng(2)
    xb = IN.to_bf16_bits((rng.standard_normal((3, 128)) * 3).astype(np.float32))
    a, q, s = O.activation_rows(xb, O.ACT_MXFP8, want_codes=True)
    x = O.activation_rows(xb, O.ACT_BF16)
    for r in range(3):
        for b in range(4):
            c, sb = torch_mx8(x[r, 32 * b:32 * b + 32])
            np.testing.assert_array_equal(q[r, 32 * b:32 * b + 32], c)
            assert s[r, b] == sb
            np.testing.assert_array_equal(a[r, 32 * b:32 * b + 32], dequant(c, sb).astype(np.float32))


def _rand_mx4_expert(rng, d, I, std=0.05):
    return [O.mxfp4_pack((rng.standard_normal((r, c)) * std).astype(np.float32)) for r, c in ((I, d), (I, d), (d, I))]


def _mx4_decode(q, s):
    E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0])
    codes = np.empty((q.shape[0], q.shape[1] * 2), np.uint8)
    codes[:, 0::2] = q & 0xF
    codes[:, 1::2] = q >> 4
    return E2M1[codes] * np.repeat(2.0 ** (s.astype(np.int64) - 127), 32, axis=1)


def test_mxfp8_expert_is_a_swiglu_ffn_on_mxfp8_operands():
    rng = np.random.default_rng(31)
    d, I, n = 256, 128, 5
    wg, wu, wd = _rand_mx4_expert(rng, d, I)
    xb = IN.to_bf16_bits(rng.standard_normal((n, d)).astype(np.float32))
    a = O.activation_rows(xb, O.ACT_MXFP8)
    y, (h, hq, hs) = O.expert_ffn(a, wg, wu, wd, O.ACT_MXFP8, want_h=True)
    G, U, D = (_mx4_decode(*m) for m in (wg, wu, wd))
    g = (a.astype(np.float64) @ G.T).astype(np.float32).astype(np.float64)
    u = (a.astype(np.float64) @ U.T).astype(np.float32).astype(np.float64)
    hf = (g / (1 + np.exp(-g)) * u).astype(np.float32)
    # h: the fp32 SwiGLU output quantised by the independent MXFP8 route, block by block
    for r in range(n):
        for b in range(I // 32):
            c, sb = torch_mx8(hf[r, 32 * b:32 * b + 32])
            blk = slice(32 * b, 32 * b + 32)
            # the two fp32 h values may differ in the last place (summation order), which can
            # move a code by one step; require equality almost everywhere
            assert np.mean(hq[r, blk] == c) >= 0.9 and abs(int(hs[r, b]) - sb) <= 1
    hd = h.astype(np.float64)
    ref = torch.from_numpy((hd @ D.T).astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.all(np.abs(y - ref) <= np.abs(ref) * 2.0 ** -7 + 1e-30)


def test_mxfp8_activations_are_closer_to_exact_than_mxfp4():
    rng = np.random.default_rng(17)
    d, I, n = 256, 256, 8
    wg, wu, wd = _rand_mx4_expert(rng, d, I)
    xb = IN.to_bf16_bits(rng.standard_normal((n, d)).astype(np.float32))
    ys = {}
    for fmt in (O.ACT_EXACT, O.ACT_MXFP8, O.ACT_MXFP4):
        ys[fmt] = O.expert_ffn(O.activation_rows(xb, fmt), wg, wu, wd, fmt).astype(np.float64)
    ref = np.linalg.norm(ys[O.ACT_EXACT])
    e8 = np.linalg.norm(ys[O.ACT_MXFP8] - ys[O.ACT_EXACT]) / ref
    e4 = np.linalg.norm(ys[O.ACT_MXFP4] - ys[O.ACT_EXACT]) / ref
    # E4M3 keeps 3 mantissa bits against E2M1's 1: about a quarter of the relative error (RNE
    # onto a grid with steps of 1/8 of the binade leaves ~2.4% RMS per operand; x and h are both
    # quantised)
    assert e8 < 0.08 and e8 < 0.35 * e4, (e8, e4)
