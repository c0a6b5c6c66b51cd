"""Pins of the oracle's MXFP4 expert path and of the layer's pairing of gate weights with expert
outputs, each against a route that shares nothing with the code it checks.

* The MXFP4 requantisation of h (the down GEMM's operand on the tensor-core path): an expert on
  grid-valued operands, where every dot product is exact in fp64 in any order, recomputed in numpy
  and quantised block by block with a brute-force nearest-code search under the OCP MX scale rule
  (Muse Spark Open explainer, section 9: gate, up and down per expert; section 11: 4-bit values
  sharing a block scale).  Codes, scales, h and y must agree bit for bit.
* The weighted sum (section 9): every token's output rebuilt from single-row expert calls, one
  per chosen slot, weighted in slot order; and the metamorphic pin that one expert's down scales
  raised by one (its outputs doubled exactly) change exactly the tokens that chose it, by exactly
  their weight times that expert's output.
"""
import numpy as np
import pytest

from bit_expert_ffn_moe_gb300 import inputs as IN
from oracle import oracle as O

E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _decode(q, s):
    """Exact fp64 values of an MXFP4 matrix, written out from the OCP MX tables."""
    codes = np.empty((q.shape[0], q.shape[1] * 2), np.int64)
    codes[:, 0::2] = q & 0xF
    codes[:, 1::2] = q >> 4
    mag = E2M1[codes & 7]
    val = np.where(codes & 8, -mag, mag)
    return val * np.repeat(2.0 ** (s.astype(np.int64) - 127), 32, axis=1)


def _brute_mx4_block(v):
    """One 32-element block by exhaustive search: scale X = floor(log2 amax) - 2 clamped to
    [-127, 127]; each element the nearest of the 16 codes (value / 2^X is exact), ties to the code
    with the even magnitude index, +0 for a zero result."""
    v = np.asarray(v, dtype=np.float64)
    amax = np.max(np.abs(v))
    if amax == 0.0:
        return np.zeros(32, np.uint8), 0
    _, e = np.frexp(amax)              # amax = m * 2^e, m in [0.5, 1)
    X = int(np.clip(e - 1 - 2, -127, 127))
    codes = np.zeros(32, np.uint8)
    for i, x in enumerate(v / 2.0 ** X):
        best = None
        for c in range(8):
            dist = abs(abs(x) - E2M1[c])
            key = (dist, c % 2)            # nearer first, then the even code
            if best is None or key < best[0]:
                best = (key, c)
        c = best[1]
        if abs(x) > 6.0:
            c = 7                          # saturate
        codes[i] = c | (8 if (x < 0 and c != 0) else 0)
    return codes, X + 127


def _grid_expert(rng, d, I):
    """Expert matrices whose values lie on the MXFP4 grid: the packer reproduces them exactly."""
    def grid_matrix(rows, K):
        mag = E2M1[rng.integers(0, 8, size=(rows, K))]
        sign = np.where(rng.integers(0, 2, size=(rows, K)) == 1, -1.0, 1.0)
        scale = 2.0 ** rng.integers(-7, -3, size=(rows, K // 32)).repeat(32, axis=1)
        w = (sign * mag * scale).astype(np.float32)
        q, s = O.mxfp4_pack(w)
        assert np.array_equal(_decode(q, s), w.astype(np.float64))
        return q, s
    return grid_matrix(I, d), grid_matrix(I, d), grid_matrix(d, I)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_mxfp4_h_requantisation_matches_an_independent_route(seed):
    rng = np.random.default_rng(400 + seed)
    d, I, n = 256, 128, 6
    wg, wu, wd = _grid_expert(rng, d, I)
    xb = IN.to_bf16_bits((rng.standard_normal((n, d)) * 2.0).astype(np.float32))
    a = O.activation_rows(xb, O.ACT_MXFP4)
    y, (h, hq, hs) = O.expert_ffn(a, wg, wu, wd, O.ACT_MXFP4, want_h=True)

    G, U, D = _decode(*wg), _decode(*wu), _decode(*wd)
    a64 = a.astype(np.float64)
    # exact in fp64 (grid values, a 2^-? window of exponents far inside 53 bits), any order
    g = (a64 @ G.T).astype(np.float32).astype(np.float64)
    u = (a64 @ U.T).astype(np.float32).astype(np.float64)
    hf = (g / (1.0 + np.exp(-g)) * u).astype(np.float32)        # SiLU(g) * u, rounded to fp32
    h_ref = np.empty((n, I))
    for r in range(n):
        for b in range(I // 32):
            c, sb = _brute_mx4_block(hf[r, 32 * b:32 * b + 32])
            packed = (c[0::2] | (c[1::2] << 4)).astype(np.uint8)
            np.testing.assert_array_equal(hq[r, 16 * b:16 * b + 16], packed, err_msg="row %d block %d" % (r, b))
            assert hs[r, b] == sb, (r, b, hs[r, b], sb)
            mag = E2M1[c & 7]
            h_ref[r, 32 * b:32 * b + 32] = np.where(c & 8, -mag, mag) * 2.0 ** (sb - 127)
    np.testing.assert_array_equal(h.astype(np.float64), h_ref)
    # the down product of grid values is exact too: y = bf16(fp32(h D^T))
    y_ref = IN.bf16_bits_to_f32(IN.to_bf16_bits((h_ref @ D.T).astype(np.float32)))
    np.testing.assert_array_equal(y, y_ref)


def _unit_row(length, col):
    r = np.zeros(length, np.float32)
    r[col] = 1.0
    return r


def test_h_requantisation_decides_on_the_fp32_value():
    """An h value just below the midpoint 1.75 of the codes 1.5 and 2 (scaled by its block scale),
    whose fp32 rounding is 1.75 itself: quantised from fp32 it is a tie and goes to the even code
    (2.0); quantised from the fp64 value it would be 1.5.  The oracle holds h in fp32 (as the
    kernels do), so it must pick 2.0."""
    d, I = 32, 32
    found = None
    for g_val in (4.0, 3.0, 2.5, 5.0, 3.5, 6.0, 2.0, 4.5, 1.75, 5.5):
        s = g_val / (1.0 + np.exp(-g_val))
        u0 = np.float32(1.75 / s)
        for step in range(-4, 5):
            u_val = np.float32(u0)
            for _ in range(abs(step)):
                u_val = np.nextafter(u_val, np.float32(np.sign(step) * np.inf), dtype=np.float32)
            h64 = s * float(u_val)
            if 1.75 - 2.0 ** -24 < h64 < 1.75 and np.float32(h64) == np.float32(1.75):
                found = (np.float32(g_val), u_val)
                break
        if found:
            break
    assert found is not None
    g_val, u_val = found
    # a = [u, g, 1.5, 0 ...]; h_0 = SiLU(a_1) * a_0 (the boundary value), h_1 = SiLU(a_1) * a_2
    # (the block maximum, in [4, 8): block scale 2^0), every other h is 0
    a = np.zeros((1, d), np.float32)
    a[0, 0], a[0, 1], a[0, 2] = u_val, g_val, 1.5
    G = np.zeros((I, d), np.float32)
    U = np.zeros((I, d), np.float32)
    G[0], U[0] = _unit_row(d, 1), _unit_row(d, 0)
    G[1], U[1] = _unit_row(d, 1), _unit_row(d, 2)
    wg, wu = O.mxfp4_pack(G), O.mxfp4_pack(U)
    wd = O.mxfp4_pack(np.zeros((d, I), np.float32))
    _, (h, hq, hs) = O.expert_ffn(a, wg, wu, wd, O.ACT_MXFP4, want_h=True)
    assert hs[0, 0] == 127                       # X = 0
    code0 = int(hq[0, 0] & 0xF)
    assert code0 == 4 and h[0, 0] == 2.0, (code0, h[0, 0])
    # the fp64 decision differs, so this case separates the two readings
    c64, _ = _brute_mx4_block(np.array([s * float(u_val) for s in [g_val / (1.0 + np.exp(-float(g_val)))]]
                                       + [float(g_val) / (1.0 + np.exp(-float(g_val))) * 1.5] + [0.0] * 30))
    assert c64[0] == 3


# ------------------------------------------------------------------ pairing in the weighted sum

def _distinct_experts(E, d, I, seed):
    rng = np.random.default_rng(seed)
    mats = {}
    for e in range(E):
        std = 0.02 * (1.0 + 0.5 * e)   # every expert its own weights and output scale
        mats[e] = {"gate": O.mxfp4_pack((rng.standard_normal((I, d)) * std).astype(np.float32)),
                   "up": O.mxfp4_pack((rng.standard_normal((I, d)) * std).astype(np.float32)),
                   "down": O.mxfp4_pack((rng.standard_normal((d, I)) * std).astype(np.float32))}
    return mats


def _router(E, d, seed):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((E, d)) / np.sqrt(d)).astype(np.float32), \
        (rng.standard_normal(E) * 0.5).astype(np.float32)


def _recompose(xb, W_r, b, k, mats, act):
    """Every token's output from single-row expert calls, one per chosen slot, weighted in slot
    order with fp64 accumulation, then rounded to fp32 and bf16."""
    ids, w = O.topk_softmax(O.router_logits(xb, W_r, b), k)
    a = O.activation_rows(xb, act)
    T, d = xb.shape
    y = np.empty((T, d), np.float32)
    per_slot = {}
    for t in range(T):
        acc = np.zeros(d)
        for j in range(k):
            e = int(ids[t, j])
            ye = O.expert_ffn(a[t:t + 1], mats[e]["gate"], mats[e]["up"], mats[e]["down"], act)[0]
            per_slot[(t, j)] = ye
            acc = acc + np.float64(w[t, j]) * ye.astype(np.float64)
        y[t] = IN.bf16_bits_to_f32(IN.to_bf16_bits(acc.astype(np.float32)[None]))[0]
    return y, ids, w, per_slot


@pytest.mark.parametrize("act", [O.ACT_BF16, O.ACT_MXFP4])
def test_layer_output_is_each_tokens_own_weighted_sum(act):
    E, d, I, k, T = 6, 128, 64, 3, 11
    mats = _distinct_experts(E, d, I, seed=61)
    W_r, b = _router(E, d, seed=62)
    xb = IN.to_bf16_bits(np.random.default_rng(63).standard_normal((T, d)).astype(np.float32))
    out = O.moe_layer(xb, W_r, b, k, lambda e: mats[e], act)
    y_ref, ids, _, _ = _recompose(xb, W_r, b, k, mats, act)
    assert len(np.unique(ids)) == E      # every expert is used, in several slots
    np.testing.assert_array_equal(out["y"], y_ref)
    # a token subset gives the same rows
    sub = [9, 2, 5]
    out_sub = O.moe_layer(xb, W_r, b, k, lambda e: mats[e], act, tokens=sub)
    np.testing.assert_array_equal(out_sub["y"], y_ref[sub])


@pytest.mark.parametrize("act", [O.ACT_BF16, O.ACT_MXFP4])
def test_raising_one_experts_down_scales_changes_only_its_tokens(act):
    E, d, I, k, T = 5, 128, 64, 2, 12
    mats = _distinct_experts(E, d, I, seed=71)
    W_r, b = _router(E, d, seed=72)
    xb = IN.to_bf16_bits(np.random.default_rng(73).standard_normal((T, d)).astype(np.float32))
    y0, ids, w, per_slot = _recompose(xb, W_r, b, k, mats, act)
    base = O.moe_layer(xb, W_r, b, k, lambda e: mats[e], act)["y"]
    np.testing.assert_array_equal(base, y0)
    e_star = int(np.bincount(ids.reshape(-1), minlength=E).argmax())
    q, s = mats[e_star]["down"]
    bumped = dict(mats)
    bumped[e_star] = dict(mats[e_star], down=(q, (s.astype(np.int64) + 1).astype(np.uint8)))
    y1 = O.moe_layer(xb, W_r, b, k, lambda e: bumped[e], act)["y"]
    chose = (ids == e_star).any(axis=1)
    assert chose.any() and (~chose).any()
    np.testing.assert_array_equal(y1[~chose], base[~chose])
    for t in np.nonzero(chose)[0]:
        acc = np.zeros(d)
        for j in range(k):
            f = 2.0 if ids[t, j] == e_star else 1.0   # a doubled bf16 row is exactly 2 x the row
            acc = acc + np.float64(w[t, j]) * (f * per_slot[(t, j)].astype(np.float64))
        expect = IN.bf16_bits_to_f32(IN.to_bf16_bits(acc.astype(np.float32)[None]))[0]
        np.testing.assert_array_equal(y1[t], expect)
        assert not np.array_equal(y1[t], base[t])
