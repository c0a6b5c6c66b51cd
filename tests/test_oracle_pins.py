"""Pins for the CPU oracle: each test checks the oracle against something other than itself --
values the sources print, the published format tables, closed forms, invariants, library
routines that the special cases reduce to, and brute force on tiny inputs.

No test here needs a GPU.
"""
import itertools
import math

import numpy as np
import pytest
import torch

from conftest import golden_lines
from oracle import oracle as O
from bit_expert_ffn_moe_gb300 import inputs as IN

# E2M1 decode written from the format definition (OCP MX v1.0, FP4 E2M1), independently of
# the oracle: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0, exponent 0 subnormal.
def e2m1_from_bits(code):
    s = -1.0 if code & 8 else 1.0
    e = (code >> 1) & 3
    m = code & 1
    return s * (0.5 * m if e == 0 else 2.0 ** (e - 1) * (1.0 + 0.5 * m))


E2M1_NP = np.array([e2m1_from_bits(c) for c in range(16)], dtype=np.float64)


def np_unpack(q, s):
    """Independent numpy decode of packed MXFP4 rows (low nibble = even element)."""
    q = np.asarray(q, dtype=np.uint8)
    codes = np.empty((q.shape[0], q.shape[1] * 2), dtype=np.uint8)
    codes[:, 0::2] = q & 0xF
    codes[:, 1::2] = q >> 4
    scale = np.ldexp(1.0, np.asarray(s, dtype=np.int64) - 127)
    return E2M1_NP[codes] * np.repeat(scale, 32, axis=1)


# ------------------------------------------------------------------ formats

def test_e2m1_e8m0_tables_match_spec():
    for line in golden_lines("e2m1_e8m0.txt"):
        parts = line.split()
        if parts[0] == "scale":
            s, v = int(parts[1]), float(parts[2])
            assert O.e8m0_value(s) == v
            assert O.e8m0_value(s) == math.ldexp(1.0, s - 127)
        else:
            code, v = int(parts[0], 16), float(parts[1])
            got = O.e2m1_value(code)
            assert got == v and math.copysign(1, got) == math.copysign(1, v)
            assert got == e2m1_from_bits(code)
    assert math.isnan(O.e8m0_value(255))


def test_e2m1_rounding_ties_to_even():
    for line in golden_lines("e2m1_rounding.txt"):
        a, code = line.split()
        assert O.e2m1_encode_magnitude(float(a)) == int(code), a


def test_e2m1_encoder_is_nearest_brute_force():
    grid = E2M1_NP[:8]
    rng = np.random.default_rng(7)
    for a in rng.uniform(0, 8, size=20000):
        c = O.e2m1_encode_magnitude(a)
        d = np.abs(grid - a)
        assert d[c] == d.min()
        winners = np.flatnonzero(d == d.min())
        if len(winners) > 1:
            assert c % 2 == 0 and c in winners


def test_bf16_conversion_matches_torch():
    rng = np.random.default_rng(3)
    v = np.concatenate([rng.standard_normal(5000).astype(np.float32) * 10,
                        np.array([0.0, -0.0, 1.0, 1.00390625, 1.005859375, 65504.0, 3.0e38, 1e-40], np.float32)])
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    for x, r in zip(v, ref):
        assert O.float_to_bf16_bits(float(x)) == int(r)


# ------------------------------------------------------------------ MX quantiser

def test_pack_handworked_blocks():
    g = dict(line.split(maxsplit=1) for line in golden_lines("mxfp4_pack_handworked.txt"))
    v0 = np.array([float(t) for t in g["values0"].split()], dtype=np.float32)
    w = np.stack([v0, v0 * np.float32(2.0 ** -5)])
    q, s = O.mxfp4_pack(w)
    assert list(s[:, 0]) == [int(g["scale0"]), int(g["scale1"])]
    assert q[0].tobytes().hex().upper() == g["bytes0"].replace(" ", "")
    assert q[1].tobytes().hex().upper() == g["bytes1"].replace(" ", "")


def test_grid_valued_blocks_round_trip_exactly():
    rng = np.random.default_rng(11)
    rows = []
    for _ in range(200):
        X = int(rng.integers(-100, 100))
        codes = rng.integers(0, 16, size=32)
        codes[rng.integers(0, 32)] = 7  # the block maximum is 6 * 2^X, so the scale is X
        rows.append(E2M1_NP[codes] * 2.0 ** X)
    w = np.array(rows, dtype=np.float32)
    q, s = O.mxfp4_pack(w)
    np.testing.assert_array_equal(np_unpack(q, s).astype(np.float32), w)
    np.testing.assert_array_equal(O.mxfp4_unpack(q, s), w)


def test_quantiser_error_bound_and_scale_rule():
    rng = np.random.default_rng(5)
    w = (rng.standard_normal((64, 256)) * np.exp(rng.uniform(-20, 20, size=(64, 1)))).astype(np.float32)
    q, s = O.mxfp4_pack(w)
    deq = np_unpack(q, s)
    blocks = w.reshape(64, 8, 32).astype(np.float64)
    amax = np.abs(blocks).max(axis=2)
    X = np.floor(np.log2(amax)) - 2
    np.testing.assert_array_equal(s, (X + 127).astype(np.uint8))
    # amax / 2^X lies in [4, 8): elements up to 6*2^X round to the grid (error <= half the
    # local spacing <= 2^X), larger ones saturate to 6*2^X.
    err = np.abs(deq.reshape(64, 8, 32) - blocks)
    scale = 2.0 ** X[..., None]
    a = np.abs(blocks) / scale
    inside = a <= 6
    assert np.all(err[inside] <= scale.repeat(32, axis=2)[inside] * 1.0 + 0)
    assert np.all(err[~inside] == (np.abs(blocks) - 6 * scale)[~inside])
    # sign is kept except for values that round to zero
    nz = deq.reshape(64, 8, 32) != 0
    assert np.all(np.sign(deq.reshape(64, 8, 32))[nz] == np.sign(blocks)[nz])


def test_quantiser_scale_invariance_and_special_blocks():
    rng = np.random.default_rng(9)
    w = rng.standard_normal((16, 64)).astype(np.float32)
    q0, s0 = O.mxfp4_pack(w)
    for n in (-30, -1, 1, 17):
        q1, s1 = O.mxfp4_pack(w * np.float32(2.0 ** n))
        np.testing.assert_array_equal(q1, q0)
        np.testing.assert_array_equal(s1.astype(int), s0.astype(int) + n)
    z = np.zeros((2, 32), np.float32)
    z[1] = -0.0
    qz, sz = O.mxfp4_pack(z)
    assert not qz.any() and not sz.any()
    codes, sb = O.mx_block_quantize(np.array([-1e-30] + [1.0] * 31))
    assert codes[0] == 0  # a value that rounds to zero is +0, never -0
    with pytest.raises(ValueError):
        O.mxfp4_unpack(np.zeros((1, 16), np.uint8), np.full((1, 1), 255, np.uint8))


# ------------------------------------------------------------------ router

def test_router_reduction_order_handworked():
    d = 256
    x = IN.to_bf16_bits(np.ones((1, d), np.float32))
    for line in golden_lines("router_order_handworked.txt"):
        name, rest = line.split(maxsplit=1)
        terms, expect = rest.split("=>")
        W = np.zeros((1, d), np.float32)
        for t in terms.split():
            i, v = t.split(":")
            W[0, int(i)] = float(v)
        got = O.router_logits(x, W, None)
        assert got[0, 0] == np.float32(float(expect)), name


def test_router_exact_on_integer_inputs():
    # every partial sum is an integer below 2^24, so any correct order gives the exact dot
    rng = np.random.default_rng(1)
    T, d, E = 5, 8192, 24
    x = rng.integers(-8, 9, size=(T, d)).astype(np.float32)
    W = rng.integers(-8, 9, size=(E, d)).astype(np.float32)
    b = rng.integers(-100, 100, size=E).astype(np.float32)
    got = O.router_logits(IN.to_bf16_bits(x), W, b)
    exact = x.astype(np.int64) @ W.astype(np.int64).T + b.astype(np.int64)
    np.testing.assert_array_equal(got, exact.astype(np.float32))


def test_router_close_to_fp64_dot():
    rng = np.random.default_rng(2)
    T, d, E = 7, 4096, 33
    xb = IN.to_bf16_bits(rng.standard_normal((T, d)).astype(np.float32))
    x = IN.bf16_bits_to_f32(xb).astype(np.float64)
    W = (rng.standard_normal((E, d)) / math.sqrt(d)).astype(np.float32)
    b = rng.standard_normal(E).astype(np.float32)
    got = O.router_logits(xb, W, b).astype(np.float64)
    exact = x @ W.astype(np.float64).T + b
    # fp32 error bound: chains of d/32 fmas + 5 butterfly adds + 1 bias add
    n = d // 32 + 6
    bound = n * 2.0 ** -24 * (np.abs(x) @ np.abs(W.astype(np.float64)).T + np.abs(b)) * 1.01
    assert np.all(np.abs(got - exact) <= bound)


def test_topk_matches_stable_sort_and_brute_force():
    rng = np.random.default_rng(4)
    # tiny E: compare with every k-subset; the top-k set is the subset whose smallest member
    # beats every non-member (ties -> lower id)
    for E, k in ((8, 2), (8, 3), (6, 6), (5, 1)):
        for _ in range(50):
            l = rng.integers(-3, 4, size=(1, E)).astype(np.float32)  # many ties
            ids, w = O.topk_softmax(l, k)
            key = lambda e: (-l[0, e], e)
            best = min(itertools.combinations(range(E), k), key=lambda S: sorted(key(e) for e in S))
            assert tuple(ids[0]) == tuple(sorted(best))
    l = rng.standard_normal((300, 128)).astype(np.float32)
    l[:, 5] = l[:, 77]  # exact ties
    ids, w = O.topk_softmax(l, 8)
    ref = np.sort(np.argsort(-l, axis=1, kind="stable")[:, :8], axis=1)
    np.testing.assert_array_equal(ids, ref)


def test_gate_weights_reproduce_the_printed_example():
    printed = np.array([float(v) for v in next(golden_lines("muse_gate_weights.txt")).split()])
    assert abs(printed.sum() - 1.0) < 1e-12
    logits = np.full((1, 256), -50.0, np.float32)
    chosen = np.array([3, 40, 77, 101, 150, 199, 230, 255])
    logits[0, chosen] = np.log(printed).astype(np.float32)
    ids, w = O.topk_softmax(logits, 8)
    np.testing.assert_array_equal(ids[0], chosen)
    np.testing.assert_allclose(w[0], printed, atol=2e-7)


def test_gate_weights_sum_to_one_and_follow_exp_ratios():
    rng = np.random.default_rng(6)
    l = (rng.standard_normal((500, 64)) * 3).astype(np.float32)
    ids, w = O.topk_softmax(l, 8)
    assert np.all(np.abs(w.astype(np.float64).sum(axis=1) - 1.0) <= 1e-6)
    sel = np.take_along_axis(l, ids, axis=1).astype(np.float64)
    ratio = w[:, 1:].astype(np.float64) / w[:, :1]
    np.testing.assert_allclose(ratio, np.exp(sel[:, 1:] - sel[:, :1]), rtol=1e-6)


def test_zero_input_routes_to_first_k_with_equal_weights():
    x = np.zeros((3, 256), np.uint16)
    W = np.random.default_rng(0).standard_normal((16, 256)).astype(np.float32)
    ids, w = O.topk_softmax(O.router_logits(x, W, np.zeros(16, np.float32)), 4)
    np.testing.assert_array_equal(ids, np.tile(np.arange(4), (3, 1)))
    np.testing.assert_array_equal(w, np.full((3, 4), 0.25, np.float32))


# ------------------------------------------------------------------ permute

def test_permute_handworked():
    ids = np.array([[1, 3], [0, 1], [1, 2]], np.int32)
    counts, offsets, perm_token, inv_pos = O.permute(ids, 4)
    np.testing.assert_array_equal(counts, [1, 3, 1, 1])
    np.testing.assert_array_equal(offsets, [0, 1, 4, 5, 6])
    np.testing.assert_array_equal(perm_token, [1, 0, 1, 2, 2, 0])
    np.testing.assert_array_equal(inv_pos, [1, 5, 0, 2, 3, 4])


def test_permute_matches_stable_argsort():
    rng = np.random.default_rng(8)
    T, E, k = 777, 64, 6
    ids = np.sort(np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]), axis=1).astype(np.int32)
    counts, offsets, perm_token, inv_pos = O.permute(ids, E)
    flat = ids.reshape(-1)
    order = np.argsort(flat, kind="stable")  # (e, t, j) order of the t-major pair list
    np.testing.assert_array_equal(perm_token, order // k)
    np.testing.assert_array_equal(inv_pos[order], np.arange(T * k))
    np.testing.assert_array_equal(counts, np.bincount(flat, minlength=E))
    np.testing.assert_array_equal(offsets, np.concatenate([[0], np.cumsum(counts)]))


# ------------------------------------------------------------------ experts and the layer

def _rand_expert(rng, d, I, std=0.05):
    mats = [rng.standard_normal((I, d)) * std, rng.standard_normal((I, d)) * std, rng.standard_normal((d, I)) * std]
    return [O.mxfp4_pack(m.astype(np.float32)) for m in mats]


def test_single_expert_is_a_dense_swiglu_ffn():
    """E = 1, k = 1: the layer reduces to y = W_d (SiLU(W_g x) * (W_u x)) (numpy fp64)."""
    rng = np.random.default_rng(12)
    d, I, T = 64, 96, 9
    wg, wu, wd = _rand_expert(rng, d, I)
    xb = IN.to_bf16_bits(rng.standard_normal((T, d)).astype(np.float32))
    res = O.moe_layer(xb, np.zeros((1, d), np.float32), None, 1,
                      lambda e: {"gate": wg, "up": wu, "down": wd}, O.ACT_EXACT)
    x = IN.bf16_bits_to_f32(xb).astype(np.float64)
    G, U, D = np_unpack(*wg), np_unpack(*wu), np_unpack(*wd)
    g = x @ G.T
    u = x @ U.T
    h = g / (1 + np.exp(-g)) * u
    y = h @ D.T
    assert np.all(res["w"] == 1.0)
    ref = IN.bf16_bits_to_f32(IN.to_bf16_bits(y.astype(np.float32)))
    err = np.abs(res["y"] - ref)
    assert np.all(err <= np.abs(ref) * 2.0 ** -7 + 1e-30)
    assert np.linalg.norm(res["y"] - y) / np.linalg.norm(y) < 4e-3


def test_handworked_grid_expert():
    """d = I = 32, weights on the E2M1 grid with scale 1: g and u are exact.
    W_g = 0.5 everywhere, W_u = 1 everywhere, W_d = row n holds 1.5 at column 0 and 0 elsewhere;
    x = 1: g = 16, u = 32, h_i = 16 * sigmoid(16) * 32, y_n = 1.5 * h_0."""
    d = I = 32
    wg = O.mxfp4_pack(np.full((I, d), 0.5, np.float32))
    wu = O.mxfp4_pack(np.full((I, d), 1.0, np.float32))
    D = np.zeros((d, I), np.float32)
    D[:, 0] = 1.5
    D[:, 1] = 6.0  # keeps each row's scale at 2^0 (amax 6); h_1 multiplies it
    wd = O.mxfp4_pack(D)
    xb = IN.to_bf16_bits(np.ones((1, d), np.float32))
    a = O.activation_rows(xb, O.ACT_EXACT)
    y, (h, _, _) = O.expert_ffn(a, wg, wu, wd, O.ACT_EXACT, want_h=True)
    hv = 16.0 / (1.0 + math.exp(-16.0)) * 32.0
    np.testing.assert_allclose(h[0], np.full(I, hv, np.float32), rtol=1e-7)
    expect = np.float32(7.5 * hv)
    assert np.all(y[0] == IN.bf16_bits_to_f32(IN.to_bf16_bits(np.array([expect]))))


def test_identical_experts_make_output_independent_of_routing():
    rng = np.random.default_rng(13)
    d, I, E, k, T = 64, 64, 6, 3, 12
    wts = _rand_expert(rng, d, I)
    xb = IN.to_bf16_bits(rng.standard_normal((T, d)).astype(np.float32))
    W_r = rng.standard_normal((E, d)).astype(np.float32)
    res = O.moe_layer(xb, W_r, None, k, lambda e: {"gate": wts[0], "up": wts[1], "down": wts[2]}, O.ACT_BF16)
    single = O.moe_layer(xb, W_r[:1], None, 1, lambda e: {"gate": wts[0], "up": wts[1], "down": wts[2]}, O.ACT_BF16)
    # sum_j w_j * y = y when the weights sum to one (within fp32 rounding, then bf16)
    np.testing.assert_allclose(res["y"], single["y"], rtol=2 ** -7, atol=1e-6)


def test_down_scale_plus_one_doubles_expert_output():
    rng = np.random.default_rng(14)
    d, I, n = 64, 64, 5
    wg, wu, (dq, ds) = _rand_expert(rng, d, I)
    a = O.activation_rows(IN.to_bf16_bits(rng.standard_normal((n, d)).astype(np.float32)), O.ACT_BF16)
    y1 = O.expert_ffn(a, wg, wu, (dq, ds), O.ACT_BF16)
    y2 = O.expert_ffn(a, wg, wu, (dq, (ds + 1).astype(np.uint8)), O.ACT_BF16)
    np.testing.assert_array_equal(y2, 2 * y1)


def test_mxfp4_activation_rows_use_the_weight_quantiser():
    rng = np.random.default_rng(15)
    xb = IN.to_bf16_bits(rng.standard_normal((4, 128)).astype(np.float32) * 3)
    a, q, s = O.activation_rows(xb, O.ACT_MXFP4, want_codes=True)
    q2, s2 = O.mxfp4_pack(IN.bf16_bits_to_f32(xb))
    np.testing.assert_array_equal(q, q2)
    np.testing.assert_array_equal(s, s2)
    np.testing.assert_array_equal(a, np_unpack(q, s).astype(np.float32))


def test_combine_is_weighted_sum_in_fp64():
    rng = np.random.default_rng(16)
    T, k, d = 6, 3, 40
    yp = IN.bf16_bits_to_f32(IN.to_bf16_bits(rng.standard_normal((T * k, d)).astype(np.float32)))
    rows = rng.permutation(T * k).reshape(T, k).astype(np.int32)
    w = rng.dirichlet(np.ones(k), size=T).astype(np.float32)
    tokens = np.array([0, 2, 5], np.int32)
    y = O.combine(yp, rows, w, tokens)
    ref = np.einsum("tj,tjc->tc", w.astype(np.float64), yp[rows].astype(np.float64))[tokens]
    np.testing.assert_array_equal(y, IN.bf16_bits_to_f32(IN.to_bf16_bits(ref.astype(np.float32))))


# ------------------------------------------------------------------ input generator

def test_splitmix64_known_answers():
    # published first outputs of SplitMix64 started from state 0
    z = IN.splitmix64_mix(np.array([(0x9E3779B97F4A7C15 * n) % 2 ** 64 for n in (1, 2, 3)], dtype=np.uint64))
    assert [int(v) for v in z] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_synth_weights_statistics():
    w = IN.synth_weights(1234, 2, 7, 256, 1024, 0.02)
    assert abs(w.std() - 0.02) < 2e-4 and abs(w.mean()) < 2e-4
    part = IN.synth_weights(1234, 2, 7, 256, 1024, 0.02, row_start=100, row_count=5)
    np.testing.assert_array_equal(part, w[100:105])


def test_synth_c_and_numpy_definitions_agree():
    a = IN.synth_weights(77, 1, 3, 64, 512, 0.02, use_c=True)
    b = IN.synth_weights(77, 1, 3, 64, 512, 0.02, use_c=False)
    np.testing.assert_array_equal(a, b)
    key = IN._host().inputs_stream_key(77, 1, 3)
    assert key == int(IN.stream_key(77, 1, 3))


# ------------------------------------------------------------------ expert output normalisation

def test_expert_norm_closed_form_and_unit_rms():
    """RMSNorm over the row: [3, 4] has mean square 12.5, so it becomes [3, 4] / sqrt(12.5 + eps);
    random rows come out with unit RMS (to within eps / mean square); a zero row stays zero."""
    eps = 1e-6
    y = O.expert_norm(np.array([[3.0, 4.0]], np.float32), eps)
    r = math.sqrt(12.5 + eps)
    np.testing.assert_array_equal(y[0], np.array([3.0 / r, 4.0 / r], np.float32))
    rng = np.random.default_rng(21)
    rows = (rng.standard_normal((7, 300)) * rng.uniform(0.01, 50.0, (7, 1))).astype(np.float32)
    out = O.expert_norm(rows, eps).astype(np.float64)
    ms = np.mean(rows.astype(np.float64) ** 2, axis=1)
    np.testing.assert_allclose(np.sqrt(np.mean(out ** 2, axis=1)), np.sqrt(ms / (ms + eps)), rtol=1e-6)
    np.testing.assert_array_equal(O.expert_norm(np.zeros((2, 32), np.float32), eps), np.zeros((2, 32), np.float32))


def test_expert_norm_removes_the_scale_of_each_expert():
    """With the normalisation, multiplying one expert's down weights by 2 (every scale byte + 1,
    an exact doubling of its bf16 outputs) leaves the layer output unchanged: bit for bit when
    eps = 0 (every step is an exact power-of-two rescaling), within a bf16 step for eps = 1e-6;
    without the normalisation the output changes."""
    rng = np.random.default_rng(22)
    d, I, E, k, T = 64, 64, 5, 2, 11
    experts = [_rand_expert(rng, d, I) for _ in range(E)]
    doubled = [list(x) for x in experts]
    dq, ds = experts[3][2]
    doubled[3][2] = (dq, (ds + 1).astype(np.uint8))
    xb = IN.to_bf16_bits(rng.standard_normal((T, d)).astype(np.float32))
    W_r = rng.standard_normal((E, d)).astype(np.float32)

    def run(ex, eps):
        return O.moe_layer(xb, W_r, None, k, lambda e: {"gate": ex[e][0], "up": ex[e][1], "down": ex[e][2]},
                           O.ACT_BF16, expert_norm_eps=eps)

    assert 3 in run(experts, None)["ids"]
    np.testing.assert_array_equal(run(experts, 0.0)["y"], run(doubled, 0.0)["y"])
    np.testing.assert_allclose(run(experts, 1e-6)["y"], run(doubled, 1e-6)["y"], rtol=2 ** -7, atol=0)
    assert not np.array_equal(run(experts, None)["y"], run(doubled, None)["y"])


def test_expert_norm_with_identical_experts_is_the_normalised_expert_output():
    """Identical experts and weights summing to one: y = RMSNorm(expert output) (numpy fp64)."""
    rng = np.random.default_rng(23)
    d, I, E, k, T = 64, 64, 4, 3, 6
    wg, wu, wd = _rand_expert(rng, d, I)
    xb = IN.to_bf16_bits(rng.standard_normal((T, d)).astype(np.float32))
    W_r = rng.standard_normal((E, d)).astype(np.float32)
    res = O.moe_layer(xb, W_r, None, k, lambda e: {"gate": wg, "up": wu, "down": wd}, O.ACT_BF16,
                      expert_norm_eps=1e-6)
    a = O.activation_rows(xb, O.ACT_BF16)
    v = O.expert_ffn(a, wg, wu, wd, O.ACT_BF16).astype(np.float64)
    ref = v / np.sqrt(np.mean(v ** 2, axis=1, keepdims=True) + 1e-6)
    np.testing.assert_allclose(res["y"], ref, rtol=2 ** -7, atol=1e-6)


# ------------------------------------------------------------------ shared latent projections

def test_dense_linear_against_numpy_fp64():
    """out = x W^T on the dequantised weights (numpy fp64, then bf16), bf16 activation values."""
    rng = np.random.default_rng(31)
    n, K, N = 5, 96, 64
    W = O.mxfp4_pack((rng.standard_normal((N, K)) * 0.05).astype(np.float32))
    xb = IN.to_bf16_bits(rng.standard_normal((n, K)).astype(np.float32))
    out = O.dense_linear(xb, W, O.ACT_BF16)
    ref = IN.bf16_bits_to_f32(xb).astype(np.float64) @ np_unpack(*W).T
    ref_b = IN.bf16_bits_to_f32(IN.to_bf16_bits(ref.astype(np.float32)))
    assert np.all(np.abs(out - ref_b) <= np.abs(ref_b) * 2.0 ** -7 + 1e-30)
    np.testing.assert_allclose(out, ref, rtol=2 ** -7, atol=1e-6)


def test_dense_linear_grid_case_is_exact_and_mxfp4_operand_is_used():
    """W row n holds 1.5 in column 0 and 6 in column 1 (scale 2^0), zeros elsewhere: out[n] =
    1.5 x0 + 6 x1 exactly.  With x0 = 0.3 the MXFP4 operand rounds x0 within its block (amax 1:
    scale 2^-2, 0.3 / 0.25 = 1.2 -> 1, so 0.25), which the MXFP4 mode must show."""
    K, N = 64, 32
    Wf = np.zeros((N, K), np.float32)
    Wf[:, 0], Wf[:, 1] = 1.5, 6.0
    W = O.mxfp4_pack(Wf)
    x = np.zeros((1, K), np.float32)
    x[0, 0], x[0, 1] = 0.3, 1.0
    xb = IN.to_bf16_bits(x)
    x0 = float(IN.bf16_bits_to_f32(xb)[0, 0])
    out_bf16 = O.dense_linear(xb, W, O.ACT_BF16)
    want = IN.bf16_bits_to_f32(IN.to_bf16_bits(np.array([np.float32(1.5 * x0 + 6.0)])))[0]
    assert np.all(out_bf16 == want)
    out_mx = O.dense_linear(xb, W, O.ACT_MXFP4)
    assert np.all(out_mx == np.float32(1.5 * 0.25 + 6.0))


def test_dense_linear_scales_exactly_with_powers_of_two():
    rng = np.random.default_rng(32)
    n, K, N = 3, 128, 32
    W = O.mxfp4_pack((rng.standard_normal((N, K)) * 0.05).astype(np.float32))
    xf = rng.standard_normal((n, K)).astype(np.float32)
    a = O.dense_linear(IN.to_bf16_bits(xf), W, O.ACT_BF16)
    b = O.dense_linear(IN.to_bf16_bits(xf * np.float32(8.0)), W, O.ACT_BF16)
    np.testing.assert_array_equal(b, a * np.float32(8.0))
