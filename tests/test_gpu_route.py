"""GPU parity of routing (ids bit-exact, weights within 2e-6) and of the permutation (bit-exact)."""
import numpy as np
import pytest
import torch

from bit_expert_ffn_moe_gb300 import binding as B
from bit_expert_ffn_moe_gb300 import inputs as IN
from bit_expert_ffn_moe_gb300.layer import make_workspace
from moe_testlib import bits_to_device, check_weights
from oracle import oracle as O

pytestmark = pytest.mark.gpu

CASES = {
    "tiny": IN.CONFIGS["tiny"],
    "decode_t1": IN.CONFIGS["decode"],
    "verify_t4": IN.CONFIGS["spec_verify"],
    "prefill": IN.CONFIGS["prefill"],
    "long_prefill_chunk": IN.CONFIGS["long_prefill"],
    "ragged": IN.small_config("ragged", T=333, d=384, E=40, k=5, I=256, zipf_s=1.3),
    # the screened router at its shape edges: the largest E and k (eight expert tiles, 32 experts
    # per lane in the candidate kernel), two K steps in all, and the largest d (64 K splits)
    "screen_e1024_k32": IN.small_config("screen_e1024_k32", T=300, d=256, E=1024, k=32, I=256, index=81),
    "screen_e1000_k17_d128": IN.small_config("screen_e1000_k17_d128", T=512, d=128, E=1000, k=17, I=256,
                                             zipf_s=1.1, index=82),
    "screen_t256_d16384": IN.small_config("screen_t256_d16384", T=256, d=16384, E=64, k=4, I=256, index=83),
}


def route_inputs(cfg, call=0):
    xb = IN.make_x(cfg, call=call)
    W_r, b = IN.make_router(cfg)
    return xb, W_r, b


def gpu_route(xb, W_r, b, k):
    T, d = xb.shape
    E = W_r.shape[0]
    ws = make_workspace(T, d, E, k, 128, B.MOE_ACT_BF16)
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    B.moe_route(bits_to_device(xb), torch.from_numpy(W_r).cuda(), None if b is None else torch.from_numpy(b).cuda(),
                T, d, E, k, ids, w, ws)
    return ids.cpu().numpy(), w.cpu().numpy(), ws


@pytest.mark.parametrize("name", list(CASES))
def test_route_matches_oracle(name):
    cfg = CASES[name]
    xb, W_r, b = route_inputs(cfg)
    ids, w, _ = gpu_route(xb, W_r, b, cfg.k)
    ids_o, w_o = O.topk_softmax(O.router_logits(xb, W_r, b), cfg.k)
    np.testing.assert_array_equal(ids, ids_o)
    check_weights(w, w_o)


@pytest.mark.parametrize("T", [64, 5, 600])  # dense router, one-launch router, screened router
def test_route_ties_and_zero_rows(T):
    d, E, k = 256, 16, 4
    rng = np.random.default_rng(5)
    x = rng.standard_normal((T, d)).astype(np.float32)
    x[::7] = 0.0                       # zero rows: all logits equal the bias
    W_r = rng.integers(-2, 3, size=(E, d)).astype(np.float32)
    W_r[3] = W_r[9]                    # duplicated experts: exact logit ties
    xb = IN.to_bf16_bits(np.round(x))  # integer inputs: exact logits, many ties
    b = np.zeros(E, np.float32)
    ids, w, _ = gpu_route(xb, W_r, b, k)
    ids_o, w_o = O.topk_softmax(O.router_logits(xb, W_r, b), k)
    np.testing.assert_array_equal(ids, ids_o)
    check_weights(w, w_o)
    np.testing.assert_array_equal(ids[0], np.arange(k))


@pytest.mark.parametrize("E,k,T,d", [(32, 6, 1024, 1024), (300, 8, 700, 512)])
def test_screened_route_near_ties(E, k, T, d):
    """Pairs of router rows that differ by a relative 2^-22 (and exact duplicates) give logits closer
    than any bound the tensor-core screen can certify, at the k-th boundary of many tokens: those
    experts must reach the fixed-order logits and be decided there, bit for bit as in the oracle."""
    rng = np.random.default_rng(11)
    base = rng.standard_normal((E // 2, d)) / np.sqrt(d)
    W_r = np.empty((E, d), np.float32)
    W_r[0::2] = base
    W_r[1::2] = base * (1.0 + 2.0 ** -22)
    W_r[5] = W_r[4]                                  # an exact tie
    b = np.repeat(rng.standard_normal(E // 2) * 0.5, 2).astype(np.float32)  # equal bias within a pair
    x = rng.standard_normal((T, d)).astype(np.float32)
    x[3] = 0.0
    x[17] *= 30.0                                    # a large row
    xb = IN.to_bf16_bits(x)
    ids, w, _ = gpu_route(xb, W_r, b, k)
    ids_o, w_o = O.topk_softmax(O.router_logits(xb, W_r, b), k)
    np.testing.assert_array_equal(ids, ids_o)
    check_weights(w, w_o)


@pytest.mark.parametrize("name", ["tiny", "prefill", "ragged"])
def test_permute_matches_oracle(name):
    cfg = CASES[name]
    xb, W_r, b = route_inputs(cfg)
    ids_o, _ = O.topk_softmax(O.router_logits(xb, W_r, b), cfg.k)
    T, k, E = cfg.T, cfg.k, cfg.E
    P = T * k
    ws = make_workspace(T, cfg.d, E, k, 128, B.MOE_ACT_BF16)
    dev = dict(dtype=torch.int32, device="cuda")
    counts, offsets = torch.empty(E, **dev), torch.empty(E + 1, **dev)
    perm, inv = torch.empty(P, **dev), torch.empty(P, **dev)
    B.moe_permute(None, torch.from_numpy(ids_o).cuda(), T, cfg.d, E, k, B.MOE_ACT_BF16, counts, offsets, perm, inv,
                  None, None, ws)
    ref = O.permute(ids_o, E)
    for got, want in zip((counts, offsets, perm, inv), ref):
        np.testing.assert_array_equal(got.cpu().numpy(), want)


def test_permute_ragged_counts():
    """Per-expert counts 0, 1, 127, 128, 129 and all tokens on one expert."""
    T, E, k = 129, 6, 2
    ids = np.zeros((T, k), np.int32)
    ids[:, 0] = 0                      # expert 0: every token (129)
    ids[:128, 1] = 2                   # expert 2: 128
    ids[128, 1] = 3                    # expert 3: 1; experts 1, 4, 5: 0
    ids[:127, 1][::1] = ids[:127, 1]
    ws = make_workspace(T, 128, E, k, 128, B.MOE_ACT_BF16)
    dev = dict(dtype=torch.int32, device="cuda")
    counts, offsets = torch.empty(E, **dev), torch.empty(E + 1, **dev)
    perm, inv = torch.empty(T * k, **dev), torch.empty(T * k, **dev)
    B.moe_permute(None, torch.from_numpy(ids).cuda(), T, 128, E, k, B.MOE_ACT_BF16, counts, offsets, perm, inv,
                  None, None, ws)
    ref = O.permute(ids, E)
    for got, want in zip((counts, offsets, perm, inv), ref):
        np.testing.assert_array_equal(got.cpu().numpy(), want)
