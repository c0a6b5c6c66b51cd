"""GPU parity of the prefill path (MOE_ACT_MXFP4, tcgen05 block-scaled grouped GEMMs): quantised
activation operand (bit-exact), h and expert outputs (tolerance), and the whole layer against
the oracle at the tiny size (all tokens) and at the prefill sizes (seeded token samples)."""
import numpy as np
import pytest
import torch

from bit_expert_ffn_moe_gb300 import binding as B
from bit_expert_ffn_moe_gb300 import inputs as IN
from bit_expert_ffn_moe_gb300.layer import DeviceLayer, layer_forward, make_workspace
from moe_testlib import (bf16_tensor_to_f32, bits_to_device, check_outputs, check_permutation, check_weights,
                         oracle_expert_weights, workspace_routing)
from oracle import oracle as O

pytestmark = pytest.mark.gpu

_layers = {}


def get_layer(cfg):
    if cfg.name not in _layers:
        _layers.clear()
        torch.cuda.empty_cache()
        _layers[cfg.name] = DeviceLayer(cfg)
    return _layers[cfg.name]


def unpad(padded, pad_offsets, counts, offsets):
    """Rows of the padded expert-grouped buffer back in compact permuted order."""
    out = []
    for e in range(len(counts)):
        out.append(padded[pad_offsets[e]:pad_offsets[e] + counts[e]])
    return np.concatenate(out, axis=0)


def mma_tiles_to_rows(buf, rows, K):
    """Inverse of the documented tensor-core code tiles: [rows][K/2] canonical codes."""
    r = np.arange(rows)[:, None]
    b = np.arange(K // 32)[None, :]
    off = ((r // 128) * (K // 256) + b // 8) * 16384 + (r % 128) * 128 + (((b % 8) ^ (r % 8)) * 16)
    idx = off[:, :, None] + np.arange(16)[None, None, :]
    return buf.reshape(-1)[idx].reshape(rows, K // 2)


def mma_scales_to_rows(buf, rows, K):
    """Inverse of the documented tensor-core scale layout: [rows][K/32]."""
    r = np.arange(rows)[:, None]
    c = np.arange(K // 32)[None, :]
    atom = (r // 128) * (K // 128) + c // 4
    off = atom * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + c % 4
    return buf[off]


def run_steps(layer, xb):
    cfg = layer.cfg
    T, d, E, k, I = cfg.T, cfg.d, cfg.E, cfg.k, cfg.I
    P = T * k
    x = bits_to_device(xb)
    fmt = B.MOE_ACT_MXFP4
    ws = make_workspace(T, d, E, k, I, fmt)
    R = B.moe_padded_rows(T, k, E)
    i32 = dict(dtype=torch.int32, device="cuda")
    u8 = dict(dtype=torch.uint8, device="cuda")
    ids, w = torch.empty((T, k), **i32), torch.empty((T, k), dtype=torch.float32, device="cuda")
    counts, offsets, perm, inv = (torch.empty(E, **i32), torch.empty(E + 1, **i32), torch.empty(P, **i32),
                                  torch.empty(P, **i32))
    xa, xa_s = torch.zeros((R, d // 2), **u8), torch.zeros(B.moe_mxfp4_mma_scale_bytes(R, d), **u8)
    h, h_s = torch.zeros((R, I // 2), **u8), torch.zeros(B.moe_mxfp4_mma_scale_bytes(R, I), **u8)
    y_perm = torch.empty((P, d), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((T, d), dtype=torch.bfloat16, device="cuda")
    B.moe_route(x, layer.W_r, layer.b, T, d, E, k, ids, w, ws)
    B.moe_permute(x, ids, T, d, E, k, fmt, counts, offsets, perm, inv, xa, xa_s, ws)
    B.moe_expert_up_swiglu(None, xa, xa_s, fmt, perm, offsets, T, d, E, k, I, layer.weights, h, h_s, ws)
    B.moe_expert_down(h, h_s, fmt, perm, offsets, T, d, E, k, I, layer.weights, y_perm, ws)
    B.moe_combine(y_perm, inv, w, T, k, d, y)
    torch.cuda.synchronize()
    assert B.moe_get_device_status(ws) == B.MOE_OK
    cn, on = counts.cpu().numpy(), offsets.cpu().numpy()
    pad = np.concatenate([[0], np.cumsum((cn + 127) // 128 * 128)])
    return dict(ids=ids.cpu().numpy(), w=w.cpu().numpy(), counts=cn, offsets=on, perm=perm.cpu().numpy(),
                inv=inv.cpu().numpy(), pad=pad, xa=xa.cpu().numpy(), xa_s=xa_s.cpu().numpy(), h=h.cpu().numpy(),
                h_s=h_s.cpu().numpy(), y_perm=bf16_tensor_to_f32(y_perm), y=bf16_tensor_to_f32(y), R=R)


def test_step_calls_tiny_against_oracle_intermediates():
    cfg = IN.CONFIGS["tiny"]
    layer = get_layer(cfg)
    xb = IN.make_x(cfg, call=0)
    g = run_steps(layer, xb)
    ref = O.moe_layer(xb, layer.W_r_host, layer.b_host, cfg.k, oracle_expert_weights(cfg, layer.seed), O.ACT_MXFP4,
                      want_intermediates=True)
    np.testing.assert_array_equal(g["ids"], ref["ids"])
    np.testing.assert_array_equal(g["perm"], ref["perm_token"])
    # activation operand: every permuted row is its token's quantised row, bit for bit
    _, xq, xs = O.activation_rows(xb, O.ACT_MXFP4, want_codes=True)
    xa_rows = unpad(mma_tiles_to_rows(g["xa"], g["R"], cfg.d), g["pad"], g["counts"], g["offsets"])
    xs_rows = unpad(mma_scales_to_rows(g["xa_s"], g["R"], cfg.d), g["pad"], g["counts"], g["offsets"])
    np.testing.assert_array_equal(xa_rows, xq[g["perm"]])
    np.testing.assert_array_equal(xs_rows, xs[g["perm"]])
    # padding rows are zero
    used = np.zeros(g["R"], bool)
    for e in range(cfg.E):
        used[g["pad"][e]:g["pad"][e] + g["counts"][e]] = True
    assert not mma_tiles_to_rows(g["xa"], g["R"], cfg.d)[~used].any()
    # h: dequantised values against the oracle's h (its quantisation decisions are taken in fp32
    # on both sides, so only values within fp32 rounding of a rounding boundary may differ)
    T, k, I = cfg.T, cfg.k, cfg.I
    h_rows = unpad(mma_tiles_to_rows(g["h"], g["R"], I), g["pad"], g["counts"], g["offsets"])
    hs_rows = unpad(mma_scales_to_rows(g["h_s"], g["R"], I), g["pad"], g["counts"], g["offsets"])
    from test_oracle_pins import np_unpack
    h_gpu = np_unpack(h_rows, hs_rows)
    h_ref = np.zeros_like(h_gpu)
    for t in range(T):
        for j in range(k):
            h_ref[g["inv"][t * k + j]] = ref["h"][(t, j)][0]
    check_outputs(h_gpu, h_ref, "h")
    same_codes = np.mean(h_gpu == h_ref)
    assert same_codes > 0.99, same_codes
    yp_ref = np.zeros_like(g["y_perm"])
    for t in range(T):
        for j in range(k):
            yp_ref[g["inv"][t * k + j]] = ref["y_perm"][(t, j)]
    check_outputs(g["y_perm"], yp_ref, "y_perm")
    check_outputs(g["y"], ref["y"], "y")


# d = 2304: 72 blocks per token row, so the layer call's operand pass (work items of 64 blocks) has
# a full and a partial segment per token; 300 tokens over 16 experts give ragged token tiles.
SEGMENTS = IN.small_config("mx_segments", T=300, d=2304, E=16, k=4, I=256, index=161, zipf_s=1.2)


@pytest.mark.parametrize("cfg", [IN.CONFIGS["tiny"], SEGMENTS], ids=["tiny", "mx_segments"])
def test_layer_call_equals_step_calls(cfg):
    """The layer call (counting top-k, one-launch permutation, each token row quantised once and
    written to its k padded rows) gives the step calls' output bit for bit."""
    layer = get_layer(cfg)
    xb = IN.make_x(cfg, call=1)
    g = run_steps(layer, xb)
    y = layer_forward(layer, bits_to_device(xb), B.MOE_ACT_MXFP4)
    np.testing.assert_array_equal(bf16_tensor_to_f32(y), g["y"])


@pytest.mark.parametrize("name,call", [("tiny", 2), ("prefill", 0), ("long_prefill", 0), ("long_prefill", 3)])
def test_layer_matches_oracle(name, call):
    cfg = IN.CONFIGS[name]
    layer = get_layer(cfg)
    xb = IN.make_x(cfg, call=call)
    ws = make_workspace(cfg.T, cfg.d, cfg.E, cfg.k, cfg.I, B.MOE_ACT_MXFP4)
    y, ids, w = layer_forward(layer, bits_to_device(xb), B.MOE_ACT_MXFP4, ws=ws, want_routing=True)
    torch.cuda.synchronize()
    assert B.moe_get_device_status(ws) == B.MOE_OK
    tokens = IN.sample_tokens(cfg, cfg.T) if cfg.sample_tokens else None
    if tokens is not None and cfg.calls > 1:  # a different sample per chunk
        rng = np.random.default_rng([cfg.sample_seed, call])
        tokens = np.sort(rng.choice(cfg.T, size=cfg.sample_tokens // cfg.calls, replace=False))
    ref = O.moe_layer(xb, layer.W_r_host, layer.b_host, cfg.k, oracle_expert_weights(cfg, layer.seed), O.ACT_MXFP4,
                      tokens=tokens)
    np.testing.assert_array_equal(ids.cpu().numpy(), ref["ids"])
    check_weights(w.cpu().numpy(), ref["w"])
    check_permutation(workspace_routing(ws, cfg.T, cfg.d, cfg.E, cfg.k, cfg.I, B.MOE_ACT_MXFP4), ref)
    yg = bf16_tensor_to_f32(y)
    if tokens is not None:
        yg = yg[tokens]
    check_outputs(yg, ref["y"], "%s call %d" % (name, call))


def test_skewed_and_ragged_expert_loads():
    """Counts that cross token-tile and padding boundaries (0, 1, 31, 32, 33, 127, 128, 129, 300)."""
    cfg = IN.small_config("ragged_mx", T=300, d=256, E=10, k=2, I=256, index=91)
    layer = DeviceLayer(cfg)
    T, d, E, k = cfg.T, cfg.d, cfg.E, cfg.k
    # force the routing: expert 0 takes every token (bias); the second slot goes to expert
    # assign[t] (one-hot feature), giving experts 1..5 the sizes below, expert 7 the rest (76)
    sizes = [1, 31, 32, 33, 127]
    assign = np.full(T, 7)
    pos = 0
    for e, s in enumerate(sizes, start=1):
        assign[pos:pos + s] = e
        pos += s
    rng = np.random.default_rng(4)
    assign = assign[rng.permutation(T)]
    W_r = np.zeros((E, d), np.float32)
    xf = IN.bf16_bits_to_f32(IN.make_x(cfg)).copy()
    xf[:, :E] = 0.0
    xf[np.arange(T), assign] = 1.0
    xb = IN.to_bf16_bits(xf)
    for e in range(E):
        W_r[e, e] = 50.0
    b = np.zeros(E, np.float32)
    b[0] = 100.0
    layer.W_r = torch.from_numpy(W_r).cuda()
    layer.b = torch.from_numpy(b).cuda()
    layer.W_r_host, layer.b_host = W_r, b
    y, ids, w = layer_forward(layer, bits_to_device(xb), B.MOE_ACT_MXFP4, want_routing=True)
    ref = O.moe_layer(xb, W_r, b, k, oracle_expert_weights(cfg, layer.seed), O.ACT_MXFP4)
    np.testing.assert_array_equal(ids.cpu().numpy(), ref["ids"])
    counts = np.bincount(ref["ids"].reshape(-1), minlength=E)
    assert counts[0] == T and set(sizes) <= set(counts.tolist())
    check_outputs(bf16_tensor_to_f32(y), ref["y"], "ragged")
