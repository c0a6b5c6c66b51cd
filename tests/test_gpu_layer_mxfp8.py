"""GPU parity of the 8-bit-activation path (MOE_ACT_MXFP8: E4M3 elements with one E8M0 scale per
32, the 4-bit-weight / 8-bit-activation configuration of the DGX Spark news item, section 2) against
the oracle's reading of it: the decode kernels for up to 16 tokens (the operands' MXFP8 values fed
to the FP4 tensor cores as pieces) and the kind::mxf8f6f4 grouped GEMMs beyond, with the quantised
token operand bit-exact, h within fp32 rounding of the oracle's decisions, and the layer output,
expert outputs and permutation as for the other formats."""
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

FMT = B.MOE_ACT_MXFP8

_layers = {}


def get_layer(cfg):
    if cfg.name not in _layers:
        _layers.clear()
        torch.cuda.empty_cache()
        _layers[cfg.name] = DeviceLayer(cfg)
    return _layers[cfg.name]


def e4m3_table():
    """Value of every E4M3 byte (bit 7 the sign), from the oracle's decoder."""
    mag = np.array([O.e4m3_value(c) if c != 0x7F else np.nan for c in range(128)], np.float64)
    return np.concatenate([mag, -mag])


def mma8_tiles_to_rows(buf, rows, K):
    """Inverse of the documented MXFP8 tensor-core code tiles: [rows][K] E4M3 bytes."""
    r = np.arange(rows)[:, None]
    c = np.arange(K // 16)[None, :]
    off = ((r // 128) * (K // 128) + c // 8) * 16384 + (r % 128) * 128 + (((c % 8) ^ (r % 8)) * 16)
    idx = off[:, :, None] + np.arange(16)[None, None, :]
    return buf.reshape(-1)[idx].reshape(rows, K)


def mma_scales_to_rows(buf, rows, K):
    """Inverse of the documented tensor-core scale layout: [rows][K/32]."""
    r = np.arange(rows)[:, None]
    c = np.arange(K // 32)[None, :]
    atom = (r // 128) * (K // 128) + c // 4
    off = atom * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + c % 4
    return buf[off]


def unpad(padded, pad_offsets, counts):
    return np.concatenate([padded[pad_offsets[e]:pad_offsets[e] + counts[e]] for e in range(len(counts))], axis=0)


def oracle_layer(layer, xb, **kw):
    cfg = layer.cfg
    return O.moe_layer(xb, layer.W_r_host, layer.b_host, cfg.k, oracle_expert_weights(cfg, layer.seed), O.ACT_MXFP8,
                       **kw)


# ------------------------------------------------------------------ up to 16 tokens: decode kernels

DECODE = {
    "tiny": IN.CONFIGS["tiny"],
    "decode": IN.CONFIGS["decode"],
    "spec_verify": IN.CONFIGS["spec_verify"],
    "mx8_t2": IN.small_config("mx8_t2", T=2, d=2048, E=6, k=3, I=1536, index=141),
    "mx8_t11": IN.small_config("mx8_t11", T=11, d=1024, E=16, k=4, I=512, index=142, zipf_s=1.2),
}


@pytest.mark.parametrize("name,calls", [("tiny", [0, 1]), ("decode", [0, 1]), ("spec_verify", [0]),
                                        ("mx8_t2", [0, 1]), ("mx8_t11", [0])])
def test_decode_layer_matches_oracle(name, calls):
    layer = get_layer(DECODE[name])
    cfg = layer.cfg
    ws = make_workspace(cfg.T, cfg.d, cfg.E, cfg.k, cfg.I, FMT)
    for call in calls:
        xb = IN.make_x(cfg, call=call)
        y, ids, w = layer_forward(layer, bits_to_device(xb), FMT, ws=ws, want_routing=True)
        ref = oracle_layer(layer, xb)
        np.testing.assert_array_equal(ids.cpu().numpy(), ref["ids"])
        check_weights(w.cpu().numpy(), ref["w"])
        check_permutation(workspace_routing(ws, cfg.T, cfg.d, cfg.E, cfg.k, cfg.I, FMT), ref)
        check_outputs(bf16_tensor_to_f32(y), ref["y"], "%s call %d" % (name, call))
    assert B.moe_get_device_status(ws) == B.MOE_OK


def pieces_sum(xa, xa_s, T, d):
    """Sum of each token's 8 piece rows, decoded from the documented FP4 tensor-core layouts."""
    from test_gpu_layer_mxfp4 import mma_tiles_to_rows
    from test_oracle_pins import np_unpack
    q = mma_tiles_to_rows(xa, 128, d)
    s = mma_scales_to_rows(xa_s, 128, d)
    v = np_unpack(q, s).astype(np.float64)
    return v[:8 * T].reshape(T, 8, d).sum(axis=1)


@pytest.mark.parametrize("name", ["tiny", "decode", "mx8_t2", "mx8_t11"])
def test_decode_step_calls_equal_layer_call(name):
    """moe_route -> moe_permute -> moe_decode_pieces -> moe_expert_ffn_decode (-> moe_combine beyond
    four tokens) gives the layer call's output bit for bit; the token pieces sum to the oracle's
    MXFP8 values of x (to within the pieces' residual, exactly for all but a few elements); the
    expert outputs match the oracle's intermediates."""
    layer = get_layer(DECODE[name])
    cfg = layer.cfg
    T, d, E, k, I = cfg.T, cfg.d, cfg.E, cfg.k, cfg.I
    P = T * k
    xb = IN.make_x(cfg, call=5)
    x = bits_to_device(xb)
    ws = make_workspace(T, d, E, k, I, FMT)
    i32 = dict(dtype=torch.int32, device="cuda")
    u8 = dict(dtype=torch.uint8, device="cuda")
    ids, w = torch.empty((T, k), **i32), torch.empty((T, k), dtype=torch.float32, device="cuda")
    counts, offsets, perm, inv = (torch.empty(E, **i32), torch.empty(E + 1, **i32), torch.empty(P, **i32),
                                  torch.empty(P, **i32))
    xa = torch.zeros(B.moe_decode_pieces_bytes(T, d, 0), **u8)
    xa_s = torch.zeros(B.moe_decode_pieces_bytes(T, d, 1), **u8)
    y_perm = torch.empty((P, d), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((T, d), dtype=torch.bfloat16, device="cuda")
    B.moe_route(x, layer.W_r, layer.b, T, d, E, k, ids, w, ws)
    B.moe_permute(x, ids, T, d, E, k, FMT, counts, offsets, perm, inv, None, None, ws)
    B.moe_decode_pieces(x, T, d, FMT, xa, xa_s)
    fused = T <= 4
    B.moe_expert_ffn_decode(xa, xa_s, FMT, perm, offsets, inv, w, T, d, E, k, I, layer.weights, y_perm,
                            y if fused else None, ws)
    if not fused:
        B.moe_combine(y_perm, inv, w, T, k, d, y)
    y_layer = layer_forward(layer, x, FMT)
    torch.cuda.synchronize()
    assert B.moe_get_device_status(ws) == B.MOE_OK
    assert torch.equal(y.view(torch.int16), y_layer.view(torch.int16))
    # the pieces against the oracle's MXFP8 operand
    a_ref = O.activation_rows(xb, O.ACT_MXFP8).astype(np.float64)
    got = pieces_sum(xa.cpu().numpy(), xa_s.cpu().numpy(), T, d)
    blockmax = np.repeat(np.abs(a_ref).reshape(T, d // 32, 32).max(axis=2), 32, axis=1)
    err = np.abs(got - a_ref)
    assert np.all(err <= blockmax * 2.0 ** -12), np.max(err / np.maximum(blockmax, 1e-300))
    assert np.mean(err == 0) > 0.999
    ref = oracle_layer(layer, xb, want_intermediates=True)
    rows = inv.cpu().numpy()
    yp_ref = np.stack([ref["y_perm"][(t, j)] for t in range(T) for j in range(k)])
    check_outputs(bf16_tensor_to_f32(y_perm)[rows], yp_ref, "y_perm")
    check_outputs(bf16_tensor_to_f32(y), ref["y"], "y")


# ------------------------------------------------------------------ more tokens: kind::mxf8f6f4 GEMMs

def run_prefill_steps(layer, xb):
    cfg = layer.cfg
    T, d, E, k, I = cfg.T, cfg.d, cfg.E, cfg.k, cfg.I
    P = T * k
    x = bits_to_device(xb)
    ws = make_workspace(T, d, E, k, I, FMT)
    R = B.moe_padded_rows(T, k, E)
    i32 = dict(dtype=torch.int32, device="cuda")
    u8 = dict(dtype=torch.uint8, device="cuda")
    ids, w = torch.empty((T, k), **i32), torch.empty((T, k), dtype=torch.float32, device="cuda")
    counts, offsets, perm, inv = (torch.empty(E, **i32), torch.empty(E + 1, **i32), torch.empty(P, **i32),
                                  torch.empty(P, **i32))
    xa, xa_s = torch.zeros((R, d), **u8), torch.zeros(B.moe_mxfp4_mma_scale_bytes(R, d), **u8)
    h, h_s = torch.zeros((R, I), **u8), torch.zeros(B.moe_mxfp4_mma_scale_bytes(R, I), **u8)
    y_perm = torch.empty((P, d), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((T, d), dtype=torch.bfloat16, device="cuda")
    B.moe_route(x, layer.W_r, layer.b, T, d, E, k, ids, w, ws)
    B.moe_permute(x, ids, T, d, E, k, FMT, counts, offsets, perm, inv, xa, xa_s, ws)
    B.moe_expert_up_swiglu(None, xa, xa_s, FMT, perm, offsets, T, d, E, k, I, layer.weights, h, h_s, ws)
    B.moe_expert_down(h, h_s, FMT, perm, offsets, T, d, E, k, I, layer.weights, y_perm, ws)
    B.moe_combine(y_perm, inv, w, T, k, d, y)
    torch.cuda.synchronize()
    assert B.moe_get_device_status(ws) == B.MOE_OK
    cn = counts.cpu().numpy()
    pad = np.concatenate([[0], np.cumsum((cn + 127) // 128 * 128)])
    return dict(ids=ids.cpu().numpy(), counts=cn, perm=perm.cpu().numpy(), inv=inv.cpu().numpy(), pad=pad,
                xa=xa.cpu().numpy(), xa_s=xa_s.cpu().numpy(), h=h.cpu().numpy(), h_s=h_s.cpu().numpy(),
                y_perm=bf16_tensor_to_f32(y_perm), y=bf16_tensor_to_f32(y), R=R)


PREFILL_SMALL = IN.small_config("mx8_prefill", T=200, d=512, E=8, k=2, I=768, index=143, zipf_s=1.2)


@pytest.mark.parametrize("cfg", [IN.CONFIGS["tiny"], PREFILL_SMALL], ids=["tiny", "mx8_prefill"])
def test_prefill_step_calls_against_oracle_intermediates(cfg):
    layer = get_layer(cfg)
    T, d, k, I = cfg.T, cfg.d, cfg.k, cfg.I
    xb = IN.make_x(cfg, call=0)
    g = run_prefill_steps(layer, xb)
    ref = oracle_layer(layer, xb, want_intermediates=True)
    np.testing.assert_array_equal(g["ids"], ref["ids"])
    np.testing.assert_array_equal(g["perm"], ref["perm_token"])
    # token operand: every permuted row is its token's MXFP8 row, bit for bit; padding rows zero
    _, xq, xs = O.activation_rows(xb, O.ACT_MXFP8, want_codes=True)
    xa_all = mma8_tiles_to_rows(g["xa"], g["R"], d)
    np.testing.assert_array_equal(unpad(xa_all, g["pad"], g["counts"]), xq[g["perm"]])
    np.testing.assert_array_equal(unpad(mma_scales_to_rows(g["xa_s"], g["R"], d), g["pad"], g["counts"]),
                                  xs[g["perm"]])
    used = np.zeros(g["R"], bool)
    for e in range(cfg.E):
        used[g["pad"][e]:g["pad"][e] + g["counts"][e]] = True
    assert not xa_all[~used].any()
    # h: MXFP8 values against the oracle's (decisions in fp32 on both sides)
    lut = e4m3_table()
    h_codes = unpad(mma8_tiles_to_rows(g["h"], g["R"], I), g["pad"], g["counts"])
    h_scales = unpad(mma_scales_to_rows(g["h_s"], g["R"], I), g["pad"], g["counts"]).astype(np.int64)
    h_gpu = lut[h_codes] * np.exp2(np.repeat(h_scales, 32, axis=1) - 127.0)
    h_ref = np.zeros_like(h_gpu)
    for t in range(T):
        for j in range(k):
            h_ref[g["inv"][t * k + j]] = ref["h"][(t, j)][0]
    check_outputs(h_gpu, h_ref, "h")
    same = np.mean(h_gpu == h_ref)
    assert same > 0.99, same
    yp_ref = np.zeros_like(g["y_perm"])
    for t in range(T):
        for j in range(k):
            yp_ref[g["inv"][t * k + j]] = ref["y_perm"][(t, j)]
    check_outputs(g["y_perm"], yp_ref, "y_perm")
    check_outputs(g["y"], ref["y"], "y")


# 72 blocks per token row (a full and a partial 64-block segment of the operand pass), ragged tiles
PREFILL_SEGMENTS = IN.small_config("mx8_segments", T=300, d=2304, E=16, k=4, I=256, index=162, zipf_s=1.2)


@pytest.mark.parametrize("cfg", [PREFILL_SMALL, PREFILL_SEGMENTS], ids=["mx8_prefill", "mx8_segments"])
def test_prefill_layer_call_equals_step_calls(cfg):
    layer = get_layer(cfg)
    xb = IN.make_x(cfg, call=1)
    g = run_prefill_steps(layer, xb)
    y = layer_forward(layer, bits_to_device(xb), FMT)
    np.testing.assert_array_equal(bf16_tensor_to_f32(y), g["y"])


@pytest.mark.parametrize("name,call", [("mx8_prefill", 2), ("mx8_t17", 0), ("prefill", 0), ("long_prefill", 1)])
def test_prefill_layer_matches_oracle(name, call):
    cfg = {"mx8_prefill": PREFILL_SMALL,
           "mx8_t17": IN.small_config("mx8_t17", T=17, d=1024, E=16, k=4, I=512, index=144)}.get(name) or IN.CONFIGS[name]
    layer = get_layer(cfg)
    xb = IN.make_x(cfg, call=call)
    ws = make_workspace(cfg.T, cfg.d, cfg.E, cfg.k, cfg.I, FMT)
    y, ids, w = layer_forward(layer, bits_to_device(xb), FMT, ws=ws, want_routing=True)
    torch.cuda.synchronize()
    assert B.moe_get_device_status(ws) == B.MOE_OK
    tokens = IN.sample_tokens(cfg, cfg.T) if cfg.sample_tokens else None
    if tokens is not None and cfg.calls > 1:  # a different sample per chunk
        rng = np.random.default_rng([cfg.sample_seed, call])
        tokens = np.sort(rng.choice(cfg.T, size=cfg.sample_tokens // cfg.calls, replace=False))
    ref = oracle_layer(layer, xb, tokens=tokens)
    np.testing.assert_array_equal(ids.cpu().numpy(), ref["ids"])
    check_weights(w.cpu().numpy(), ref["w"])
    check_permutation(workspace_routing(ws, cfg.T, cfg.d, cfg.E, cfg.k, cfg.I, FMT), ref)
    yg = bf16_tensor_to_f32(y)
    if tokens is not None:
        yg = yg[tokens]
    check_outputs(yg, ref["y"], "%s call %d" % (name, call))


def test_mxfp8_needs_tensor_core_weight_copies():
    cfg = IN.small_config("mx8_nomma", T=4, d=256, E=4, k=2, I=256, index=145)
    layer = DeviceLayer(cfg, mma_layouts=False)
    x = torch.zeros((cfg.T, cfg.d), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(B.MoeError) as e:
        layer_forward(layer, x, FMT)
    assert e.value.status == B.MOE_ERR_INVALID_ARG
