"""GPU parity of the decode-shape path (MOE_ACT_BF16): the whole layer against the oracle on both
of its kernel paths (tensor-core GEMMs on activation pieces when the weights carry their
tensor-core copies, CUDA-core GEMVs otherwise), and the step-by-step entry points (the GEMVs)
against the fused layer call on the GEMV path."""
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


# Small shapes: ring_t3 on the warp-per-row GEMVs with several tokens per expert; ring_t2 and
# ring_t1 on the CTA-split GEMVs (one or two tokens, down weights through the copy-engine ring).
SMALL = {
    "ring_t3": IN.small_config("ring_t3", T=3, d=1024, E=12, k=4, I=512, index=93),
    "ring_t2": IN.small_config("ring_t2", T=2, d=2048, E=6, k=3, I=1536, index=94),
    "ring_t1": IN.small_config("ring_t1", T=1, d=1024, E=16, k=4, I=1024, index=95),
    # more experts than SMs: the decode kernel takes the plan from the router launches instead of
    # routing its tokens itself
    "many_e": IN.small_config("many_e", T=2, d=1024, E=200, k=4, I=512, index=96),
}


def get_layer(name, mma=True):
    """mma: with the tensor-core weight copies (the layer call then runs the tensor-core GEMMs for
    up to 16 tokens); without them every bf16-path call runs the GEMVs."""
    key = (name, mma)
    if key not in _layers:
        _layers.clear()
        torch.cuda.empty_cache()
        _layers[key] = DeviceLayer(SMALL[name] if name in SMALL else IN.CONFIGS[name], mma_layouts=mma)
    return _layers[key]


def oracle_layer(layer, xb, act_fmt, tokens=None):
    cfg = layer.cfg
    return O.moe_layer(xb, layer.W_r_host, layer.b_host, cfg.k, oracle_expert_weights(cfg, layer.seed), act_fmt,
                       tokens=tokens)


@pytest.mark.parametrize("mma", [True, False])
@pytest.mark.parametrize("name,calls", [("tiny", [0, 1]), ("decode", [0, 1, 2]), ("spec_verify", [0]),
                                        ("ring_t3", [0, 1]), ("ring_t2", [0, 1]), ("ring_t1", [0, 1, 2]),
                                        ("many_e", [0, 1])])
def test_layer_matches_oracle(name, calls, mma):
    layer = get_layer(name, mma)
    cfg = layer.cfg
    ws = make_workspace(cfg.T, cfg.d, cfg.E, cfg.k, cfg.I, B.MOE_ACT_BF16)
    for call in calls:
        xb = IN.make_x(cfg, call=call)
        y, ids, w = layer_forward(layer, bits_to_device(xb), B.MOE_ACT_BF16, ws=ws, want_routing=True)
        ref = oracle_layer(layer, xb, O.ACT_BF16)
        np.testing.assert_array_equal(ids.cpu().numpy(), ref["ids"])
        check_weights(w.cpu().numpy(), ref["w"])
        # the permutation the layer call built in its workspace (the one-launch router for T <= 8)
        check_permutation(workspace_routing(ws, cfg.T, cfg.d, cfg.E, cfg.k, cfg.I, B.MOE_ACT_BF16), ref)
        check_outputs(bf16_tensor_to_f32(y), ref["y"], "%s call %d" % (name, call))
    assert B.moe_get_device_status(ws) == B.MOE_OK


@pytest.mark.parametrize("name", ["tiny", "ring_t3", "ring_t2", "ring_t1"])
def test_step_calls_equal_layer_call_and_oracle_h(name):
    layer = get_layer(name, mma=False)  # the step calls and the layer call both on the GEMVs
    cfg = layer.cfg
    T, d, E, k, I = cfg.T, cfg.d, cfg.E, cfg.k, cfg.I
    P = T * k
    xb = IN.make_x(cfg, call=3)
    x = bits_to_device(xb)
    ws = make_workspace(T, d, E, k, I, B.MOE_ACT_BF16)
    i32 = dict(dtype=torch.int32, device="cuda")
    ids, w = torch.empty((T, k), **i32), torch.empty((T, k), dtype=torch.float32, device="cuda")
    counts, offsets, perm, inv = (torch.empty(E, **i32), torch.empty(E + 1, **i32), torch.empty(P, **i32),
                                  torch.empty(P, **i32))
    h = torch.empty((P, I), dtype=torch.bfloat16, device="cuda")
    y_perm = torch.empty((P, d), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((T, d), dtype=torch.bfloat16, device="cuda")
    B.moe_route(x, layer.W_r, layer.b, T, d, E, k, ids, w, ws)
    B.moe_permute(x, ids, T, d, E, k, B.MOE_ACT_BF16, counts, offsets, perm, inv, None, None, ws)
    B.moe_expert_up_swiglu(x, None, None, B.MOE_ACT_BF16, perm, offsets, T, d, E, k, I, layer.weights, h, None, ws)
    B.moe_expert_down(h, None, B.MOE_ACT_BF16, perm, offsets, T, d, E, k, I, layer.weights, y_perm, ws)
    B.moe_combine(y_perm, inv, w, T, k, d, y)
    y_fused = layer_forward(layer, x, B.MOE_ACT_BF16)
    assert torch.equal(y.view(torch.int16), y_fused.view(torch.int16))
    # h and y_perm rows against the oracle's intermediates
    ref = O.moe_layer(xb, layer.W_r_host, layer.b_host, k, oracle_expert_weights(cfg, layer.seed), O.ACT_BF16,
                      want_intermediates=True)
    inv_h = inv.cpu().numpy().reshape(T, k)
    h_gpu = bf16_tensor_to_f32(h)
    yp_gpu = bf16_tensor_to_f32(y_perm)
    h_ref = np.stack([ref["h"][(t, j)][0] for t in range(T) for j in range(k)])
    yp_ref = np.stack([ref["y_perm"][(t, j)] for t in range(T) for j in range(k)])
    rows = inv_h.reshape(-1)
    check_outputs(h_gpu[rows], h_ref, "h")
    check_outputs(yp_gpu[rows], yp_ref, "y_perm")


def test_zero_tokens_and_zero_input():
    layer = get_layer("tiny")
    cfg = layer.cfg
    x0 = torch.zeros((0, cfg.d), dtype=torch.bfloat16, device="cuda")
    ws = make_workspace(1, cfg.d, cfg.E, cfg.k, cfg.I, B.MOE_ACT_BF16)
    y0 = torch.empty((0, cfg.d), dtype=torch.bfloat16, device="cuda")
    B.moe_layer_forward(x0, layer.W_r, layer.b, 0, cfg.d, cfg.E, cfg.k, cfg.I, layer.weights, B.MOE_ACT_BF16, y0,
                        None, None, ws)
    xz = torch.zeros((5, cfg.d), dtype=torch.bfloat16, device="cuda")
    y, ids, w = layer_forward(layer, xz, B.MOE_ACT_BF16, want_routing=True)
    assert torch.count_nonzero(y.float()) == 0
    np.testing.assert_array_equal(ids.cpu().numpy(), np.tile(np.arange(cfg.k), (5, 1)))


def test_bad_arguments_are_rejected():
    layer = get_layer("tiny")
    cfg = layer.cfg
    x = torch.zeros((4, cfg.d), dtype=torch.bfloat16, device="cuda")
    y = torch.empty_like(x)
    ws = make_workspace(4, cfg.d, cfg.E, cfg.k, cfg.I, B.MOE_ACT_BF16)
    with pytest.raises(B.MoeError) as e:
        B.moe_layer_forward(x, layer.W_r, layer.b, 4, cfg.d, cfg.E, cfg.k, cfg.I, layer.weights, B.MOE_ACT_BF16, y,
                            None, None, ws, ws_bytes=1024)
    assert e.value.status == B.MOE_ERR_WORKSPACE
    with pytest.raises(B.MoeError) as e:
        B.moe_layer_forward(x, layer.W_r, layer.b, 4, cfg.d, cfg.E, cfg.E + 1, cfg.I, layer.weights,
                            B.MOE_ACT_BF16, y, None, None, ws)
    assert e.value.status == B.MOE_ERR_UNSUPPORTED_SHAPE


@pytest.mark.parametrize("name", ["tiny", "decode", "spec_verify", "ring_t3", "ring_t2"])
def test_tensor_core_step_calls_equal_layer_call(name):
    """moe_route -> moe_permute -> moe_decode_pieces -> moe_expert_ffn_decode (-> moe_combine
    beyond four tokens) gives the layer call's output bit for bit, and the expert outputs match the
    oracle's intermediates."""
    layer = get_layer(name, mma=True)
    cfg = layer.cfg
    T, d, E, k, I = cfg.T, cfg.d, cfg.E, cfg.k, cfg.I
    P = T * k
    xb = IN.make_x(cfg, call=4)
    x = bits_to_device(xb)
    ws = make_workspace(T, d, E, k, I, B.MOE_ACT_BF16)
    i32 = dict(dtype=torch.int32, device="cuda")
    u8 = dict(dtype=torch.uint8, device="cuda")
    ids, w = torch.empty((T, k), **i32), torch.empty((T, k), dtype=torch.float32, device="cuda")
    counts, offsets, perm, inv = (torch.empty(E, **i32), torch.empty(E + 1, **i32), torch.empty(P, **i32),
                                  torch.empty(P, **i32))
    xa = torch.empty(B.moe_decode_pieces_bytes(T, d, 0), **u8)
    xa_s = torch.empty(B.moe_decode_pieces_bytes(T, d, 1), **u8)
    y_perm = torch.empty((P, d), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((T, d), dtype=torch.bfloat16, device="cuda")
    B.moe_route(x, layer.W_r, layer.b, T, d, E, k, ids, w, ws)
    B.moe_permute(x, ids, T, d, E, k, B.MOE_ACT_BF16, counts, offsets, perm, inv, None, None, ws)
    B.moe_decode_pieces(x, T, d, B.MOE_ACT_BF16, xa, xa_s)
    fused = T <= 4
    B.moe_expert_ffn_decode(xa, xa_s, B.MOE_ACT_BF16, perm, offsets, inv, w, T, d, E, k, I, layer.weights, y_perm,
                            y if fused else None, ws)
    if not fused:
        B.moe_combine(y_perm, inv, w, T, k, d, y)
    y_layer = layer_forward(layer, x, B.MOE_ACT_BF16)
    torch.cuda.synchronize()
    assert B.moe_get_device_status(ws) == B.MOE_OK
    assert torch.equal(y.view(torch.int16), y_layer.view(torch.int16))
    ref = O.moe_layer(xb, layer.W_r_host, layer.b_host, k, oracle_expert_weights(cfg, layer.seed), O.ACT_BF16,
                      want_intermediates=True)
    rows = inv.cpu().numpy()
    yp_ref = np.stack([ref["y_perm"][(t, j)] for t in range(T) for j in range(k)])
    check_outputs(bf16_tensor_to_f32(y_perm)[rows], yp_ref, "y_perm")
    check_outputs(bf16_tensor_to_f32(y), ref["y"], "y")
