"""GPU parity of the layer with each expert's output normalised before the weighted sum (RMSNorm
over d, eps 1e-6, the oracle's reading R8), on the GEMV path (one, two and many tokens) and on the
tcgen05 path, and of the step entry point moe_combine_norm against the fused call."""
import numpy as np
import pytest
import torch

from bit_expert_ffn_moe_gb300 import binding as B
from bit_expert_ffn_moe_gb300 import inputs as IN
from bit_expert_ffn_moe_gb300.layer import DeviceLayer, layer_forward, make_workspace
from moe_testlib import bf16_tensor_to_f32, bits_to_device, check_outputs, check_weights, oracle_expert_weights
from oracle import oracle as O

pytestmark = pytest.mark.gpu

EPS = 1e-6

CASES = [
    # (config, activation format, calls, sampled tokens or None)
    (IN.CONFIGS["tiny"], "bf16", [0, 1], None),
    (IN.small_config("norm_t1", T=1, d=1024, E=16, k=4, I=1024, index=120), "bf16", [0, 1], None),
    (IN.small_config("norm_t2", T=2, d=2048, E=6, k=3, I=1536, index=121), "bf16", [0], None),
    (IN.CONFIGS["decode"], "bf16", [0], None),
    (IN.CONFIGS["tiny"], "mxfp4", [0, 1], None),
    (IN.CONFIGS["prefill"], "mxfp4", [0], 64),
    # 8-bit activations: the decode kernels (one token) and the kind::mxf8f6f4 GEMMs (200 tokens)
    (IN.small_config("norm_mx8_t1", T=1, d=1024, E=16, k=4, I=1024, index=122), "mxfp8", [0], None),
    (IN.small_config("norm_mx8_pf", T=200, d=512, E=8, k=2, I=768, index=123), "mxfp8", [0], None),
]
ACT = {"bf16": (B.MOE_ACT_BF16, O.ACT_BF16), "mxfp4": (B.MOE_ACT_MXFP4, O.ACT_MXFP4),
       "mxfp8": (B.MOE_ACT_MXFP8, O.ACT_MXFP8)}


@pytest.mark.parametrize("cfg,fmt,calls,n_sample", CASES, ids=[c[0].name + "-" + c[1] for c in CASES])
def test_normalised_layer_matches_oracle(cfg, fmt, calls, n_sample):
    layer = DeviceLayer(cfg)
    act, oact = ACT[fmt]
    ws = make_workspace(cfg.T, cfg.d, cfg.E, cfg.k, cfg.I, act)
    for call in calls:
        xb = IN.make_x(cfg, call=call)
        y, ids, w = layer_forward(layer, bits_to_device(xb), act, ws=ws, want_routing=True, expert_norm_eps=EPS)
        tokens = None if n_sample is None else IN.sample_tokens(cfg, n_sample)
        ref = O.moe_layer(xb, layer.W_r_host, layer.b_host, cfg.k, oracle_expert_weights(cfg, layer.seed), oact,
                          tokens=tokens, expert_norm_eps=EPS)
        np.testing.assert_array_equal(ids.cpu().numpy(), ref["ids"])
        check_weights(w.cpu().numpy(), ref["w"])
        yg = bf16_tensor_to_f32(y)
        if tokens is not None:
            yg = yg[tokens]
        check_outputs(yg, ref["y"], "%s %s call %d" % (cfg.name, fmt, call))
        # the normalised output differs from the plain layer's
        y_plain = layer_forward(layer, bits_to_device(xb), act, ws=ws)
        assert not torch.equal(y.view(torch.int16), y_plain.view(torch.int16))
    assert B.moe_get_device_status(ws) == B.MOE_OK


@pytest.mark.parametrize("name,fmt", [("norm_t2", "bf16"), ("tiny", "bf16"), ("tiny", "mxfp4")])
def test_step_combine_norm_equals_layer_call(name, fmt):
    cfg = IN.CONFIGS[name] if name in IN.CONFIGS else next(c[0] for c in CASES if c[0].name == name)
    layer = DeviceLayer(cfg)
    act = B.MOE_ACT_BF16 if fmt == "bf16" else B.MOE_ACT_MXFP4
    T, d, E, k, I = cfg.T, cfg.d, cfg.E, cfg.k, cfg.I
    P = T * k
    xb = IN.make_x(cfg, call=2)
    x = bits_to_device(xb)
    ws = make_workspace(T, d, E, k, I, act)
    i32 = dict(dtype=torch.int32, device="cuda")
    u8 = dict(dtype=torch.uint8, device="cuda")
    ids, w = torch.empty((T, k), **i32), torch.empty((T, k), dtype=torch.float32, device="cuda")
    counts, offsets, perm, inv = (torch.empty(E, **i32), torch.empty(E + 1, **i32), torch.empty(P, **i32),
                                  torch.empty(P, **i32))
    y_perm = torch.empty((P, d), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((T, d), dtype=torch.bfloat16, device="cuda")
    B.moe_route(x, layer.W_r, layer.b, T, d, E, k, ids, w, ws)
    if act == B.MOE_ACT_BF16:
        B.moe_permute(x, ids, T, d, E, k, act, counts, offsets, perm, inv, None, None, ws)
        h = torch.empty((P, I), dtype=torch.bfloat16, device="cuda")
        B.moe_expert_up_swiglu(x, None, None, act, perm, offsets, T, d, E, k, I, layer.weights, h, None, ws)
        B.moe_expert_down(h, None, act, perm, offsets, T, d, E, k, I, layer.weights, y_perm, ws)
    else:
        R = B.moe_padded_rows(T, k, E)
        xa, xa_s = torch.zeros((R, d // 2), **u8), torch.zeros(B.moe_mxfp4_mma_scale_bytes(R, d), **u8)
        h, h_s = torch.zeros((R, I // 2), **u8), torch.zeros(B.moe_mxfp4_mma_scale_bytes(R, I), **u8)
        B.moe_permute(x, ids, T, d, E, k, act, counts, offsets, perm, inv, xa, xa_s, ws)
        B.moe_expert_up_swiglu(None, xa, xa_s, act, perm, offsets, T, d, E, k, I, layer.weights, h, h_s, ws)
        B.moe_expert_down(h, h_s, act, perm, offsets, T, d, E, k, I, layer.weights, y_perm, ws)
    B.moe_combine_norm(y_perm, inv, w, T, k, d, EPS, y)
    y_layer = layer_forward(layer, x, act, expert_norm_eps=EPS)
    assert torch.equal(y.view(torch.int16), y_layer.view(torch.int16))
    assert B.moe_get_device_status(ws) == B.MOE_OK
