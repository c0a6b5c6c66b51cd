"""GPU parity of NVFP4 expert weights (E2M1 codes, one E4M3 scale per 16 values, one fp32 global
scale per matrix): the packer and unpacker bit for bit against the oracle's; on the bf16-activation
path the layer against the oracle on every GEMV kernel variant -- warp-per-row gate/up and down,
the CTA-split gate/up for one and two token rows, the copy-engine down ring for one, two and four
tokens, the fused weighted sum and the unfused one of the expert-normalised layer; with MXFP4
activations the tcgen05 kind::mxf4nvf4 grouped GEMMs (tiny, ragged token tiles, the prefill
workload) and their step calls."""
import numpy as np
import pytest
import torch

from bit_expert_ffn_moe_gb300 import binding as B
from bit_expert_ffn_moe_gb300 import inputs as IN
from bit_expert_ffn_moe_gb300.layer import DeviceLayer, layer_forward, make_workspace
from moe_testlib import bf16_tensor_to_f32, bits_to_device, check_outputs, check_weights, oracle_expert_weights_nv
from oracle import oracle as O

pytestmark = pytest.mark.gpu


def adversarial_weights(seed, n, rows, K):
    """Random rows over a wide range of magnitudes, plus blocks that hit the rule's corner cases:
    exact rounding ties, an all-zero block, blocks too small for the smallest E4M3 scale, and
    blocks whose scale is an E4M3 subnormal."""
    rng = np.random.default_rng(seed)
    w = (rng.standard_normal((n, rows, K)) * np.exp(rng.uniform(-4, 4, (n, rows, 1)))).astype(np.float32)
    w[0] *= np.float32(1e-3)
    w[0, 0, 0] = 2688.0  # global scale exactly 1 for matrix 0
    w[0, 1, :16] = [6.0, 1.25, 2.5, 5.0, 0.25, 0.75, -1.75, -3.5, -0.25, 3.0, 0.0, -6.0, 4.0, 1.0, 0.5, -2.0]
    w[0, 2, :16] = 0.0
    w[0, 3, :16] = np.float32(1e-7)
    w[0, 4, :16] = np.linspace(-0.01, 0.01, 16, dtype=np.float32)
    return w


PACK_CASES = [(1, 64, 256), (3, 40, 96), (2, 128, 2048), (5, 7, 32)]


@pytest.mark.parametrize("n,rows,K", PACK_CASES, ids=["%dx%dx%d" % c for c in PACK_CASES])
def test_pack_and_unpack_match_oracle_bit_for_bit(n, rows, K):
    w = adversarial_weights(100 + n + rows + K, n, rows, K)
    q_ref, s_ref, gs_ref = O.nvfp4_pack(w)
    wd = torch.from_numpy(w).cuda()
    q = torch.empty((n, rows, K // 2), dtype=torch.uint8, device="cuda")
    s = torch.empty((n, rows, K // 16), dtype=torch.uint8, device="cuda")
    gs = torch.empty(n, dtype=torch.float32, device="cuda")
    B.moe_nvfp4_pack(wd, n, rows, K, q, s, gs)
    np.testing.assert_array_equal(gs.cpu().numpy(), gs_ref)
    np.testing.assert_array_equal(s.cpu().numpy(), s_ref)
    np.testing.assert_array_equal(q.cpu().numpy(), q_ref)
    out = torch.empty((n, rows, K), dtype=torch.float32, device="cuda")
    B.moe_nvfp4_unpack(q, s, gs, n, rows, K, out)
    np.testing.assert_array_equal(out.cpu().numpy(), O.nvfp4_unpack(q_ref, s_ref, gs_ref).astype(np.float32))


def test_device_packed_layer_weights_equal_the_oracle_packing():
    cfg = IN.small_config("nv_pack", T=4, d=256, E=3, k=2, I=96, index=140)
    layer = DeviceLayer(cfg, wfmt="nvfp4")
    get = oracle_expert_weights_nv(cfg, layer.seed)
    for e in range(cfg.E):
        ref = get(e)
        for name, tid in (("gate", IN.TENSOR_GATE), ("up", IN.TENSOR_UP), ("down", IN.TENSOR_DOWN)):
            q, s, g = ref[name]
            np.testing.assert_array_equal(layer.q[tid][e].cpu().numpy(), q)
            np.testing.assert_array_equal(layer.s[tid][e].cpu().numpy(), s)
            assert layer.gs[tid][e].item() == g


CASES = {
    # warp-per-row gate/up and down (more than four tokens)
    "nv_tiny": IN.small_config("nv_tiny", T=16, d=256, E=8, k=2, I=512, index=141),
    # CTA-split gate/up (one row) + down ring (one token)
    "nv_t1": IN.small_config("nv_t1", T=1, d=1024, E=16, k=4, I=1024, index=142),
    # CTA-split gate/up (two rows) + down ring (two tokens)
    "nv_t2": IN.small_config("nv_t2", T=2, d=2048, E=6, k=3, I=1536, index=143),
    # CTA-split gate/up in two passes + down ring (four-token variant)
    "nv_t3": IN.small_config("nv_t3", T=3, d=1024, E=12, k=4, I=512, index=144),
    # ragged: I % 32 only, several tokens per expert
    "nv_ragged": IN.small_config("nv_ragged", T=9, d=384, E=5, k=3, I=96, index=145),
}

_layers = {}


def get_layer(name):
    if name not in _layers:
        _layers.clear()
        torch.cuda.empty_cache()
        _layers[name] = DeviceLayer(CASES[name] if name in CASES else IN.CONFIGS[name], wfmt="nvfp4")
    return _layers[name]


def oracle_layer(layer, xb, tokens=None, eps=None):
    cfg = layer.cfg
    return O.moe_layer(xb, layer.W_r_host, layer.b_host, cfg.k, oracle_expert_weights_nv(cfg, layer.seed), O.ACT_BF16,
                       tokens=tokens, expert_norm_eps=eps)


LAYER_CASES = [("nv_tiny", [0, 1]), ("nv_t1", [0, 1]), ("nv_t2", [0]), ("nv_t3", [0, 1]), ("nv_ragged", [0]),
               ("decode", [0, 1]), ("spec_verify", [0])]


@pytest.mark.parametrize("name,calls", LAYER_CASES, ids=[c[0] for c in LAYER_CASES])
def test_nvfp4_layer_matches_oracle(name, calls):
    layer = get_layer(name)
    cfg = layer.cfg
    ws = make_workspace(cfg.T, cfg.d, cfg.E, cfg.k, cfg.I, B.MOE_ACT_BF16)
    for call in calls:
        xb = IN.make_x(cfg, call=call)
        y, ids, w = layer_forward(layer, bits_to_device(xb), B.MOE_ACT_BF16, ws=ws, want_routing=True)
        ref = oracle_layer(layer, xb)
        np.testing.assert_array_equal(ids.cpu().numpy(), ref["ids"])
        check_weights(w.cpu().numpy(), ref["w"])
        check_outputs(bf16_tensor_to_f32(y), ref["y"], "nvfp4 %s call %d" % (name, call))
    assert B.moe_get_device_status(ws) == B.MOE_OK


@pytest.mark.parametrize("name", ["nv_tiny", "nv_t1", "nv_t3"])
def test_nvfp4_expert_normalised_layer_matches_oracle(name):
    layer = get_layer(name)
    cfg = layer.cfg
    xb = IN.make_x(cfg, call=2)
    y = layer_forward(layer, bits_to_device(xb), B.MOE_ACT_BF16, expert_norm_eps=O.EXPERT_NORM_EPS)
    ref = oracle_layer(layer, xb, eps=O.EXPERT_NORM_EPS)
    check_outputs(bf16_tensor_to_f32(y), ref["y"], "nvfp4 normalised " + name)


@pytest.mark.parametrize("name", ["nv_tiny", "nv_t2"])
def test_nvfp4_step_calls_equal_layer_call(name):
    layer = get_layer(name)
    cfg = layer.cfg
    T, d, E, k, I = cfg.T, cfg.d, cfg.E, cfg.k, cfg.I
    P = T * k
    x = bits_to_device(IN.make_x(cfg, call=3))
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
    assert B.moe_get_device_status(ws) == B.MOE_OK


NV_MX = {
    "nv_tiny": CASES["nv_tiny"],
    # several token tiles per expert and ragged ones, I = 768 (three 256-value K steps of down)
    "nv_mx_prefill": IN.small_config("nv_mx_prefill", T=300, d=512, E=10, k=2, I=768, index=146, zipf_s=1.2),
}


def get_nv_mx_layer(name):
    key = "mx:" + name
    if key not in _layers:
        _layers.clear()
        torch.cuda.empty_cache()
        _layers[key] = DeviceLayer(NV_MX[name] if name in NV_MX else IN.CONFIGS[name], wfmt="nvfp4")
    return _layers[key]


@pytest.mark.parametrize("name,call", [("nv_tiny", 0), ("nv_tiny", 1), ("nv_mx_prefill", 0), ("prefill", 0)])
def test_nvfp4_weights_on_the_tensor_cores_match_oracle(name, call):
    """MXFP4 activations x NVFP4 weights on tcgen05 kind::mxf4nvf4 (16-element UE4M3 scales): the
    operands keep their E2M1 codes, their E8M0 block scales become UE4M3 powers of two with one
    power-of-two factor per row, and the epilogues apply that factor and the weight matrices'
    global scales."""
    layer = get_nv_mx_layer(name)
    cfg = layer.cfg
    xb = IN.make_x(cfg, call=call)
    ws = make_workspace(cfg.T, cfg.d, cfg.E, cfg.k, cfg.I, B.MOE_ACT_MXFP4)
    y, ids, w = layer_forward(layer, bits_to_device(xb), B.MOE_ACT_MXFP4, ws=ws, want_routing=True)
    torch.cuda.synchronize()
    assert B.moe_get_device_status(ws) == B.MOE_OK
    tokens = IN.sample_tokens(cfg, cfg.T) if cfg.sample_tokens else None
    ref = O.moe_layer(xb, layer.W_r_host, layer.b_host, cfg.k, oracle_expert_weights_nv(cfg, layer.seed),
                      O.ACT_MXFP4, tokens=tokens)
    np.testing.assert_array_equal(ids.cpu().numpy(), ref["ids"])
    check_weights(w.cpu().numpy(), ref["w"])
    yg = bf16_tensor_to_f32(y)
    if tokens is not None:
        yg = yg[tokens]
    check_outputs(yg, ref["y"], "nvfp4 x mxfp4 %s call %d" % (name, call))


def test_nvfp4_tensor_core_step_calls_equal_layer_call_and_oracle_h():
    layer = get_nv_mx_layer("nv_mx_prefill")
    cfg = layer.cfg
    T, d, E, k, I = cfg.T, cfg.d, cfg.E, cfg.k, cfg.I
    P = T * k
    fmt = B.MOE_ACT_MXFP4
    xb = IN.make_x(cfg, call=2)
    x = bits_to_device(xb)
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
    y_layer = layer_forward(layer, x, fmt)
    torch.cuda.synchronize()
    assert B.moe_get_device_status(ws) == B.MOE_OK
    assert torch.equal(y.view(torch.int16), y_layer.view(torch.int16))
    ref = O.moe_layer(xb, layer.W_r_host, layer.b_host, k, oracle_expert_weights_nv(cfg, layer.seed), fmt,
                      want_intermediates=True)
    # h: the MXFP4 values against the oracle's (decisions in fp32 on both sides)
    from test_gpu_layer_mxfp4 import mma_scales_to_rows, mma_tiles_to_rows, unpad
    from test_oracle_pins import np_unpack
    cn, on = counts.cpu().numpy(), offsets.cpu().numpy()
    pad = np.concatenate([[0], np.cumsum((cn + 127) // 128 * 128)])
    h_gpu = np_unpack(unpad(mma_tiles_to_rows(h.cpu().numpy(), R, I), pad, cn, on),
                      unpad(mma_scales_to_rows(h_s.cpu().numpy(), R, I), pad, cn, on))
    rows = inv.cpu().numpy()
    h_ref = np.zeros_like(h_gpu)
    yp_ref = np.zeros((P, d), np.float32)
    for t in range(T):
        for j in range(k):
            h_ref[rows[t * k + j]] = ref["h"][(t, j)][0]
            yp_ref[rows[t * k + j]] = ref["y_perm"][(t, j)]
    check_outputs(h_gpu, h_ref, "h")
    assert np.mean(h_gpu == h_ref) > 0.99
    check_outputs(bf16_tensor_to_f32(y_perm), yp_ref, "y_perm")
    check_outputs(bf16_tensor_to_f32(y), ref["y"], "y")


def test_nvfp4_tensor_core_layer_with_normalised_expert_outputs():
    layer = get_nv_mx_layer("nv_mx_prefill")
    cfg = layer.cfg
    xb = IN.make_x(cfg, call=3)
    y = layer_forward(layer, bits_to_device(xb), B.MOE_ACT_MXFP4, expert_norm_eps=O.EXPERT_NORM_EPS)
    ref = O.moe_layer(xb, layer.W_r_host, layer.b_host, cfg.k, oracle_expert_weights_nv(cfg, layer.seed),
                      O.ACT_MXFP4, expert_norm_eps=O.EXPERT_NORM_EPS)
    check_outputs(bf16_tensor_to_f32(y), ref["y"], "nvfp4 x mxfp4 normalised")


def test_nvfp4_weights_are_refused_where_no_kernel_takes_them():
    layer = get_layer("nv_tiny")
    cfg = layer.cfg
    x = bits_to_device(IN.make_x(cfg))
    # MXFP8 activations: kind::mxf8f6f4 takes E8M0 scales per 32 only
    with pytest.raises(B.MoeError) as err:
        layer_forward(layer, x, B.MOE_ACT_MXFP8)
    assert err.value.status == B.MOE_ERR_UNSUPPORTED_SHAPE
    # MXFP4 activations without the weights' tensor-core copies
    bare = DeviceLayer(cfg, wfmt="nvfp4", mma_layouts=False)
    with pytest.raises(B.MoeError) as err:
        layer_forward(bare, x, B.MOE_ACT_MXFP4)
    assert err.value.status == B.MOE_ERR_INVALID_ARG
