"""GPU parity of the dense MXFP4 linear map (the shared latent projections, the oracle's reading
R9) on the GEMV path and the tcgen05 path, and of a latent layer composed from it: narrow x to the
latent width, the MoE layer at that width, widen the result back."""
import numpy as np
import pytest
import torch

from bit_expert_ffn_moe_gb300 import binding as B
from bit_expert_ffn_moe_gb300 import inputs as IN
from bit_expert_ffn_moe_gb300.layer import DeviceLayer, layer_forward, make_workspace
from moe_testlib import bf16_tensor_to_f32, bits_to_device, check_outputs, oracle_expert_weights, oracle_matrix
from oracle import oracle as O

pytestmark = pytest.mark.gpu

TENSOR_W_IN, TENSOR_W_OUT = 10, 11


def device_matrix(q, s, with_mma):
    """Host-packed MXFP4 bytes on the device (+ the tensor-core copies for the MXFP4 path)."""
    N, K = q.shape[0], q.shape[1] * 2
    qd, sd = torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda()
    keep = [qd, sd]
    q_mma = s_mma = None
    if with_mma:
        q_mma = torch.empty(N * K // 2, dtype=torch.uint8, device="cuda")
        s_mma = torch.empty(B.moe_mxfp4_mma_scale_bytes(N, K), dtype=torch.uint8, device="cuda")
        B.moe_mxfp4_codes_to_mma(qd, N, K, q_mma)
        B.moe_mxfp4_scales_to_mma(sd, N, K, s_mma)
        keep += [q_mma, s_mma]
    return B.mxfp4_matrix_struct(qd, sd, q_mma, s_mma), keep


ACT = {"bf16": B.MOE_ACT_BF16, "mxfp4": B.MOE_ACT_MXFP4, "mxfp8": B.MOE_ACT_MXFP8}
OACT = {"bf16": O.ACT_BF16, "mxfp4": O.ACT_MXFP4, "mxfp8": O.ACT_MXFP8}


def gpu_dense(xb, W, N, fmt):
    T, K = xb.shape
    act = ACT[fmt]
    ws = torch.empty(B.moe_dense_workspace_size(T, K, N, act), dtype=torch.uint8, device="cuda")
    B.moe_workspace_init(ws)
    y = torch.empty((T, N), dtype=torch.bfloat16, device="cuda")
    B.moe_dense_linear(bits_to_device(xb), T, K, N, W, act, y, ws)
    assert B.moe_get_device_status(ws) == B.MOE_OK
    return y


DENSE_CASES = [
    # (T, K, N, format, rows checked or None for all)
    (1, 8192, 4096, "bf16", None),      # decode-sized latent projection (one-token ring GEMV)
    (2, 512, 256, "bf16", None),
    (5, 256, 512, "bf16", None),        # warp-per-row GEMV
    (50, 256, 512, "mxfp4", None),      # one ragged token tile
    (300, 512, 256, "mxfp4", None),     # two full tiles and a ragged one
    (4096, 8192, 4096, "mxfp4", 48),    # prefill-sized, sampled rows
    (50, 256, 512, "mxfp8", None),      # kind::mxf8f6f4: one ragged token tile
    (300, 512, 256, "mxfp8", None),
    (4096, 8192, 4096, "mxfp8", 48),
]


@pytest.mark.parametrize("T,K,N,fmt,n_check", DENSE_CASES, ids=["%dx%dx%d-%s" % c[:4] for c in DENSE_CASES])
def test_dense_linear_matches_oracle(T, K, N, fmt, n_check):
    seed = 5000 + T + K + N
    q, s = oracle_matrix(seed, TENSOR_W_IN, 0, N, K, 0.02)
    W, _keep = device_matrix(q, s, fmt != "bf16")
    rng = np.random.default_rng(seed)
    xb = IN.to_bf16_bits(rng.standard_normal((T, K)).astype(np.float32))
    y = bf16_tensor_to_f32(gpu_dense(xb, W, N, fmt))
    rows = np.arange(T) if n_check is None else np.sort(rng.choice(T, n_check, replace=False))
    ref = O.dense_linear(xb[rows], (q, s), OACT[fmt])
    check_outputs(y[rows], ref, "dense %dx%dx%d %s" % (T, K, N, fmt))


LATENT_CASES = [
    # (name, T, d, latent width, E, k, I, format)
    ("latent_tiny_bf16", 16, 512, 256, 8, 2, 256, "bf16"),
    ("latent_tiny_mx", 16, 512, 256, 8, 2, 256, "mxfp4"),
    ("latent_decode_bf16", 1, 8192, 4096, 128, 8, 2048, "bf16"),
]


@pytest.mark.parametrize("name,T,d,dl,E,k,I,fmt", LATENT_CASES, ids=[c[0] for c in LATENT_CASES])
def test_latent_layer_matches_oracle(name, T, d, dl, E, k, I, fmt):
    cfg = IN.small_config(name, T=T, d=dl, E=E, k=k, I=I, index=130 + [c[0] for c in LATENT_CASES].index(name))
    layer = DeviceLayer(cfg)  # experts and router at the latent width
    act = B.MOE_ACT_BF16 if fmt == "bf16" else B.MOE_ACT_MXFP4
    oact = O.ACT_BF16 if fmt == "bf16" else O.ACT_MXFP4
    w_in = oracle_matrix(cfg.seed, TENSOR_W_IN, 0, dl, d, 0.02)
    w_out = oracle_matrix(cfg.seed, TENSOR_W_OUT, 0, d, dl, 0.02)
    Win, _k1 = device_matrix(*w_in, fmt == "mxfp4")
    Wout, _k2 = device_matrix(*w_out, fmt == "mxfp4")
    rng = np.random.default_rng(cfg.seed)
    xb = IN.to_bf16_bits(rng.standard_normal((T, d)).astype(np.float32))
    # GPU: narrow, the layer at the latent width, widen
    xl = gpu_dense(xb, Win, dl, fmt)
    yl, ids, _w = layer_forward(layer, xl, act, want_routing=True)
    y = bf16_tensor_to_f32(gpu_dense(yl.view(torch.int16).cpu().numpy().view(np.uint16), Wout, d, fmt))
    # oracle: the same three steps on its own values
    xl_o = O.dense_linear(xb, w_in, oact)
    ref_l = O.moe_layer(IN.to_bf16_bits(xl_o), layer.W_r_host, layer.b_host, k, oracle_expert_weights(cfg, layer.seed),
                        oact)
    y_o = O.dense_linear(IN.to_bf16_bits(ref_l["y"]), w_out, oact)
    np.testing.assert_array_equal(ids.cpu().numpy(), ref_l["ids"])
    check_outputs(bf16_tensor_to_f32(xl), xl_o, name + " narrowed")
    check_outputs(y, y_o, name)
