"""GPU parity at the edges of the supported shapes and at the degenerate cases of the method:
the largest E and k (1024 experts, k = 32), the one-launch router at its largest T and the tiled
router just above it, the smallest hidden size, k = 1, a single expert (the layer is then a
dense SwiGLU FFN) and every expert chosen by every token (k = E), on both expert paths; the layer
call's permutation (read out of its workspace) bit for bit in each."""
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

ROUTE_EDGES = {
    # one-launch router (T <= 8): 32 logits per lane in the top-k registers, k at its maximum
    "e1024_k32_t7": IN.small_config("e1024_k32_t7", T=7, d=256, E=1024, k=32, I=256, index=96),
    # one-launch router at its largest T
    "e300_t8": IN.small_config("e300_t8", T=8, d=512, E=300, k=8, I=256, index=97),
    # tiled router + top-k kernel, E not a multiple of 32
    "e1000_k17_t70": IN.small_config("e1000_k17_t70", T=70, d=256, E=1000, k=17, I=256, index=98),
    # smallest hidden size, k = 1, just above the one-launch router's T
    "d128_e3_k1_t9": IN.small_config("d128_e3_k1_t9", T=9, d=128, E=3, k=1, I=256, index=99),
}


@pytest.mark.parametrize("name", list(ROUTE_EDGES))
def test_route_and_permute_at_shape_edges(name):
    cfg = ROUTE_EDGES[name]
    T, d, E, k = cfg.T, cfg.d, cfg.E, cfg.k
    xb = IN.make_x(cfg)
    W_r, b = IN.make_router(cfg)
    ws = make_workspace(T, d, E, k, 256, B.MOE_ACT_BF16)
    dev = dict(dtype=torch.int32, device="cuda")
    ids = torch.empty((T, k), **dev)
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    B.moe_route(bits_to_device(xb), torch.from_numpy(W_r).cuda(), None if b is None else torch.from_numpy(b).cuda(),
                T, d, E, k, ids, w, ws)
    ids_o, w_o = O.topk_softmax(O.router_logits(xb, W_r, b), k)
    np.testing.assert_array_equal(ids.cpu().numpy(), ids_o)
    check_weights(w.cpu().numpy(), w_o)
    P = T * k
    counts, offsets = torch.empty(E, **dev), torch.empty(E + 1, **dev)
    perm, inv = torch.empty(P, **dev), torch.empty(P, **dev)
    B.moe_permute(None, torch.from_numpy(ids_o).cuda(), T, d, E, k, B.MOE_ACT_BF16, counts, offsets, perm, inv,
                  None, None, ws)
    for got, want in zip((counts, offsets, perm, inv), O.permute(ids_o, E)):
        np.testing.assert_array_equal(got.cpu().numpy(), want)
    assert B.moe_get_device_status(ws) == B.MOE_OK


LAYER_EDGES = [
    # (name, T, d, E, k, I, activation format, seed index)
    ("dense_t1_bf16", 1, 256, 1, 1, 256, "bf16", 110),       # CTA-split GEMVs, one expert
    ("dense_t2_bf16", 2, 512, 1, 1, 512, "bf16", 111),       # two tokens on the one expert
    ("dense_t5_bf16", 5, 256, 1, 1, 256, "bf16", 112),       # warp-per-row GEMVs
    ("dense_t50_mx", 50, 256, 1, 1, 256, "mxfp4", 113),      # tcgen05 path, one ragged token tile
    ("all_experts_t2_bf16", 2, 256, 4, 4, 256, "bf16", 114),  # two rows on every expert
    ("all_experts_t3_bf16", 3, 256, 4, 4, 256, "bf16", 115),
    ("all_experts_t40_mx", 40, 256, 4, 4, 256, "mxfp4", 116),
    # the layer call's counting top-k (32 keys per lane) and one-launch permutation at 1000
    # experts, k = 17 (the ids read one by one): GEMVs beyond 8 tokens, and the screened router
    # with the tcgen05 path from 256 tokens on
    ("e1000_k17_t70_bf16", 70, 256, 1000, 17, 256, "bf16", 117),
    ("e1000_k17_t300_mx", 300, 256, 1000, 17, 256, "mxfp4", 118),
]


@pytest.mark.parametrize("name,T,d,E,k,I,fmt,index", LAYER_EDGES)
def test_layer_at_degenerate_routing(name, T, d, E, k, I, fmt, index):
    cfg = IN.small_config(name, T=T, d=d, E=E, k=k, I=I, index=index)
    layer = DeviceLayer(cfg)
    act = B.MOE_ACT_BF16 if fmt == "bf16" else B.MOE_ACT_MXFP4
    xb = IN.make_x(cfg)
    ws = make_workspace(T, d, E, k, I, act)
    y, ids, w = layer_forward(layer, bits_to_device(xb), act, ws=ws, want_routing=True)
    ref = O.moe_layer(xb, layer.W_r_host, layer.b_host, k, oracle_expert_weights(cfg, layer.seed),
                      O.ACT_BF16 if fmt == "bf16" else O.ACT_MXFP4)
    ids_h = ids.cpu().numpy()
    np.testing.assert_array_equal(ids_h, ref["ids"])
    # k = E: every token holds every expert, in ascending order
    if k == E:
        np.testing.assert_array_equal(ids_h, np.tile(np.arange(E), (T, 1)))
    check_weights(w.cpu().numpy(), ref["w"])
    # the permutation the layer call built in its workspace, bit for bit
    check_permutation(workspace_routing(ws, T, d, E, k, I, act), ref)
    if E == 1:
        np.testing.assert_array_equal(w.cpu().numpy(), np.ones((T, 1), np.float32))
    check_outputs(bf16_tensor_to_f32(y), ref["y"], name)
    assert B.moe_get_device_status(ws) == B.MOE_OK
