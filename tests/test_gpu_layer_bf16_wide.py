"""GPU parity of the bf16-activation path with more than four tokens at the full decode widths:
the warp-per-row GEMVs whose lanes own 8 (d = 8192), 4 (d = 4096) or 2 (I = 2048 and 1536)
32-element blocks of a row, for MXFP4 and NVFP4 expert weights, and the tensor-core decode GEMMs
(MXFP4 weights with their tensor-core copies, up to 16 tokens), every token against the oracle
(Muse Spark Open explainer, section 9: gate, up and down per expert, weighted sum; section 11:
4-bit block-scaled weights), with the layer call's permutation bit-exact (section 12)."""
import numpy as np
import pytest
import torch

from bit_expert_ffn_moe_gb300 import binding as B
from bit_expert_ffn_moe_gb300 import inputs as IN
from bit_expert_ffn_moe_gb300.layer import DeviceLayer, layer_forward, make_workspace
from moe_testlib import (bf16_tensor_to_f32, bits_to_device, check_outputs, check_permutation, check_weights,
                         oracle_expert_weights, oracle_expert_weights_nv, workspace_routing)
from oracle import oracle as O

pytestmark = pytest.mark.gpu

WIDE = IN.small_config("wide_8192", T=16, d=8192, E=128, k=8, I=2048, index=71)
MID = IN.small_config("wide_4096", T=8, d=4096, E=64, k=8, I=1536, index=72, zipf_s=1.1)

_layers = {}


def get_layer(cfg, wfmt, mma):
    key = (cfg.name, wfmt, mma)
    if key not in _layers:
        _layers.clear()
        torch.cuda.empty_cache()
        _layers[key] = DeviceLayer(cfg, mma_layouts=mma, wfmt=wfmt)
    return _layers[key]


# (weight format, tensor-core weight copies): MXFP4 on the GEMVs, MXFP4 on the tensor-core decode
# GEMMs (up to 16 tokens), NVFP4 (GEMVs only)
PATHS = [("mxfp4", False), ("mxfp4", True), ("nvfp4", False)]


@pytest.mark.parametrize("cfg,T", [(WIDE, 5), (WIDE, 8), (WIDE, 16), (MID, 8), (MID, 7)])
@pytest.mark.parametrize("wfmt,mma", PATHS)
def test_wide_rows_match_oracle(wfmt, mma, cfg, T):
    layer = get_layer(cfg, wfmt, mma)
    d, E, k, I = cfg.d, cfg.E, cfg.k, cfg.I
    xb = IN.make_x(cfg, call=T)[:T]
    ws = make_workspace(T, d, E, k, I, B.MOE_ACT_BF16)
    y, ids, w = layer_forward(layer, bits_to_device(xb), B.MOE_ACT_BF16, ws=ws, want_routing=True)
    torch.cuda.synchronize()
    assert B.moe_get_device_status(ws) == B.MOE_OK
    weights = oracle_expert_weights_nv(cfg, layer.seed) if wfmt == "nvfp4" else oracle_expert_weights(cfg, layer.seed)
    ref = O.moe_layer(xb, layer.W_r_host, layer.b_host, k, weights, O.ACT_BF16)
    np.testing.assert_array_equal(ids.cpu().numpy(), ref["ids"])
    check_weights(w.cpu().numpy(), ref["w"])
    check_permutation(workspace_routing(ws, T, d, E, k, I, B.MOE_ACT_BF16), ref)
    check_outputs(bf16_tensor_to_f32(y), ref["y"], "%s %s T=%d" % (cfg.name, wfmt, T))
