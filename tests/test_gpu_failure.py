"""Failure detection without a GPU fault: a bounded device wait that runs out reports
MOE_ERR_TIMEOUT through the workspace status word, the read clears it, and the same context then
runs the layer correctly."""
import numpy as np
import pytest
import torch

from bit_expert_ffn_moe_gb300 import binding as B
from bit_expert_ffn_moe_gb300 import inputs as IN
from bit_expert_ffn_moe_gb300.layer import DeviceLayer, layer_forward, make_workspace
from moe_testlib import bf16_tensor_to_f32, bits_to_device, check_outputs, oracle_expert_weights
from oracle import oracle as O

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    cfg = IN.CONFIGS["tiny"]
    ws = make_workspace(cfg.T, cfg.d, cfg.E, cfg.k, cfg.I, B.MOE_ACT_BF16)
    assert B.moe_get_device_status(ws) == B.MOE_OK
    B.moe_selftest_wait_timeout(ws, 2000)  # 2 ms
    assert B.moe_get_device_status(ws) == B.MOE_ERR_TIMEOUT
    assert B.moe_get_device_status(ws) == B.MOE_OK  # the read cleared it
    layer = DeviceLayer(cfg)
    xb = IN.make_x(cfg, call=5)
    y = layer_forward(layer, bits_to_device(xb), B.MOE_ACT_BF16, ws=ws)
    torch.cuda.synchronize()
    assert B.moe_get_device_status(ws) == B.MOE_OK
    ref = O.moe_layer(xb, layer.W_r_host, layer.b_host, cfg.k, oracle_expert_weights(cfg, layer.seed), O.ACT_BF16)
    check_outputs(bf16_tensor_to_f32(y), ref["y"], "after timeout")
