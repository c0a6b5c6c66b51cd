"""GPU: the host-buffer layer call (moe_layer_forward_host) copies x in, runs the same layer and copies
y out -- its y, ids and w equal moe_layer_forward's bit for bit (decode on the tensor cores, the
MXFP4-activation prefill path), and y against the oracle; with copy streams and two alternating
staging pairs, consecutive calls on different inputs give each call's own result."""
import numpy as np
import pytest
import torch

from bit_expert_ffn_moe_gb300 import binding as B
from bit_expert_ffn_moe_gb300 import inputs as IN
from bit_expert_ffn_moe_gb300.layer import DeviceLayer, layer_forward, make_workspace
from moe_testlib import bf16_tensor_to_f32, bits_to_device, check_outputs, oracle_expert_weights
from oracle import oracle as O

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,fmt,ofmt", [("tiny", B.MOE_ACT_BF16, O.ACT_BF16),
                                           ("decode", B.MOE_ACT_BF16, O.ACT_BF16),
                                           ("mx300", B.MOE_ACT_MXFP4, O.ACT_MXFP4)])
def test_host_buffer_layer_equals_device_layer(name, fmt, ofmt):
    cfg = (IN.small_config("mx300", T=300, d=512, E=12, k=3, I=512, index=97) if name == "mx300"
           else IN.CONFIGS[name])
    layer = DeviceLayer(cfg)
    T, d = cfg.T, cfg.d
    ws = make_workspace(T, d, cfg.E, cfg.k, cfg.I, fmt)
    xb = IN.make_x(cfg, call=1)
    y_ref, ids_ref, w_ref = layer_forward(layer, bits_to_device(xb), fmt, ws=ws, want_routing=True)

    x_host = torch.from_numpy(xb.view(np.int16).copy()).view(torch.bfloat16).pin_memory()
    y_host = torch.zeros((T, d), dtype=torch.bfloat16).pin_memory()
    x_dev = torch.empty((T, d), dtype=torch.bfloat16, device="cuda")
    y_dev = torch.empty((T, d), dtype=torch.bfloat16, device="cuda")
    ids = torch.empty((T, cfg.k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, cfg.k), dtype=torch.float32, device="cuda")
    B.moe_layer_forward_host(x_host, layer.W_r, layer.b, T, d, cfg.E, cfg.k, cfg.I, layer.weights, fmt, y_host, ids,
                             w, x_dev, y_dev, ws)
    torch.cuda.synchronize()
    assert torch.equal(y_host.view(torch.int16), y_ref.cpu().view(torch.int16))
    assert torch.equal(ids.cpu(), ids_ref.cpu())
    assert torch.equal(w.cpu(), w_ref.cpu())
    tokens = np.arange(min(T, 16))
    y_o = O.moe_layer(xb, layer.W_r_host, layer.b_host, cfg.k, oracle_expert_weights(cfg, layer.seed), ofmt,
                      tokens=tokens)
    check_outputs(bf16_tensor_to_f32(y_host[tokens]), y_o["y"])


@pytest.mark.parametrize("name,fmt", [("decode", B.MOE_ACT_BF16), ("tiny", B.MOE_ACT_BF16),
                                      ("mx300", B.MOE_ACT_MXFP4)])
def test_host_buffer_layer_with_copy_streams(name, fmt):
    cfg = (IN.small_config("mx300", T=300, d=512, E=12, k=3, I=512, index=97) if name == "mx300"
           else IN.CONFIGS[name])
    layer = DeviceLayer(cfg)
    T, d = cfg.T, cfg.d
    ws = make_workspace(T, d, cfg.E, cfg.k, cfg.I, fmt)
    calls = 5
    xbs = [IN.make_x(cfg, call=c) for c in range(calls)]
    refs = [layer_forward(layer, bits_to_device(xb), fmt, ws=ws).cpu() for xb in xbs]
    x_host = [torch.from_numpy(xb.view(np.int16).copy()).view(torch.bfloat16).pin_memory() for xb in xbs]
    y_host = [torch.zeros((T, d), dtype=torch.bfloat16).pin_memory() for _ in range(calls)]
    x_dev = [torch.empty((T, d), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    y_dev = [torch.empty((T, d), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    st, ins, outs = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    for c in range(calls):
        B.moe_layer_forward_host(x_host[c], layer.W_r, layer.b, T, d, cfg.E, cfg.k, cfg.I, layer.weights,
                                 fmt, y_host[c], None, None, x_dev[c % 2], y_dev[c % 2], ws, stream=st,
                                 in_stream=ins, out_stream=outs)
    outs.synchronize()
    st.synchronize()
    for c in range(calls):
        assert torch.equal(y_host[c].view(torch.int16), refs[c].view(torch.int16)), "call %d" % c


def test_host_buffer_staging_table_beyond_its_capacity():
    """More staging buffers than the event table holds (64): the x buffers alternate between two
    addresses while every call takes a fresh y buffer, so old entries are released while the x
    buffers stay in use; every call still gets its own result."""
    cfg = IN.CONFIGS["tiny"]
    layer = DeviceLayer(cfg)
    T, d = cfg.T, cfg.d
    ws = make_workspace(T, d, cfg.E, cfg.k, cfg.I, B.MOE_ACT_BF16)
    calls = 80
    xbs = [IN.make_x(cfg, call=c % 7) for c in range(calls)]
    refs = {c: layer_forward(layer, bits_to_device(xbs[c]), B.MOE_ACT_BF16, ws=ws).cpu() for c in range(7)}
    x_host = [torch.from_numpy(xb.view(np.int16).copy()).view(torch.bfloat16).pin_memory() for xb in xbs]
    y_host = [torch.zeros((T, d), dtype=torch.bfloat16).pin_memory() for _ in range(calls)]
    x_dev = [torch.empty((T, d), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    y_dev = [torch.empty((T, d), dtype=torch.bfloat16, device="cuda") for _ in range(calls)]  # all distinct
    st, ins, outs = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    for c in range(calls):
        B.moe_layer_forward_host(x_host[c], layer.W_r, layer.b, T, d, cfg.E, cfg.k, cfg.I, layer.weights,
                                 B.MOE_ACT_BF16, y_host[c], None, None, x_dev[c % 2], y_dev[c], ws, stream=st,
                                 in_stream=ins, out_stream=outs)
    torch.cuda.synchronize()
    for c in range(calls):
        assert torch.equal(y_host[c].view(torch.int16), refs[c % 7].view(torch.int16)), "call %d" % c


def test_host_buffer_staging_roles_swap():
    """Two device buffers that swap roles on every call (x of one call is y of the next): the copy
    into a buffer waits for the copy out of it, and the layer's write into it for every reader."""
    cfg = IN.CONFIGS["decode"]
    layer = DeviceLayer(cfg)
    T, d = cfg.T, cfg.d
    ws = make_workspace(T, d, cfg.E, cfg.k, cfg.I, B.MOE_ACT_BF16)
    calls = 12
    xbs = [IN.make_x(cfg, call=c) for c in range(calls)]
    refs = [layer_forward(layer, bits_to_device(xb), B.MOE_ACT_BF16, ws=ws).cpu() for xb in xbs]
    x_host = [torch.from_numpy(xb.view(np.int16).copy()).view(torch.bfloat16).pin_memory() for xb in xbs]
    y_host = [torch.zeros((T, d), dtype=torch.bfloat16).pin_memory() for _ in range(calls)]
    bufs = [torch.empty((T, d), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    st, ins, outs = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    for c in range(calls):
        B.moe_layer_forward_host(x_host[c], layer.W_r, layer.b, T, d, cfg.E, cfg.k, cfg.I, layer.weights,
                                 B.MOE_ACT_BF16, y_host[c], None, None, bufs[c % 2], bufs[(c + 1) % 2], ws,
                                 stream=st, in_stream=ins, out_stream=outs)
    torch.cuda.synchronize()
    for c in range(calls):
        assert torch.equal(y_host[c].view(torch.int16), refs[c].view(torch.int16)), "call %d" % c
