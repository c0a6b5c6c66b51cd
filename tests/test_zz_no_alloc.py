"""moe_route_noalloc: the router entry point for callers that cannot allocate device memory or
keep a workspace (for instance code running inside a global-mode CUDA graph capture, or a host
whose fixed memory pool refuses further allocations).  Its scratch is a fixed array inside the
library, so its results must equal the oracle's and moe_route's (which uses a caller workspace)
call after call, and sizes beyond that array must be refused.  Collected last on purpose."""
import numpy as np
import pytest
import torch

from bit_expert_ffn_moe_gb300 import binding as B
from bit_expert_ffn_moe_gb300 import inputs as IN
from bit_expert_ffn_moe_gb300.layer import make_workspace
from moe_testlib import bits_to_device, check_weights
from oracle import oracle as O

pytestmark = pytest.mark.gpu

# two calls in a row of different sizes and inputs; the decode shapes take the one-launch router in
# moe_route and the tiled router in moe_route_noalloc
SHAPES = [IN.small_config("noalloc_a", T=1000, d=1024, E=96, k=6, I=128, index=81, zipf_s=1.2),
          IN.small_config("noalloc_b", T=4096, d=512, E=128, k=8, I=128, index=82),
          IN.small_config("noalloc_decode", T=1, d=8192, E=128, k=8, I=128, index=83),
          IN.small_config("noalloc_verify", T=4, d=8192, E=128, k=8, I=128, index=84)]


def route_both(cfg, call):
    xb = IN.make_x(cfg, call=call)
    W_r, b = IN.make_router(cfg)
    T, d, E, k = cfg.T, cfg.d, cfg.E, cfg.k
    x, Wd, bd = bits_to_device(xb), torch.from_numpy(W_r).cuda(), torch.from_numpy(b).cuda()
    i32 = dict(dtype=torch.int32, device="cuda")
    ids0, w0 = torch.empty((T, k), **i32), torch.empty((T, k), dtype=torch.float32, device="cuda")
    ids1, w1 = torch.full((T, k), -1, **i32), torch.full((T, k), -1.0, dtype=torch.float32, device="cuda")
    ws = make_workspace(T, d, E, k, 128, B.MOE_ACT_BF16)
    B.moe_route(x, Wd, bd, T, d, E, k, ids0, w0, ws)
    B.moe_route_noalloc(x, Wd, bd, T, d, E, k, ids1, w1)
    torch.cuda.synchronize()
    ids_o, w_o = O.topk_softmax(O.router_logits(xb, W_r, b), k)
    return ids0.cpu().numpy(), w0.cpu().numpy(), ids1.cpu().numpy(), w1.cpu().numpy(), ids_o, w_o


@pytest.mark.parametrize("repeat", [0, 1])
def test_noalloc_route_equals_oracle_and_workspace_route_on_consecutive_calls(repeat):
    for call, cfg in enumerate(SHAPES):
        ids0, w0, ids1, w1, ids_o, w_o = route_both(cfg, call + 10 * repeat)
        np.testing.assert_array_equal(ids1, ids_o)
        np.testing.assert_array_equal(ids0, ids_o)
        check_weights(w1, w_o)
        check_weights(w1, w0.astype(np.float64))


def test_noalloc_route_rejects_sizes_beyond_its_scratch():
    T, d, E, k = 4097, 128, 128, 2   # T * E = 524416 > 524288
    x = torch.zeros((T, d), dtype=torch.bfloat16, device="cuda")
    W_r = torch.zeros((E, d), dtype=torch.float32, device="cuda")
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    with pytest.raises(B.MoeError) as e:
        B.moe_route_noalloc(x, W_r, None, T, d, E, k, ids, w)
    assert e.value.status == B.MOE_ERR_UNSUPPORTED_SHAPE
    with pytest.raises(B.MoeError) as e:   # the shape rules of moe_route hold too (d % 128)
        B.moe_route_noalloc(x[:, :96].contiguous(), W_r[:, :96].contiguous(), None, 8, 96, E, k, ids, w)
    assert e.value.status == B.MOE_ERR_UNSUPPORTED_SHAPE
