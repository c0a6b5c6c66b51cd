"""Shared helpers of the parity tests: the oracle's side of a workload (expert weights generated
on the host from the same counters and packed by the oracle's own packer), tolerance checks."""
from __future__ import annotations

import functools

import numpy as np

from bit_expert_ffn_moe_gb300 import inputs as IN
from oracle import oracle as O

# Output tolerance (stated for the layer): relative Frobenius error <= 5e-3 and max abs error
# <= 3e-2 x RMS of the oracle output, over the checked tokens.
REL_FRO = 5e-3
MAX_ABS_RMS = 3e-2
W_ABS = 2e-6     # gate weights
W_SUM = 1e-6     # |sum_j w - 1|


@functools.lru_cache(maxsize=512)
def oracle_matrix(seed: int, tensor_id: int, expert: int, rows: int, K: int, std: float):
    w = IN.synth_weights(seed, tensor_id, expert, rows, K, std)
    return O.mxfp4_pack(w)


def oracle_expert_weights(cfg: IN.Config, seed: int):
    shapes = IN.expert_matrix_shapes(cfg)

    def get(e):
        out = {}
        for name, tid in (("gate", IN.TENSOR_GATE), ("up", IN.TENSOR_UP), ("down", IN.TENSOR_DOWN)):
            rows, K = shapes[tid]
            out[name] = oracle_matrix(seed, tid, e, rows, K, cfg.weight_std)
        return out
    return get


@functools.lru_cache(maxsize=512)
def oracle_matrix_nv(seed: int, tensor_id: int, expert: int, rows: int, K: int, std: float):
    """One expert matrix packed by the oracle's NVFP4 packer: (q, s, global scale)."""
    w = IN.synth_weights(seed, tensor_id, expert, rows, K, std)
    return O.nvfp4_pack(w)


def oracle_expert_weights_nv(cfg: IN.Config, seed: int):
    shapes = IN.expert_matrix_shapes(cfg)

    def get(e):
        out = {}
        for name, tid in (("gate", IN.TENSOR_GATE), ("up", IN.TENSOR_UP), ("down", IN.TENSOR_DOWN)):
            rows, K = shapes[tid]
            out[name] = oracle_matrix_nv(seed, tid, e, rows, K, cfg.weight_std)
        return out
    return get


def check_outputs(y_gpu: np.ndarray, y_ref: np.ndarray, what: str = "y"):
    y_gpu = np.asarray(y_gpu, dtype=np.float64)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    assert np.all(np.isfinite(y_gpu)), what + ": non-finite output"
    ref_norm = np.linalg.norm(y_ref)
    assert ref_norm > 0, what + ": oracle output is all zero"
    rel = np.linalg.norm(y_gpu - y_ref) / ref_norm
    rms = np.sqrt(np.mean(y_ref ** 2))
    mx = np.max(np.abs(y_gpu - y_ref))
    assert rel <= REL_FRO, "%s: relative Frobenius error %.3g > %.3g" % (what, rel, REL_FRO)
    assert mx <= MAX_ABS_RMS * rms, "%s: max abs error %.3g > %.3g x RMS %.3g" % (what, mx, MAX_ABS_RMS, rms)
    return rel, mx / rms


def check_weights(w_gpu, w_ref):
    w_gpu = np.asarray(w_gpu, dtype=np.float64)
    assert np.max(np.abs(w_gpu - w_ref)) <= W_ABS
    assert np.max(np.abs(w_gpu.sum(axis=-1) - 1.0)) <= W_SUM


def bf16_tensor_to_f32(t) -> np.ndarray:
    import torch
    return t.detach().to(torch.float32).cpu().numpy()


def bits_to_device(bits: np.ndarray, device="cuda"):
    import torch
    return torch.from_numpy(bits.view(np.int16).copy()).to(device).view(torch.bfloat16)


def workspace_routing(ws, T, d, E, k, I, fmt):
    """counts, offsets, perm_token, inv_pos as the last layer call left them in its workspace."""
    import torch

    from bit_expert_ffn_moe_gb300 import binding as B
    torch.cuda.synchronize()
    ptrs = B.moe_workspace_routing(ws, T, d, E, k, I, fmt)
    base = ws.data_ptr()
    out = []
    for p, n in zip(ptrs, (E, E + 1, T * k, T * k)):
        off = p - base
        assert 0 <= off and off % 4 == 0 and off + 4 * n <= ws.numel()
        out.append(ws[off:off + 4 * n].view(torch.int32).cpu().numpy().copy())
    return out


def check_permutation(routing, ref):
    """Bit-exact counts, offsets, perm_token and inv_pos against the oracle's permutation."""
    counts, offsets, perm, inv = routing
    np.testing.assert_array_equal(counts, ref["counts"])
    np.testing.assert_array_equal(offsets, ref["offsets"])
    np.testing.assert_array_equal(perm, ref["perm_token"])
    np.testing.assert_array_equal(inv, ref["inv_pos"])
