"""Thin ctypes binding of libmoe_gb300.so (include/moe.h).

Argument marshalling only: every function has the C entry point's name and arguments,
accepts torch tensors (device memory) or raw integer addresses for the pointer arguments,
runs on torch's current CUDA stream unless ``stream`` is given, and raises ``MoeError`` for a
non-OK status.  All work happens in the library's CUDA kernels; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

from . import _build

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED_SHAPE = 2
MOE_ERR_WORKSPACE = 3
MOE_ERR_CUDA = 4
MOE_ERR_TIMEOUT = 5
MOE_ERR_DEVICE = 6

MOE_ACT_BF16 = 0
MOE_ACT_MXFP4 = 1
MOE_ACT_MXFP8 = 2

MOE_W_MXFP4 = 0
MOE_W_NVFP4 = 1

# every entry point declared in include/moe.h
EXPORTED = (
    "moe_status_string", "moe_abi_version", "moe_last_cuda_error", "moe_mxfp4_pack", "moe_mxfp4_unpack", "moe_mxfp4_mma_scale_bytes",
    "moe_mxfp4_scales_to_mma", "moe_mxfp4_codes_to_mma", "moe_workspace_size", "moe_padded_rows", "moe_workspace_init",
    "moe_get_device_status", "moe_route", "moe_route_noalloc", "moe_permute", "moe_expert_up_swiglu", "moe_expert_down", "moe_combine",
    "moe_combine_norm", "moe_layer_forward", "moe_layer_forward_host", "moe_layer_forward_norm", "moe_synth_weights", "moe_selftest_wait_timeout",
    "moe_dense_workspace_size", "moe_dense_linear", "moe_nvfp4_pack", "moe_nvfp4_unpack", "moe_workspace_routing",
    "moe_decode_pieces_bytes", "moe_decode_pieces", "moe_expert_ffn_decode",
)


class MoeError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        msg = "%s failed: %s" % (fn, status_string(status))
        if status == MOE_ERR_CUDA:
            msg += " (%s)" % load().moe_last_cuda_error().decode()
        super().__init__(msg)


class moe_expert_weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s", "gate_q_mma", "gate_s_mma",
                 "up_q_mma", "up_s_mma", "down_q_mma", "down_s_mma")] + \
               [("wfmt", ctypes.c_int32)] + [(n, ctypes.c_void_p) for n in ("gate_gs", "up_gs", "down_gs")]


class moe_mxfp4_matrix(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("q", "s", "q_mma", "s_mma")]


_lib = None
P = ctypes.c_void_p
I32, I64, U32, U64 = ctypes.c_int, ctypes.c_int64, ctypes.c_uint32, ctypes.c_uint64
SZ = ctypes.c_size_t
WP = ctypes.POINTER(moe_expert_weights)
MP = ctypes.POINTER(moe_mxfp4_matrix)

_SIGS = {
    "moe_status_string": (ctypes.c_char_p, [I32]),
    "moe_abi_version": (I32, []),
    "moe_last_cuda_error": (ctypes.c_char_p, []),
    "moe_mxfp4_pack": (I32, [P, I64, I64, P, P, P]),
    "moe_mxfp4_unpack": (I32, [P, P, I64, I64, P, P]),
    "moe_mxfp4_mma_scale_bytes": (SZ, [I64, I64]),
    "moe_mxfp4_scales_to_mma": (I32, [P, I64, I64, P, P]),
    "moe_mxfp4_codes_to_mma": (I32, [P, I64, I64, P, P]),
    "moe_workspace_size": (SZ, [I32, I32, I32, I32, I32, I32]),
    "moe_padded_rows": (I64, [I32, I32, I32]),
    "moe_workspace_init": (I32, [P, SZ, P]),
    "moe_get_device_status": (I32, [P, P, ctypes.POINTER(I32)]),
    "moe_route": (I32, [P, P, P, I32, I32, I32, I32, P, P, P, SZ, P]),
    "moe_route_noalloc": (I32, [P, P, P, I32, I32, I32, I32, P, P, P]),
    "moe_permute": (I32, [P, P, I32, I32, I32, I32, I32, P, P, P, P, P, P, P, SZ, P]),
    "moe_expert_up_swiglu": (I32, [P, P, P, I32, P, P, I32, I32, I32, I32, I32, WP, P, P, P, SZ, P]),
    "moe_expert_down": (I32, [P, P, I32, P, P, I32, I32, I32, I32, I32, WP, P, P, SZ, P]),
    "moe_combine": (I32, [P, P, P, I32, I32, I32, P, P]),
    "moe_layer_forward": (I32, [P, P, P, I32, I32, I32, I32, I32, WP, I32, P, P, P, P, SZ, P]),
    "moe_layer_forward_host": (I32, [P, P, P, I32, I32, I32, I32, I32, WP, I32, P, P, P, P, P, P, SZ, P, P, P]),
    "moe_combine_norm": (I32, [P, P, P, I32, I32, I32, ctypes.c_float, P, P]),
    "moe_dense_workspace_size": (SZ, [I32, I32, I32, I32]),
    "moe_dense_linear": (I32, [P, I32, I32, I32, MP, I32, P, P, SZ, P]),
    "moe_layer_forward_norm": (I32, [P, P, P, I32, I32, I32, I32, I32, WP, I32, ctypes.c_float, P, P, P, P, SZ, P]),
    "moe_synth_weights": (I32, [U64, U32, U32, U32, I64, I64, ctypes.c_float, P, P]),
    "moe_selftest_wait_timeout": (I32, [P, SZ, I32, P]),
    "moe_nvfp4_pack": (I32, [P, I64, I64, I64, P, P, P, P]),
    "moe_nvfp4_unpack": (I32, [P, P, P, I64, I64, I64, P, P]),
    "moe_decode_pieces_bytes": (SZ, [I32, I32, I32]),
    "moe_decode_pieces": (I32, [P, I32, I32, I32, P, P, P]),
    "moe_expert_ffn_decode": (I32, [P, P, I32, P, P, P, P, I32, I32, I32, I32, I32, WP, P, P, P, SZ, P]),
    "moe_workspace_routing": (I32, [P, SZ, I32, I32, I32, I32, I32, I32, ctypes.POINTER(P), ctypes.POINTER(P),
                                    ctypes.POINTER(P), ctypes.POINTER(P)]),
}


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load the CUDA library (building it in-tree first if needed).  Raises if unavailable."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if build_if_missing:
        path = _build.build()
    if not os.path.exists(path):
        raise RuntimeError("libmoe_gb300.so is not built (run __graft_entry__.build())")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def _p(t) -> Optional[int]:
    """Pointer argument: a torch tensor (its data pointer), an int address, or None."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn: str, status: int) -> None:
    if status != MOE_OK:
        raise MoeError(fn, status)


def status_string(status: int) -> str:
    return load().moe_status_string(int(status)).decode()


def expert_weights_struct(gate_q, gate_s, up_q, up_s, down_q, down_s, gate_q_mma=None, gate_s_mma=None,
                          up_q_mma=None, up_s_mma=None, down_q_mma=None, down_s_mma=None) -> moe_expert_weights:
    return moe_expert_weights(*[_p(t) for t in (gate_q, gate_s, up_q, up_s, down_q, down_s, gate_q_mma, gate_s_mma,
                                                up_q_mma, up_s_mma, down_q_mma, down_s_mma)])


def nvfp4_expert_weights_struct(gate_q, gate_s, gate_gs, up_q, up_s, up_gs, down_q, down_s,
                                down_gs, gate_q_mma=None, gate_s_mma=None, up_q_mma=None, up_s_mma=None,
                                down_q_mma=None, down_s_mma=None) -> moe_expert_weights:
    """NVFP4 expert weights: codes, E4M3 scales [.][K/16] and per-expert global scales [E], with the
    tensor-core copies (code tiles; the scales laid out as for a matrix of width 2K) when given."""
    W = expert_weights_struct(gate_q, gate_s, up_q, up_s, down_q, down_s, gate_q_mma, gate_s_mma, up_q_mma,
                              up_s_mma, down_q_mma, down_s_mma)
    W.wfmt = MOE_W_NVFP4
    W.gate_gs, W.up_gs, W.down_gs = _p(gate_gs), _p(up_gs), _p(down_gs)
    return W


def mxfp4_matrix_struct(q, s, q_mma=None, s_mma=None) -> moe_mxfp4_matrix:
    return moe_mxfp4_matrix(*[_p(t) for t in (q, s, q_mma, s_mma)])


# ------------------------------------------------------------------ entry points

def moe_abi_version() -> int:
    return load().moe_abi_version()


def moe_mxfp4_pack(w, rows, K, q, s, stream=None):
    _check("moe_mxfp4_pack", load().moe_mxfp4_pack(_p(w), rows, K, _p(q), _p(s), _stream(stream)))


def moe_mxfp4_unpack(q, s, rows, K, w, stream=None):
    _check("moe_mxfp4_unpack", load().moe_mxfp4_unpack(_p(q), _p(s), rows, K, _p(w), _stream(stream)))


def moe_nvfp4_pack(w, n_mats, rows, K, q, s, gs, stream=None):
    _check("moe_nvfp4_pack", load().moe_nvfp4_pack(_p(w), n_mats, rows, K, _p(q), _p(s), _p(gs), _stream(stream)))


def moe_nvfp4_unpack(q, s, gs, n_mats, rows, K, w, stream=None):
    _check("moe_nvfp4_unpack", load().moe_nvfp4_unpack(_p(q), _p(s), _p(gs), n_mats, rows, K, _p(w),
                                                       _stream(stream)))


def moe_mxfp4_mma_scale_bytes(rows, K) -> int:
    return int(load().moe_mxfp4_mma_scale_bytes(rows, K))


def moe_mxfp4_scales_to_mma(s, rows, K, s_mma, stream=None):
    _check("moe_mxfp4_scales_to_mma", load().moe_mxfp4_scales_to_mma(_p(s), rows, K, _p(s_mma), _stream(stream)))


def moe_mxfp4_codes_to_mma(q, rows, K, q_mma, stream=None):
    _check("moe_mxfp4_codes_to_mma", load().moe_mxfp4_codes_to_mma(_p(q), rows, K, _p(q_mma), _stream(stream)))


def moe_workspace_size(T, d, E, k, I, fmt) -> int:
    return int(load().moe_workspace_size(T, d, E, k, I, fmt))


def moe_padded_rows(T, k, E) -> int:
    return int(load().moe_padded_rows(T, k, E))


def moe_workspace_init(ws, ws_bytes=None, stream=None):
    nbytes = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    _check("moe_workspace_init", load().moe_workspace_init(_p(ws), nbytes, _stream(stream)))


def moe_get_device_status(ws, stream=None) -> int:
    out = I32(0)
    _check("moe_get_device_status", load().moe_get_device_status(_p(ws), _stream(stream), ctypes.byref(out)))
    return out.value


def _ws_bytes(ws, ws_bytes):
    if ws is None:
        return 0
    return ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes


def moe_route(x, W_r, b, T, d, E, k, ids, w, ws, ws_bytes=None, stream=None):
    _check("moe_route", load().moe_route(_p(x), _p(W_r), _p(b), T, d, E, k, _p(ids), _p(w), _p(ws),
                                         _ws_bytes(ws, ws_bytes), _stream(stream)))


def moe_decode_pieces_bytes(T, d, scales):
    return load().moe_decode_pieces_bytes(T, d, int(scales))


def moe_decode_pieces(x, T, d, fmt, xa, xa_s, stream=None):
    _check("moe_decode_pieces", load().moe_decode_pieces(_p(x), T, d, fmt, _p(xa), _p(xa_s), _stream(stream)))


def moe_expert_ffn_decode(xa, xa_s, fmt, perm_token, offsets, inv_pos, w, T, d, E, k, I, W: moe_expert_weights, y_perm,
                          y, ws, ws_bytes=None, stream=None):
    _check("moe_expert_ffn_decode",
           load().moe_expert_ffn_decode(_p(xa), _p(xa_s), fmt, _p(perm_token), _p(offsets), _p(inv_pos), _p(w), T, d,
                                        E, k, I, ctypes.byref(W), _p(y_perm), _p(y), _p(ws), _ws_bytes(ws, ws_bytes),
                                        _stream(stream)))


def moe_workspace_routing(ws, T, d, E, k, I, fmt, ws_bytes=None):
    """Device addresses (ints) of counts, offsets, perm_token and inv_pos inside a layer workspace."""
    ptrs = [P() for _ in range(4)]
    _check("moe_workspace_routing",
           load().moe_workspace_routing(_p(ws), _ws_bytes(ws, ws_bytes), T, d, E, k, I, fmt,
                                        *[ctypes.byref(q) for q in ptrs]))
    return tuple(int(q.value) for q in ptrs)


def moe_route_noalloc(x, W_r, b, T, d, E, k, ids, w, stream=None):
    _check("moe_route_noalloc", load().moe_route_noalloc(_p(x), _p(W_r), _p(b), T, d, E, k, _p(ids), _p(w),
                                                         _stream(stream)))


def moe_permute(x, ids, T, d, E, k, fmt, counts, offsets, perm_token, inv_pos, xa, xa_s, ws, ws_bytes=None,
                stream=None):
    _check("moe_permute", load().moe_permute(_p(x), _p(ids), T, d, E, k, fmt, _p(counts), _p(offsets),
                                             _p(perm_token), _p(inv_pos), _p(xa), _p(xa_s), _p(ws),
                                             _ws_bytes(ws, ws_bytes), _stream(stream)))


def moe_expert_up_swiglu(x, xa, xa_s, fmt, perm_token, offsets, T, d, E, k, I, W: moe_expert_weights, h, h_s, ws,
                         ws_bytes=None, stream=None):
    _check("moe_expert_up_swiglu",
           load().moe_expert_up_swiglu(_p(x), _p(xa), _p(xa_s), fmt, _p(perm_token), _p(offsets), T, d, E, k, I,
                                       ctypes.byref(W), _p(h), _p(h_s), _p(ws), _ws_bytes(ws, ws_bytes),
                                       _stream(stream)))


def moe_expert_down(h, h_s, fmt, perm_token, offsets, T, d, E, k, I, W: moe_expert_weights, y_perm, ws,
                    ws_bytes=None, stream=None):
    _check("moe_expert_down",
           load().moe_expert_down(_p(h), _p(h_s), fmt, _p(perm_token), _p(offsets), T, d, E, k, I, ctypes.byref(W),
                                  _p(y_perm), _p(ws), _ws_bytes(ws, ws_bytes), _stream(stream)))


def moe_combine(y_perm, inv_pos, w, T, k, d, y, stream=None):
    _check("moe_combine", load().moe_combine(_p(y_perm), _p(inv_pos), _p(w), T, k, d, _p(y), _stream(stream)))


def moe_layer_forward(x, W_r, b, T, d, E, k, I, W: moe_expert_weights, fmt, y, ids, w, ws, ws_bytes=None,
                      stream=None):
    _check("moe_layer_forward",
           load().moe_layer_forward(_p(x), _p(W_r), _p(b), T, d, E, k, I, ctypes.byref(W), fmt, _p(y), _p(ids),
                                    _p(w), _p(ws), _ws_bytes(ws, ws_bytes), _stream(stream)))


def moe_layer_forward_host(x_host, W_r, b, T, d, E, k, I, W: moe_expert_weights, fmt, y_host, ids, w, x_dev, y_dev,
                           ws, ws_bytes=None, stream=None, in_stream=None, out_stream=None):
    """x_host / y_host: host tensors (pinned for asynchronous copies) or int addresses; x_dev / y_dev:
    the device staging buffers; in_stream / out_stream (optional, both or neither): the streams of
    the copy in and the copy out."""
    ins = None if in_stream is None else _stream(in_stream)
    outs = None if out_stream is None else _stream(out_stream)
    _check("moe_layer_forward_host",
           load().moe_layer_forward_host(_p(x_host), _p(W_r), _p(b), T, d, E, k, I, ctypes.byref(W), fmt, _p(y_host),
                                         _p(ids), _p(w), _p(x_dev), _p(y_dev), _p(ws), _ws_bytes(ws, ws_bytes),
                                         _stream(stream), ins, outs))


def moe_combine_norm(y_perm, inv_pos, w, T, k, d, eps, y, stream=None):
    _check("moe_combine_norm", load().moe_combine_norm(_p(y_perm), _p(inv_pos), _p(w), T, k, d, float(eps), _p(y),
                                                       _stream(stream)))


def moe_layer_forward_norm(x, W_r, b, T, d, E, k, I, W: moe_expert_weights, fmt, eps, y, ids, w, ws, ws_bytes=None,
                           stream=None):
    _check("moe_layer_forward_norm",
           load().moe_layer_forward_norm(_p(x), _p(W_r), _p(b), T, d, E, k, I, ctypes.byref(W), fmt, float(eps), _p(y),
                                         _p(ids), _p(w), _p(ws), _ws_bytes(ws, ws_bytes), _stream(stream)))


def moe_dense_workspace_size(T, K, N, fmt) -> int:
    return int(load().moe_dense_workspace_size(T, K, N, fmt))


def moe_dense_linear(x, T, K, N, W: moe_mxfp4_matrix, fmt, y, ws, ws_bytes=None, stream=None):
    _check("moe_dense_linear", load().moe_dense_linear(_p(x), T, K, N, ctypes.byref(W), fmt, _p(y), _p(ws),
                                                       _ws_bytes(ws, ws_bytes), _stream(stream)))


def moe_synth_weights(seed, tensor_id, expert_first, n_experts, rows, K, c, out, stream=None):
    _check("moe_synth_weights", load().moe_synth_weights(seed, tensor_id, expert_first, n_experts, rows, K,
                                                         float(c), _p(out), _stream(stream)))


def moe_selftest_wait_timeout(ws, limit_us, ws_bytes=None, stream=None):
    n = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    _check("moe_selftest_wait_timeout", load().moe_selftest_wait_timeout(_p(ws), n, int(limit_us), _stream(stream)))
