"""Device-resident MoE layer state: expert weights (MXFP4, generated and packed on the GPU by the
library), router weights, and a workspace.  Convenience for tests and the benchmark; the
compute path is entirely the library's kernels (see binding.py)."""
from __future__ import annotations

from typing import Optional

import numpy as np
import torch

from . import binding as B
from . import inputs as IN


class DeviceLayer:
    """One synthetic layer of workload ``cfg`` on ``device``.  ``layer`` selects an independent
    copy (different weight seed), used to rotate layers so that L2 cannot carry experts.
    ``wfmt``: "mxfp4" (E8M0 scale per 32 values) or "nvfp4" (E4M3 scale per 16 values and a
    global scale per expert matrix; read by the bf16-activation GEMVs and, with its tensor-core
    copies, by the MXFP4-activation grouped GEMMs (kind::mxf4nvf4))."""

    def __init__(self, cfg: IN.Config, device="cuda", layer: int = 0, mma_layouts: bool = True,
                 chunk_bytes: int = 1 << 30, wfmt: str = "mxfp4"):
        assert wfmt in ("mxfp4", "nvfp4")
        self.cfg = cfg
        self.wfmt = wfmt
        nv = wfmt == "nvfp4"
        self.device = torch.device(device)
        self.seed = cfg.seed + 7919 * layer
        E, I, d = cfg.E, cfg.I, cfg.d
        u8 = dict(dtype=torch.uint8, device=self.device)
        self.q = {}
        self.s = {}
        self.gs = {}
        self.s_mma = {}
        shapes = IN.expert_matrix_shapes(cfg)
        c = float(IN.weight_scale(cfg.weight_std))
        for tid, (rows, K) in shapes.items():
            q = torch.empty((E, rows, K // 2), **u8)
            s = torch.empty((E, rows, K // (16 if nv else 32)), **u8)
            gs = torch.empty(E, dtype=torch.float32, device=self.device) if nv else None
            per = rows * K * 4
            n_chunk = max(1, min(E, chunk_bytes // per))
            buf = torch.empty((n_chunk, rows, K), dtype=torch.float32, device=self.device)
            for e0 in range(0, E, n_chunk):
                n = min(n_chunk, E - e0)
                B.moe_synth_weights(self.seed, tid, e0, n, rows, K, c, buf)
                if nv:
                    B.moe_nvfp4_pack(buf, n, rows, K, q[e0:e0 + n], s[e0:e0 + n], gs[e0:e0 + n])
                else:
                    B.moe_mxfp4_pack(buf, n * rows, K, q[e0:e0 + n], s[e0:e0 + n])
            del buf
            self.q[tid], self.s[tid], self.gs[tid] = q, s, gs
        G, U, D = IN.TENSOR_GATE, IN.TENSOR_UP, IN.TENSOR_DOWN
        self.q_mma = {}
        if mma_layouts and d % 256 == 0 and I % 256 == 0:  # copies for the tensor-core paths
            for tid, (rows, K) in shapes.items():
                self.q_mma[tid] = torch.empty(E * rows * K // 2, **u8)
                B.moe_mxfp4_codes_to_mma(self.q[tid], E * rows, K, self.q_mma[tid])
                # NVFP4: 16-element scales [rows][K/16] lay out like the scales of a width-2K matrix
                Ks = 2 * K if nv else K
                self.s_mma[tid] = torch.empty(B.moe_mxfp4_mma_scale_bytes(E * rows, Ks), **u8)
                B.moe_mxfp4_scales_to_mma(self.s[tid], E * rows, Ks, self.s_mma[tid])
        W_r, b = IN.make_router(cfg)
        if layer != 0:  # independent router per layer copy
            rng = np.random.default_rng([cfg.seed, 77, layer])
            W_r = (rng.standard_normal(W_r.shape) / np.sqrt(cfg.d)).astype(np.float32)
        self.W_r_host, self.b_host = W_r, b
        self.W_r = torch.from_numpy(W_r).to(self.device)
        self.b = torch.from_numpy(b).to(self.device)
        if nv:
            self.weights = B.nvfp4_expert_weights_struct(self.q[G], self.s[G], self.gs[G], self.q[U], self.s[U],
                                                         self.gs[U], self.q[D], self.s[D], self.gs[D],
                                                         self.q_mma.get(G), self.s_mma.get(G), self.q_mma.get(U),
                                                         self.s_mma.get(U), self.q_mma.get(D), self.s_mma.get(D))
        else:
            self.weights = B.expert_weights_struct(self.q[G], self.s[G], self.q[U], self.s[U], self.q[D], self.s[D],
                                                   self.q_mma.get(G), self.s_mma.get(G), self.q_mma.get(U),
                                                   self.s_mma.get(U), self.q_mma.get(D), self.s_mma.get(D))

    def weight_bytes_per_expert(self) -> int:
        """Bytes of one expert's three matrices as the expert kernels read them."""
        cfg = self.cfg
        if self.wfmt == "nvfp4":
            return 3 * cfg.I * cfg.d // 2 + 3 * cfg.I * cfg.d // 16 + 3 * 4
        return 3 * cfg.I * cfg.d // 2 + 3 * cfg.I * cfg.d // 32


class DeviceMatrix:
    """One synthetic MXFP4 matrix [rows][K] on ``device`` (the library's generator, matrix 0 of
    ``tensor_id`` under ``seed``), with the tensor-core copies when ``mma``: the shared latent
    projections of a latent layer."""

    def __init__(self, rows: int, K: int, seed: int, tensor_id: int, std: float = 0.02, mma: bool = True,
                 device="cuda"):
        dev = torch.device(device)
        u8 = dict(dtype=torch.uint8, device=dev)
        buf = torch.empty((rows, K), dtype=torch.float32, device=dev)
        B.moe_synth_weights(seed, tensor_id, 0, 1, rows, K, float(IN.weight_scale(std)), buf)
        self.q = torch.empty((rows, K // 2), **u8)
        self.s = torch.empty((rows, K // 32), **u8)
        B.moe_mxfp4_pack(buf, rows, K, self.q, self.s)
        del buf
        self.q_mma = self.s_mma = None
        if mma:
            self.q_mma = torch.empty(rows * K // 2, **u8)
            self.s_mma = torch.empty(B.moe_mxfp4_mma_scale_bytes(rows, K), **u8)
            B.moe_mxfp4_codes_to_mma(self.q, rows, K, self.q_mma)
            B.moe_mxfp4_scales_to_mma(self.s, rows, K, self.s_mma)
        self.rows, self.K = rows, K
        self.struct = B.mxfp4_matrix_struct(self.q, self.s, self.q_mma, self.s_mma)


def make_workspace(T: int, d: int, E: int, k: int, I: int, fmt: int, device="cuda") -> torch.Tensor:
    n = B.moe_workspace_size(T, d, E, k, I, fmt)
    if n == 0:
        raise ValueError("unsupported shape")
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    B.moe_workspace_init(ws)
    return ws


def layer_forward(layer: DeviceLayer, x: torch.Tensor, fmt: int, ws: Optional[torch.Tensor] = None,
                  want_routing: bool = False, stream=None, expert_norm_eps: Optional[float] = None):
    """y = MoE(x) for bf16 x [T][d] (as int16/uint16 bit patterns or torch.bfloat16); with
    expert_norm_eps, each expert output is normalised before the weighted sum."""
    cfg = layer.cfg
    T = x.shape[0]
    if ws is None:
        ws = make_workspace(T, cfg.d, cfg.E, cfg.k, cfg.I, fmt, x.device)
    y = torch.empty((T, cfg.d), dtype=torch.bfloat16, device=x.device)
    ids = torch.empty((T, cfg.k), dtype=torch.int32, device=x.device) if want_routing else None
    w = torch.empty((T, cfg.k), dtype=torch.float32, device=x.device) if want_routing else None
    if expert_norm_eps is None:
        B.moe_layer_forward(x, layer.W_r, layer.b, T, cfg.d, cfg.E, cfg.k, cfg.I, layer.weights, fmt, y, ids, w, ws,
                            stream=stream)
    else:
        B.moe_layer_forward_norm(x, layer.W_r, layer.b, T, cfg.d, cfg.E, cfg.k, cfg.I, layer.weights, fmt,
                                 expert_norm_eps, y, ids, w, ws, stream=stream)
    if want_routing:
        return y, ids, w
    return y
