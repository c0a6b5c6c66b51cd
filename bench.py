#!/usr/bin/env python3
"""Benchmark of the MoE expert-FFN layer on GB300.

Default workload (N=1): decode, batch 1 -- T=1 token per layer call, d=8192, E=128, top-8,
I=2048, MXFP4 expert weights, bf16 activations; one step = one whole layer call (route ->
permute -> gate/up+SwiGLU -> down -> weighted sum) on the next of 1000 seeded tokens; four
independent layer copies (13.7 GB of expert weights) are rotated so that L2 cannot carry experts
from one step to the next.

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle instead (bounded
sample, host cores).  Under torchrun each rank runs its own replica (weak scaling, no data-path
collective); the step time is the maximum over ranks.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/sec on 1 GB300 + % of roofline (HBM BW decode, FP4 peak prefill)"
UNIT = "tokens/s"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
NOMINAL_FP4_OVER_BF16 = 13.5 / 2.25  # dense FP4 : dense bf16 nominal ratio on GB300 (6x)
NOMINAL_FP8_OVER_BF16 = 4.5 / 2.25   # dense FP8 (kind::mxf8f6f4) : dense bf16 (2x)
ACT_FMTS = {"bf16": 0, "mxfp4": 1, "mxfp8": 2}  # moe_act_fmt values


def grouped_gemm_path(fmt: int, T: int) -> bool:
    """Whether the layer runs the tensor-bound grouped prefill GEMMs (MXFP4 always; MXFP8 beyond 16
    tokens, below which it runs the decode kernels)."""
    return fmt == 1 or (fmt == 2 and T > 16)


def tensor_peak_ratio(fmt: int) -> float:
    return NOMINAL_FP8_OVER_BF16 if fmt == 2 else NOMINAL_FP4_OVER_BF16
N_LAYER_COPIES = 4


# ------------------------------------------------------------------ byte / flop model
# Per-expert sizes as the Muse Spark Open explainer models them (sections 10-13): an expert is
# three matrices; reading it costs its packed bytes, computing one token costs 2 flops per
# weight.  MXFP4 stores 4 bits per weight plus one byte per 32 weights (4.25 bits); NVFP4 one byte
# per 16 weights (4.5 bits, the explainer's section 11 figure) plus a 4-byte global scale per matrix.

WEIGHT_BITS = {"mxfp4": 4.25, "nvfp4": 4.5}
GLOBAL_SCALE_BYTES = {"mxfp4": 0, "nvfp4": 4}

def matrix_bytes(rows: int, K: int, bits_per_weight: float = 4.25) -> float:
    return rows * K * bits_per_weight / 8.0


def expert_bytes(d: int, I: int, bits_per_weight: float = 4.25) -> float:
    return 3 * matrix_bytes(I, d, bits_per_weight)


def up_bytes_per_expert(d: int, I: int, wfmt: str = "mxfp4") -> float:
    return 2 * (matrix_bytes(I, d, WEIGHT_BITS[wfmt]) + GLOBAL_SCALE_BYTES[wfmt])


def expert_read_bytes(d: int, I: int, wfmt: str = "mxfp4") -> float:
    return 3 * (matrix_bytes(I, d, WEIGHT_BITS[wfmt]) + GLOBAL_SCALE_BYTES[wfmt])


def down_bytes_per_expert(d: int, I: int) -> float:
    return matrix_bytes(d, I)


def flops_per_token_expert(d: int, I: int) -> float:
    return 2.0 * 3 * d * I


def read_time_us(nbytes: float, bw_bytes_per_s: float) -> float:
    return nbytes / bw_bytes_per_s * 1e6


def crossover_tokens(read_us: float, compute_us_per_token: float) -> float:
    return read_us / compute_us_per_token


def layer_algorithmic_bytes(d: int, I: int, E: int, T: int, n_active: float, wfmt: str = "mxfp4") -> float:
    """Touched experts + router weights and bias + x in + y out."""
    return n_active * expert_read_bytes(d, I, wfmt) + E * d * 4 + E * 4 + 2 * T * d * 2


# ------------------------------------------------------------------ environment helpers

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        hbm = p.get("hbm_gbs") or p.get("hbm_GBps") or p.get("hbm")
        bf16 = p.get("bf16_tflops")
        bf16s = p.get("bf16_tflops_sustained", bf16)
        if hbm:
            return dict(hbm_gbs=float(hbm), bf16_tflops=float(bf16 or FALLBACK_BF16_TFLOPS),
                        bf16_tflops_sustained=float(bf16s or FALLBACK_BF16_TFLOPS), source="measured")
    return dict(hbm_gbs=FALLBACK_HBM_GBS, bf16_tflops=FALLBACK_BF16_TFLOPS, bf16_tflops_sustained=1700.0,
                source="fallback")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms during the timed region."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.QUERY,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.path or not os.path.exists(self.path):
            return None
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# the sources each profiled kernel is compiled from (a summary's counters hold while their hash matches)
DECODE_KERNEL_SOURCES = ["bit_expert_ffn_moe_gb300/csrc/decode_mma.cu", "bit_expert_ffn_moe_gb300/csrc/tcgen05.cuh",
                         "bit_expert_ffn_moe_gb300/csrc/common.cuh", "bit_expert_ffn_moe_gb300/csrc/route_common.cuh"]
GROUPED_KERNEL_SOURCES = ["bit_expert_ffn_moe_gb300/csrc/umma.cu", "bit_expert_ffn_moe_gb300/csrc/tcgen05.cuh",
                          "bit_expert_ffn_moe_gb300/csrc/common.cuh"]


def source_hash(paths):
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_workload(args, cfg, tag=""):
    """The workload name an ncu summary must carry for its counters to stand for the timed launch:
    the summaries are captured on the plain layer, so a launch at the latent width (--latent) or in
    another mode (tag, e.g. the decode kernel on MXFP8 activations) matches none of them."""
    name = cfg.name + tag
    if getattr(args, "latent", 0):
        name += "+latent%d" % args.latent
    return name


def ncu_traffic(profile_name: str, kernel_sources, workload: str):
    """dram bytes per launch recorded in profiles/<profile_name> for the kernel, or None when
    the summary is missing, was captured on another workload, or the kernel's sources changed
    since the capture."""
    path = os.path.join(ROOT, "profiles", profile_name)
    if not os.path.exists(path):
        return None
    vals = {}
    with open(path) as f:
        for line in f:
            if ":" in line and line.strip().startswith(("source_hash", "dram_bytes_per_launch", "workload")):
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip().strip("`")
    if vals.get("source_hash") != source_hash(kernel_sources) or vals.get("workload") != workload:
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ------------------------------------------------------------------ distributed plumbing

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_dist(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist


def max_over_ranks(value: float, world: int, device) -> float:
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ GPU arm

def run_gpu(args, cfg, rank, world, local):
    import numpy as np
    import torch

    from bit_expert_ffn_moe_gb300 import binding as B
    from bit_expert_ffn_moe_gb300 import inputs as IN
    from bit_expert_ffn_moe_gb300.layer import DeviceLayer, make_workspace

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist(world, "nccl")
    B.load(build_if_missing=False)
    fmt = ACT_FMTS[args.fmt]
    T, d, E, k, I = cfg.T, cfg.d, cfg.E, cfg.k, cfg.I  # d: the model width of x and y
    cm = moe_cfg(args, cfg)  # the layer's configuration (its width dl = cm.d)
    dl = cm.d
    n_calls = max(cfg.calls, 1)

    # tensor-core weight copies: every MXFP4 path; NVFP4 weights use theirs with MXFP4 activations
    layers = [DeviceLayer(cm, device=dev, layer=i + 1000 * rank,
                          mma_layouts=(args.weights == "mxfp4" or args.fmt == "mxfp4"), wfmt=args.weights)
              for i in range(args.layers)]
    lat = Latent(cfg, dl, fmt, dev, layers) if args.latent else None
    # all seeded inputs resident in HBM before timing
    xs_host = np.stack([IN.make_x(cfg, call=(c + rank * 100000) % (1 << 20)) for c in range(min(n_calls, 1000))])
    xs = torch.from_numpy(xs_host.view(np.int16).copy()).to(dev).view(torch.bfloat16)
    n_x = xs.shape[0]
    ws = make_workspace(T, dl, E, k, I, fmt, dev)
    y = torch.empty((T, d), dtype=torch.bfloat16, device=dev)
    ids = torch.empty((args.steps, T, k), dtype=torch.int32, device=dev)
    wts = torch.empty((args.steps, T, k), dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def call(s, x, y_out, ids_s, w_s, ws_l, st):
        """One step: the layer, or narrow -> layer at the latent width -> widen."""
        L = layers[s % len(layers)]
        if lat is None:
            layer_call(B, args, x, L, T, d, E, k, I, fmt, y_out, ids_s, w_s, ws_l, st)
            return
        lat.narrow(s, x, lat.xl, st)
        layer_call(B, args, lat.xl, L, T, dl, E, k, I, fmt, lat.yl, ids_s, w_s, ws_l, st)
        lat.widen(s, lat.yl, y_out, st)

    def step(s, st, record_routing=True):
        call(s, xs[s % n_x], y, ids[s] if record_routing else None, wts[s] if record_routing else None, ws,
             st.cuda_stream)

    # warm-up (eager), then capture the K timed steps in one CUDA graph
    with torch.cuda.stream(stream):
        for s in range(args.warmup):
            step(s % args.steps, stream)
    stream.synchronize()
    graph = None
    if not args.no_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for s in range(args.steps):
                step(s, stream)
        with torch.cuda.stream(stream):
            graph.replay()  # one untimed replay
        stream.synchronize()

    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        t_wall0 = time.perf_counter()
        with torch.cuda.stream(stream):  # the graph replays on the current stream
            start.record(stream)
            if graph is not None:
                graph.replay()
            else:
                for s in range(args.steps):
                    step(s, stream)
            end.record(stream)
        end.synchronize()
        t_wall = time.perf_counter() - t_wall0
    torch.cuda.synchronize(dev)
    barrier(world)
    ms_total = start.elapsed_time(end)
    ms_total = max_over_ranks(ms_total, world, dev)
    status = B.moe_get_device_status(ws, stream=stream.cuda_stream)
    if status == B.MOE_OK and lat is not None:
        status = lat.status(stream.cuda_stream)
    if status != B.MOE_OK:
        raise RuntimeError("device status after timed region: %s" % B.status_string(status))
    yf = y.float()
    if not torch.isfinite(yf).all() or torch.count_nonzero(yf) == 0:
        raise RuntimeError("refusing to record: output is non-finite or all zero")
    ids_h = ids.cpu().numpy()
    counts_ok = all(np.bincount(ids_h[s].reshape(-1), minlength=E).sum() == T * k for s in range(args.steps))
    if not counts_ok:
        raise RuntimeError("refusing to record: routing counts do not sum to T*k")
    n_active = [len(np.unique(ids_h[s])) for s in range(args.steps)]

    tokens = T * args.steps * world
    value = tokens / (ms_total / 1e3)
    ms_per_step = ms_total / args.steps
    pk = peaks()
    bw = pk["hbm_gbs"] * 1e9
    mean_active = float(np.mean(n_active))
    layer_bytes = layer_algorithmic_bytes(dl, I, E, T, mean_active, args.weights)
    if lat is not None:  # + the projections, x and y at the model width instead of dl
        layer_bytes += lat.bytes_per_step() + 2 * T * (d - dl) * 2

    # ---- dominant kernel, timed alone with events on its own stream (same inputs, same layers)
    xs_k = xs
    if lat is not None:  # the gate/up kernel's inputs are the narrowed rows
        xs_k = torch.empty((n_x, T, dl), dtype=torch.bfloat16, device=dev)
        with torch.cuda.stream(stream):
            for i in range(n_x):
                lat.narrow(0, xs[i], xs_k[i], stream.cuda_stream)
        stream.synchronize()
    roof = kernel_roofline(args, cm, layers, xs_k, fmt, dev, stream, pk)

    # ---- end to end through the C ABI with host buffers
    host_call = None
    if lat is None and norm_eps(args) is None:
        fn = B.load().moe_layer_forward_host
        # per layer copy: its router pointers and weight struct, marshalled once (the loop then only
        # passes integers to the C entry point)
        lay_args = [(L.W_r.data_ptr(), None if L.b is None else L.b.data_ptr(), ctypes.byref(L.weights))
                    for L in layers]

        def host_call(s, x_host, y_host, x_dev, y_dev, ws_l, st, cst):
            wr, bb, wp = lay_args[s % len(lay_args)]
            status = fn(x_host, wr, bb, T, d, E, k, I, wp, fmt, y_host, None, None, x_dev, y_dev, ws_l[0], ws_l[1],
                        st, cst[0], cst[1])
            if status != B.MOE_OK:
                raise B.MoeError("moe_layer_forward_host", status)
    e2e = end_to_end(args, cfg, cm, xs_host, fmt, dev, stream, call, host_call)

    # ---- the oracle sample's rows through the same layer copy (checked in main)
    parity_y = parity_ids = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        parity_y, parity_ids = [], []
        ids_p = torch.empty((T, k), dtype=torch.int32, device=dev)
        w_p = torch.empty((T, k), dtype=torch.float32, device=dev)
        with torch.cuda.stream(stream):
            for xb, rows in parity_inputs(cfg, args.cpu_sample_tokens):
                x = torch.from_numpy(xb.view(np.int16).copy()).to(dev).view(torch.bfloat16)
                call(sample_layer_index(args), x, y, ids_p, w_p, ws, stream.cuda_stream)
                yh = y.float().cpu().numpy()
                parity_y.append(yh if rows is None else yh[rows])
                parity_ids.append(ids_p.cpu().numpy().copy())

    out = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": dtype_name(fmt, args.weights), "data": "synthetic",
        "config": {"workload": workload_name(args, cfg),
                   "T": T, "d": d, "E": E, "k": k, "I": I, "act": args.fmt, "weights": args.weights,
                   "expert_norm_eps": norm_eps(args),
                   "latent_width": dl if lat is not None else None,
                   "layer_copies_rotated": len(layers),
                   "l2": "inputs larger than L2: %d layer copies, %.1f GB of expert weights rotated"
                         % (len(layers), len(layers) * E * expert_read_bytes(dl, I, args.weights) / 1e9),
                   "cuda_graph": graph is not None, "parallelism": "replicas" if world > 1 else "single GPU"},
        "layer_roofline": layer_roofline(fmt, cm, layer_bytes, ms_per_step, bw, pk, mean_active, world,
                                         lat.flops_per_step() if lat is not None else 0.0),
        "roofline": roof,
        "e2e": e2e,
        "gpu_launches": launches_per_step(fmt, T, d, E, k, norm_eps(args) is not None, lat is not None,
                                          fmt != B.MOE_ACT_MXFP4 and args.weights == "mxfp4"
                                          and B.moe_decode_pieces_bytes(T, dl, 0) > 0 and I % 256 == 0,
                                          fmt == B.MOE_ACT_MXFP4 and args.weights == "nvfp4") * args.steps,
        "clocks": clk.summary(),
        "wall_s_timed": round(t_wall, 4),
        "_parity_y": parity_y,
        "_parity_ids": parity_ids,
    }
    return out


def layer_roofline(fmt, cfg, layer_bytes, ms_per_step, bw, pk, mean_active, world, extra_flops=0.0):
    """Whole-layer fraction of the roofline the workload is quoted against: HBM bytes for the
    decode path; for the prefill path the FP4 (MXFP8 activations: FP8) tensor peak (useful flops
    6 P d I per step, plus extra_flops of the latent projections), with the HBM fraction beside it."""
    out = {"bound": "hbm", "algorithmic_bytes_per_step": layer_bytes,
           "achieved_GBps": round(layer_bytes / (ms_per_step / 1e3) / 1e9, 1),
           "peak_GBps": pk["hbm_gbs"], "frac": round(layer_bytes / (ms_per_step / 1e3) / bw, 4),
           "peak_source": pk["source"], "mean_active_experts": round(mean_active, 2)}
    if grouped_gemm_path(fmt, cfg.T):
        ratio = tensor_peak_ratio(fmt)
        flops = (6.0 * cfg.T * cfg.k * cfg.d * cfg.I + extra_flops) * world
        peak_tf = pk["bf16_tflops"] * ratio * world
        peak_sus = pk["bf16_tflops_sustained"] * ratio * world
        achieved = flops / (ms_per_step / 1e3) / 1e12
        # the read-vs-compute roofline of the step: whichever of the weight read and the FP4 math
        # takes longer bounds it
        t_bytes = layer_bytes * world / bw
        t_flops = flops / (peak_tf * 1e12)
        t_roof = max(t_bytes, t_flops)
        out = {"bound": "tensor", "algorithmic_flops_per_step": flops, "achieved_TFLOPs": round(achieved, 1),
               "peak_TFLOPs": round(peak_tf, 1), "frac": round(achieved / peak_tf, 4),
               "peak_source": pk["source"] + " bf16 burst x %.0f (nominal %s : bf16 dense ratio)"
                              % (ratio, "FP8" if fmt == 2 else "FP4"),
               "frac_of_sustained_peak": round(achieved / peak_sus, 4), "sustained_peak_TFLOPs": round(peak_sus, 1),
               "max_roofline": {"t_bytes_us": round(t_bytes * 1e6, 2), "t_flops_us": round(t_flops * 1e6, 2),
                                "bound": "hbm" if t_bytes >= t_flops else "tensor",
                                "frac": round(t_roof / (ms_per_step / 1e3), 4)},
               "hbm": out}
    return out


def dtype_name(fmt, wfmt="mxfp4"):
    if fmt == 0:
        return "%s weights x bf16 activations, fp32 accumulate" % wfmt
    return "mxfp4 x mxfp8 (E4M3), fp32 accumulate" if fmt == 2 else "%s x mxfp4, fp32 accumulate" % wfmt


EXPERT_NORM_EPS = 1e-6


def norm_eps(args):
    """eps of the per-expert output normalisation, or None when the layer runs without it."""
    return EXPERT_NORM_EPS if getattr(args, "expert_norm", False) else None


def layer_call(B, args, x, L, T, d, E, k, I, fmt, y, ids, w, ws, stream):
    """One layer call through the C ABI (with the per-expert normalisation when asked for)."""
    if norm_eps(args) is None:
        B.moe_layer_forward(x, L.W_r, L.b, T, d, E, k, I, L.weights, fmt, y, ids, w, ws, stream=stream)
    else:
        B.moe_layer_forward_norm(x, L.W_r, L.b, T, d, E, k, I, L.weights, fmt, norm_eps(args), y, ids, w, ws,
                                 stream=stream)


TENSOR_W_IN, TENSOR_W_OUT = 10, 11  # generator streams of the shared latent projections


def workload_name(args, cfg):
    name = cfg.note
    if getattr(args, "latent", 0):
        name += " + shared latent projections %d -> %d -> %d" % (cfg.d, args.latent, cfg.d)
    if norm_eps(args):
        name += " + per-expert RMSNorm before the weighted sum"
    if getattr(args, "weights", "mxfp4") == "nvfp4":
        name += ", NVFP4 expert weights (E4M3 scale per 16 values, fp32 scale per matrix)"
    return name


def moe_cfg(args, cfg):
    """The layer's own configuration: the workload's, or its latent width with --latent."""
    import dataclasses
    return dataclasses.replace(cfg, d=args.latent) if getattr(args, "latent", 0) else cfg


class Latent:
    """Shared latent projections around the layer (Muse Spark Open explainer, section 9): per layer
    copy a narrowing matrix [dl][dm] and a widening matrix [dm][dl] (MXFP4), their workspaces and
    the intermediate rows at the latent width."""

    def __init__(self, cfg, dl, fmt, dev, layers):
        import torch

        from bit_expert_ffn_moe_gb300 import binding as B
        from bit_expert_ffn_moe_gb300.layer import DeviceMatrix
        self.B, self.fmt, self.T, self.dm, self.dl = B, fmt, cfg.T, cfg.d, dl
        mma = fmt != B.MOE_ACT_BF16
        self.win = [DeviceMatrix(dl, cfg.d, L.seed, TENSOR_W_IN, cfg.weight_std, mma, dev) for L in layers]
        self.wout = [DeviceMatrix(cfg.d, dl, L.seed, TENSOR_W_OUT, cfg.weight_std, mma, dev) for L in layers]

        def ws(K, N):
            w = torch.empty(B.moe_dense_workspace_size(cfg.T, K, N, fmt), dtype=torch.uint8, device=dev)
            B.moe_workspace_init(w)
            return w
        self.ws_in, self.ws_out = ws(cfg.d, dl), ws(dl, cfg.d)
        self.xl = torch.empty((cfg.T, dl), dtype=torch.bfloat16, device=dev)
        self.yl = torch.empty((cfg.T, dl), dtype=torch.bfloat16, device=dev)

    def narrow(self, s, x, out, st):
        self.B.moe_dense_linear(x, self.T, self.dm, self.dl, self.win[s % len(self.win)].struct, self.fmt, out,
                                self.ws_in, stream=st)

    def widen(self, s, yl, y, st):
        self.B.moe_dense_linear(yl, self.T, self.dl, self.dm, self.wout[s % len(self.wout)].struct, self.fmt, y,
                                self.ws_out, stream=st)

    def bytes_per_step(self):
        return 2.0 * self.dm * self.dl * 17 / 32

    def flops_per_step(self):
        return 4.0 * self.T * self.dm * self.dl

    def status(self, st):
        B = self.B
        for w in (self.ws_in, self.ws_out):
            v = B.moe_get_device_status(w, stream=st)
            if v != B.MOE_OK:
                return v
        return B.MOE_OK


def screened_route(T, d, E):
    """Whether the library routes T tokens with the tensor-core screen (router split, screen,
    candidates, exact logits, top-k: five launches instead of the dense logits + top-k)."""
    return T >= 256 and d % 128 == 0 and d <= 32768 and E <= 1024 and T * E <= (1 << 25)


def launches_per_step(fmt, T, d, E, k, expert_norm=False, latent=False, mma_decode=False, nv_grouped=False):
    # Route + permutation: up to 8 tokens one launch (the decode router, or the expert kernel itself);
    # beyond, logits, top-k (which also counts the picks per expert) and the permutation (offsets,
    # plan and rows in one launch); the screened router (many tokens) adds three launches.
    # BF16 GEMVs: route (+ permutation), gate/up, down+sum; with the expert normalisation the down
    # GEMV and the (normalising) sum are separate launches.  MXFP4 (any T): logits, top-k,
    # permutation, the operand rows (quantised and written to their padded rows), up, down, sum.
    # Each latent projection: plan + GEMV (BF16) or plan + operand rows + GEMM (MXFP4).
    proj = (2 if fmt == 0 else 3) * 2 if latent else 0
    proj += 3 if screened_route(T, d, E) else 0
    route = 1 if T <= 8 else 3
    if fmt == 0 or (fmt == 2 and mma_decode):
        if mma_decode:
            # up to 8 tokens (E <= 152): one launch that routes, builds the token pieces and runs both
            # GEMMs; else route + permutation, token pieces, the expert kernel; + a separate sum when
            # the weighted sum is not fused (more than four tokens, or normalised expert outputs)
            sep_sum = 0 if (T <= 4 and not expert_norm) else 1
            return (1 if (T <= 8 and E <= 152) else route + 2) + sep_sum + proj
        return route + 2 + (1 if expert_norm else 0) + proj
    return 7 + (2 if nv_grouped else 0) + proj  # NVFP4 weights: + the two operand-scale conversions


def kernel_roofline(args, cfg, layers, xs, fmt, dev, stream, pk):
    """Average duration of the dominant kernel over the same steps, timed with CUDA events on the
    stream it is launched on, and its algorithmic bytes per launch."""
    import numpy as np
    import torch

    from bit_expert_ffn_moe_gb300 import binding as B
    from bit_expert_ffn_moe_gb300.layer import make_workspace

    T, d, E, k, I = cfg.T, cfg.d, cfg.E, cfg.k, cfg.I
    P = T * k
    ws = make_workspace(T, d, E, k, I, fmt, dev)
    i32 = dict(dtype=torch.int32, device=dev)
    ids, w = torch.empty((T, k), **i32), torch.empty((T, k), dtype=torch.float32, device=dev)
    counts, offsets, perm, inv = torch.empty(E, **i32), torch.empty(E + 1, **i32), torch.empty(P, **i32), \
        torch.empty(P, **i32)
    h = torch.empty((P, I), dtype=torch.bfloat16, device=dev)
    n = min(args.steps, 200)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    active = []
    if grouped_gemm_path(fmt, T):
        return kernel_roofline_mxfp4(args, cfg, layers, xs, fmt, dev, stream, pk, n)
    if args.weights == "mxfp4" and B.moe_decode_pieces_bytes(T, d, 0) > 0 and I % 256 == 0:
        return kernel_roofline_decode_mma(args, cfg, layers, xs, fmt, dev, stream, pk, n)
    st = stream.cuda_stream
    with torch.cuda.stream(stream):
        for s in range(n + 3):
            L = layers[s % len(layers)]
            x = xs[s % xs.shape[0]]
            B.moe_route(x, L.W_r, L.b, T, d, E, k, ids, w, ws, stream=st)
            B.moe_permute(x, ids, T, d, E, k, fmt, counts, offsets, perm, inv, None, None, ws, stream=st)
            if s >= 3:
                evs[s - 3][0].record(stream)
            B.moe_expert_up_swiglu(x, None, None, fmt, perm, offsets, T, d, E, k, I, L.weights, h, None, ws,
                                   stream=st)
            if s >= 3:
                evs[s - 3][1].record(stream)
                active.append(torch.count_nonzero(counts))
    stream.synchronize()
    dur = [a.elapsed_time(b) for a, b in evs]
    n_act = float(np.mean([int(a.item()) for a in active]))
    per_launch = n_act * up_bytes_per_expert(d, I, args.weights) + T * d * 2 + P * I * 2
    avg_ms = float(np.mean(dur))
    achieved = per_launch / (avg_ms / 1e3) / 1e9
    profile = "gemv_up_decode.md" if args.weights == "mxfp4" else "gemv_up_decode_nvfp4.md"
    traffic = ncu_traffic(profile, ["bit_expert_ffn_moe_gb300/csrc/gemv.cu",
                                    "bit_expert_ffn_moe_gb300/csrc/common.cuh"], traffic_workload(args, cfg))
    return {"kernel": "gemv_up_kernel (gate/up + SwiGLU, decode)", "bound": "hbm",
            "timing": "each launch bracketed by events through the step API (eager; inside the timed graph the "
                      "launch overlaps its neighbours through programmatic dependent launch)",
            "achieved": round(achieved, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
            "frac": round(achieved / pk["hbm_gbs"], 4), "traffic": traffic,
            "algorithmic_bytes_per_launch": per_launch, "avg_launch_us": round(avg_ms * 1e3, 3),
            "launches_timed": n, "peak_source": pk["source"] + " (HBM copy bandwidth)"}


def kernel_roofline_decode_mma(args, cfg, layers, xs, fmt, dev, stream, pk, n):
    """bf16 decode path on the tensor cores: the fused expert kernel (umma_decode_layer_kernel: gate/up
    + SwiGLU + down, and the weighted sum for up to four tokens) timed with CUDA events on its stream
    through moe_expert_ffn_decode, after moe_route, moe_permute and moe_decode_pieces (the token pieces).
    Algorithmic bytes per launch: every touched expert's gate, up and down weights, plus y."""
    import numpy as np
    import torch

    from bit_expert_ffn_moe_gb300 import binding as B
    from bit_expert_ffn_moe_gb300.layer import make_workspace

    T, d, E, k, I = cfg.T, cfg.d, cfg.E, cfg.k, cfg.I
    P = T * k
    ws = make_workspace(T, d, E, k, I, fmt, dev)
    i32 = dict(dtype=torch.int32, device=dev)
    u8 = dict(dtype=torch.uint8, device=dev)
    ids, w = torch.empty((T, k), **i32), torch.empty((T, k), dtype=torch.float32, device=dev)
    counts, offsets, perm, inv = torch.empty(E, **i32), torch.empty(E + 1, **i32), torch.empty(P, **i32), \
        torch.empty(P, **i32)
    xa = torch.empty(B.moe_decode_pieces_bytes(T, d, 0), **u8)
    xa_s = torch.empty(B.moe_decode_pieces_bytes(T, d, 1), **u8)
    y_perm = torch.empty((P, d), dtype=torch.bfloat16, device=dev)
    y = torch.empty((T, d), dtype=torch.bfloat16, device=dev) if T <= 4 else None
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    active = []
    st = stream.cuda_stream
    with torch.cuda.stream(stream):
        for s in range(n + 3):
            L = layers[s % len(layers)]
            x = xs[s % xs.shape[0]]
            B.moe_route(x, L.W_r, L.b, T, d, E, k, ids, w, ws, stream=st)
            B.moe_permute(x, ids, T, d, E, k, fmt, counts, offsets, perm, inv, None, None, ws, stream=st)
            B.moe_decode_pieces(x, T, d, fmt, xa, xa_s, stream=st)
            if s >= 3:
                evs[s - 3][0].record(stream)
            B.moe_expert_ffn_decode(xa, xa_s, fmt, perm, offsets, inv, w, T, d, E, k, I, L.weights, y_perm, y, ws,
                                    stream=st)
            if s >= 3:
                evs[s - 3][1].record(stream)
                active.append(torch.count_nonzero(counts))
    stream.synchronize()
    if B.moe_get_device_status(ws) != B.MOE_OK:
        raise RuntimeError("device-side error in the decode roofline loop")
    avg_ms = float(np.mean([a.elapsed_time(b) for a, b in evs]))
    n_act = float(np.mean([int(a.item()) for a in active]))
    per_launch = n_act * expert_read_bytes(d, I, "mxfp4") + T * d * 2
    achieved = per_launch / (avg_ms / 1e3) / 1e9
    profile = "umma_decode_layer.md" if cfg.name == "decode" else "umma_decode_layer_%s.md" % cfg.name
    traffic = ncu_traffic(profile, DECODE_KERNEL_SOURCES,
                          traffic_workload(args, cfg, "+mxfp8" if fmt == B.MOE_ACT_MXFP8 else ""))
    return {"kernel": "umma_decode_layer_kernel (tcgen05 kind::mxf4 gate/up + SwiGLU + down%s, decode)"
                      % (" + weighted sum" if y is not None else ""),
            "bound": "hbm", "achieved": round(achieved, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
            "frac": round(achieved / pk["hbm_gbs"], 4), "traffic": traffic,
            "algorithmic_bytes_per_launch": per_launch, "avg_launch_us": round(avg_ms * 1e3, 3),
            "launches_timed": n, "peak_source": pk["source"] + " (HBM copy bandwidth)",
            "timing": "each launch bracketed by events through the step API (eager; in the timed graph the "
                      "launch also overlaps its predecessors through programmatic dependent launch)"}


def kernel_roofline_mxfp4(args, cfg, layers, xs, fmt, dev, stream, pk, n):
    """Prefill path: the tcgen05 gate/up kernel (umma_grouped_kernel<1, fp8>) timed with CUDA events
    on its stream through the step API, against the dense FP4 (MXFP8 activations: FP8) tensor peak
    (the measured or fallback bf16 peak times the nominal ratio); its HBM rate is reported beside."""
    import numpy as np
    import torch

    from bit_expert_ffn_moe_gb300 import binding as B
    from bit_expert_ffn_moe_gb300.layer import make_workspace

    T, d, E, k, I = cfg.T, cfg.d, cfg.E, cfg.k, cfg.I
    P = T * k
    R = B.moe_padded_rows(T, k, E)
    ws = make_workspace(T, d, E, k, I, fmt, dev)
    i32 = dict(dtype=torch.int32, device=dev)
    u8 = dict(dtype=torch.uint8, device=dev)
    ids, w = torch.empty((T, k), **i32), torch.empty((T, k), dtype=torch.float32, device=dev)
    counts, offsets, perm, inv = torch.empty(E, **i32), torch.empty(E + 1, **i32), torch.empty(P, **i32), \
        torch.empty(P, **i32)
    per_byte = 1 if fmt == 2 else 2  # values per code byte of the token operand and h
    xa, xa_s = torch.empty(R * d // per_byte, **u8), torch.empty(B.moe_mxfp4_mma_scale_bytes(R, d), **u8)
    h, h_s = torch.empty(R * I // per_byte, **u8), torch.empty(B.moe_mxfp4_mma_scale_bytes(R, I), **u8)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    active = []
    st = stream.cuda_stream
    with torch.cuda.stream(stream):
        for s in range(n + 3):
            L = layers[s % len(layers)]
            x = xs[s % xs.shape[0]]
            B.moe_route(x, L.W_r, L.b, T, d, E, k, ids, w, ws, stream=st)
            B.moe_permute(x, ids, T, d, E, k, fmt, counts, offsets, perm, inv, xa, xa_s, ws, stream=st)
            if s >= 3:
                evs[s - 3][0].record(stream)
            B.moe_expert_up_swiglu(None, xa, xa_s, fmt, perm, offsets, T, d, E, k, I, L.weights, h, h_s, ws,
                                   stream=st)
            if s >= 3:
                evs[s - 3][1].record(stream)
                active.append(torch.count_nonzero(counts))
    stream.synchronize()
    if B.moe_get_device_status(ws) != B.MOE_OK:
        raise RuntimeError("device-side error in the prefill roofline loop")
    avg_ms = float(np.mean([a.elapsed_time(b) for a, b in evs]))
    n_act = float(np.mean([int(a.item()) for a in active]))
    flops = 4.0 * P * d * I  # gate and up: 2 flops per weight per token row
    achieved = flops / (avg_ms / 1e3) / 1e12
    ratio = tensor_peak_ratio(fmt)
    peak_tf = pk["bf16_tflops"] * ratio
    act_bytes = 33 / 32 if fmt == 2 else 17 / 32  # per value: codes + scale of the token operand / h
    hbm_bytes = n_act * up_bytes_per_expert(d, I, args.weights) + P * d * act_bytes + P * I * act_bytes
    fp8 = fmt == 2
    nv = args.weights == "nvfp4"
    kind = 2 if nv else int(fp8)
    profile = "umma_grouped_prefill_mxfp8.md" if fp8 else ("umma_grouped_prefill_nvfp4.md" if nv
                                                           else "umma_grouped_prefill.md")
    if cfg.name != "prefill":  # another workload's capture (e.g. umma_grouped_long_prefill.md)
        profile = profile.replace("umma_grouped_prefill", "umma_grouped_" + cfg.name)
    traffic = ncu_traffic(profile, GROUPED_KERNEL_SOURCES, traffic_workload(args, cfg))
    return {"kernel": "umma_grouped_kernel<1, %d> (tcgen05 %s gate/up + SwiGLU, prefill)"
                      % (kind, ["kind::mxf4", "kind::mxf8f6f4", "kind::mxf4nvf4"][kind]), "bound": "tensor",
            "achieved": round(achieved, 1), "peak": round(peak_tf, 1), "unit": "TFLOP/s",
            "frac": round(achieved / peak_tf, 4), "traffic": traffic,
            "algorithmic_flops_per_launch": flops, "avg_launch_us": round(avg_ms * 1e3, 3), "launches_timed": n,
            "hbm_achieved_GBps": round(hbm_bytes / (avg_ms / 1e3) / 1e9, 1),
            "hbm_frac": round(hbm_bytes / (avg_ms / 1e3) / 1e9 / pk["hbm_gbs"], 4),
            "algorithmic_bytes_per_launch": hbm_bytes,
            "peak_source": pk["source"] + " bf16 x %.0f (nominal %s : bf16 dense ratio)"
                           % (ratio, "FP8" if fp8 else "FP4")}


def end_to_end(args, cfg, cm, xs_host, fmt, dev, stream, call, host_call=None):
    """Same metric through the C ABI with host buffers: every step copies its x from pinned host
    memory and its y back to pinned host memory inside the timed region.  The plain layer goes
    through the host-buffer layer call (moe_layer_forward_host: copy in, layer, copy out, one C
    call per step, the copies on an input and an output copy stream with two alternating staging
    pairs).  The options without a host-buffer entry point (expert normalisation, latent
    projections) run the copies on a second stream with double-buffered device x and y, so the
    copy of step s + 1's input and of step s's output overlap step s's layer call."""
    import numpy as np
    import torch

    from bit_expert_ffn_moe_gb300.layer import make_workspace

    T, d, E, k, I = cfg.T, cfg.d, cfg.E, cfg.k, cfg.I
    n = min(args.steps, 500)
    x_pin = torch.from_numpy(xs_host[:n].view(np.int16).copy()).view(torch.bfloat16).pin_memory()
    y_pin = torch.empty((min(n, 4), T, d), dtype=torch.bfloat16).pin_memory()  # a ring of host outputs
    x_dev = [torch.empty((T, d), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    y_dev = [torch.empty((T, d), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    ws = make_workspace(T, cm.d, E, k, I, fmt, dev)
    cs = torch.cuda.Stream(device=dev)  # copies
    st = stream.cuda_stream
    ev_in = [torch.cuda.Event() for _ in range(2)]     # x of a buffer has landed
    ev_done = [torch.cuda.Event() for _ in range(2)]   # the layer call of a buffer is finished
    ev_out = [torch.cuda.Event() for _ in range(2)]    # y of a buffer has been read back

    def h2d(s):
        b = s % 2
        with torch.cuda.stream(cs):
            if s >= 2:
                cs.wait_event(ev_done[b])  # step s - 2 has consumed this x buffer
            x_dev[b].copy_(x_pin[s % x_pin.shape[0]], non_blocking=True)
            ev_in[b].record(cs)

    def run(steps):
        h2d(0)
        for s in range(steps):
            b = s % 2
            if s + 1 < steps:
                h2d(s + 1)
            with torch.cuda.stream(stream):
                stream.wait_event(ev_in[b])
                if s >= 2:
                    stream.wait_event(ev_out[b])  # y of step s - 2 has left this buffer
                call(s, x_dev[b], y_dev[b], None, None, ws, st)
                ev_done[b].record(stream)
            with torch.cuda.stream(cs):
                cs.wait_event(ev_done[b])
                y_pin[s % y_pin.shape[0]].copy_(y_dev[b], non_blocking=True)
                ev_out[b].record(cs)

    if host_call is not None:
        xh = [x_pin[i].data_ptr() for i in range(x_pin.shape[0])]
        yh = [y_pin[i].data_ptr() for i in range(y_pin.shape[0])]
        xd = [t.data_ptr() for t in x_dev]
        yd = [t.data_ptr() for t in y_dev]
        ws_a = (ws.data_ptr(), ws.numel() * ws.element_size())
        cs_out = torch.cuda.Stream(device=dev)  # copies out (cs: copies in)
        cst = (cs.cuda_stream, cs_out.cuda_stream)

        def run(steps):
            for s in range(steps):
                host_call(s, xh[s % len(xh)], yh[s % len(yh)], xd[s % 2], yd[s % 2], ws_a, st, cst)
        note = ("moe_layer_forward_host per step (eager, no graph, one C-ABI call): pinned H2D of x, the layer, "
                "D2H of y; the copies on two copy streams (in, out) with two alternating staging pairs, so they "
                "overlap the neighbouring steps' layers")
        start_stream, end_stream = cs, cs_out
    else:
        note = ("eager C-ABI calls per step (no graph); every step's pinned H2D of x and D2H of y inside the "
                "timed region, on a copy stream with double-buffered device x and y, so step s + 1's input and "
                "step s's output move while step s computes")
        start_stream = end_stream = cs
    run(3)
    torch.cuda.synchronize(dev)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    start.record(start_stream)
    stream.wait_event(start)
    run(n)
    end.record(end_stream)  # after the last read-back (on a copy stream, which waited for the last layer call)
    end.synchronize()
    wall = time.perf_counter() - t0
    ms = start.elapsed_time(end)
    return {"value": round(T * n / (ms / 1e3), 1), "unit": UNIT, "h2d_bytes_per_step": T * d * 2,
            "d2h_bytes_per_step": T * d * 2, "steps": n, "wall_tokens_per_s": round(T * n / wall, 1),
            "note": note}


# ------------------------------------------------------------------ CPU oracle arm

# Output tolerance of the layer (the parity tests' bar): relative Frobenius error and max abs
# error over the RMS of the oracle output, over the checked tokens.
PARITY_REL_FRO, PARITY_MAX_ABS_RMS = 5e-3, 3e-2


def sample_layer_index(args):
    """The layer copy the oracle sample and the bench's parity gate use."""
    return 1 if getattr(args, "layers", 2) > 1 else 0


def parity_inputs(cfg, n_tokens):
    """The inputs of the oracle sample: (bf16 bits x [T][d], checked rows or None for all).
    Decode sizes: n_tokens whole layer calls; prefill sizes: one call (chunk 0) and the workload's
    seeded token sample (256 tokens of the prefill chunk, 512 of a long-prefill chunk), or n_tokens
    evenly spread rows when the workload names no sample."""
    import numpy as np

    from bit_expert_ffn_moe_gb300 import inputs as IN
    if cfg.T <= 8:
        return [(IN.make_x(cfg, call=c), None) for c in range(n_tokens)]
    if cfg.sample_tokens:
        return [(IN.make_x(cfg, call=0), IN.sample_tokens(cfg, cfg.T))]
    return [(IN.make_x(cfg, call=0), np.arange(0, cfg.T, max(1, cfg.T // n_tokens))[:n_tokens])]


def parity_gate(gpu_ys, oracle_ys, gpu_ids=None, oracle_ids=None):
    """Compare the GPU's outputs of the sampled tokens with the oracle's (and its routing of every
    token of those calls, which must be identical); refuse to record a timing whose output or
    routing is wrong."""
    import numpy as np
    routing = None
    if gpu_ids is not None and oracle_ids is not None:
        gi = [np.asarray(a) for a in gpu_ids]
        oi = [np.asarray(a) for a in oracle_ids]
        routing = bool(len(gi) == len(oi) and all(a.shape == b.shape and np.array_equal(a, b) for a, b in zip(gi, oi)))
        if not routing:
            raise RuntimeError("refusing to record: routing differs from the oracle")
    g = np.concatenate([np.asarray(y, dtype=np.float64).reshape(-1, np.shape(y)[-1]) for y in gpu_ys])
    o = np.concatenate([np.asarray(y, dtype=np.float64).reshape(-1, np.shape(y)[-1]) for y in oracle_ys])
    if g.shape != o.shape:
        raise RuntimeError("refusing to record: parity sample shapes differ %s vs %s" % (g.shape, o.shape))
    ref = np.linalg.norm(o)
    rms = np.sqrt(np.mean(o ** 2))
    rel = float(np.linalg.norm(g - o) / ref) if ref > 0 else float("inf")
    mx = float(np.max(np.abs(g - o)) / rms) if rms > 0 else float("inf")
    ok = bool(np.all(np.isfinite(g)) and rel <= PARITY_REL_FRO and mx <= PARITY_MAX_ABS_RMS)
    out = {"rows_checked": int(g.shape[0]), "rel_fro": rel, "max_abs_over_rms": mx,
           "tolerance": {"rel_fro": PARITY_REL_FRO, "max_abs_over_rms": PARITY_MAX_ABS_RMS}, "ok": ok}
    if routing is not None:
        out["routing_bit_exact"] = routing
        out["tokens_routed"] = int(sum(np.asarray(a).shape[0] for a in gpu_ids))
    if not ok:
        raise RuntimeError("refusing to record: output differs from the oracle: %s" % json.dumps(out))
    return out


def oracle_sample(args, cfg, n_tokens, threads=None):
    """Time the CPU oracle (as it stands) on a bounded sample of the workload: routing,
    dequantisation of the touched experts, expert GEMVs and the weighted sum (with --latent also
    the two projections of the sampled tokens).  Weight generation is untimed.  threads: OpenMP
    threads for this sample (default: all host cores).  The result's "ys" holds the outputs of
    the rows that parity_inputs() names."""
    from oracle import oracle as O

    O.set_threads(threads or len(os.sched_getaffinity(0)))
    try:
        res = _oracle_sample(args, cfg, n_tokens)
        res["cores"] = O.max_threads()
    finally:
        O.set_threads(len(os.sched_getaffinity(0)))
    return res


def _oracle_sample(args, cfg, n_tokens):
    import numpy as np

    from bit_expert_ffn_moe_gb300 import inputs as IN
    from oracle import oracle as O

    threads = O.max_threads()
    cm = moe_cfg(args, cfg)
    li = sample_layer_index(args)
    layer_seed = cfg.seed + 7919 * li
    W_r, b = IN.make_router(cm)
    if li != 0:  # the router of that layer copy
        rng = np.random.default_rng([cm.seed, 77, li])
        W_r = (rng.standard_normal(W_r.shape) / np.sqrt(cm.d)).astype(np.float32)
    shapes = IN.expert_matrix_shapes(cm)
    cache = {}

    def weights(e):
        if e not in cache:
            out = {}
            for name, tid in (("gate", IN.TENSOR_GATE), ("up", IN.TENSOR_UP), ("down", IN.TENSOR_DOWN)):
                rows, K = shapes[tid]
                w = IN.synth_weights(layer_seed, tid, e, rows, K, cfg.weight_std)
                out[name] = O.nvfp4_pack(w) if getattr(args, "weights", "mxfp4") == "nvfp4" else O.mxfp4_pack(w)
            cache[e] = out
        return cache[e]

    act = {"bf16": O.ACT_BF16, "mxfp4": O.ACT_MXFP4, "mxfp8": O.ACT_MXFP8}[args.fmt]
    eps = norm_eps(args)
    if getattr(args, "latent", 0):
        win = O.mxfp4_pack(IN.synth_weights(layer_seed, TENSOR_W_IN, 0, cm.d, cfg.d, cfg.weight_std))
        wout = O.mxfp4_pack(IN.synth_weights(layer_seed, TENSOR_W_OUT, 0, cfg.d, cm.d, cfg.weight_std))

        def full(xb):  # narrow -> layer -> widen, on the sampled rows
            xl = IN.to_bf16_bits(O.dense_linear(xb, win, act))
            yl = O.moe_layer(xl, W_r, b, cfg.k, weights, act, expert_norm_eps=eps)["y"]
            return O.dense_linear(IN.to_bf16_bits(yl), wout, act)

        xs = [xb if rows is None else xb[rows] for xb, rows in parity_inputs(cfg, n_tokens)]
        for xb in xs:  # pre-generate the touched experts (untimed: input generation)
            xl = IN.to_bf16_bits(O.dense_linear(xb, win, act))
            for e in np.unique(O.topk_softmax(O.router_logits(xl, W_r, b), cfg.k)[0]):
                weights(int(e))
        t0 = time.perf_counter()
        ys = [full(xb) for xb in xs]
        dt = time.perf_counter() - t0
        rows = sum(xb.shape[0] for xb in xs)
        return dict(value=round(rows / dt, 3), unit=UNIT, cores=threads, kind="oracle",
                    sample="%d token rows through narrow -> layer (routing of those rows) -> widen, fp64 oracle, "
                           "weights pre-generated" % rows, seconds=round(dt, 2), ys=ys, ids=None)
    if cfg.T <= 8:
        # decode sizes: whole layer calls
        xs = [xb for xb, _ in parity_inputs(cfg, n_tokens)]
        for xb in xs:  # pre-generate the experts the sample touches (untimed: input generation)
            ids, _ = O.topk_softmax(O.router_logits(xb, W_r, b), cfg.k)
            for e in np.unique(ids):
                weights(int(e))
        touched, routed = [], []
        for xb in xs:
            ids, _ = O.topk_softmax(O.router_logits(xb, W_r, b), cfg.k)
            touched.append(len(np.unique(ids)))
            routed.append(ids)
        t0 = time.perf_counter()
        ys = [O.moe_layer(xb, W_r, b, cfg.k, weights, act, expert_norm_eps=eps)["y"] for xb in xs]
        dt = time.perf_counter() - t0
        return dict(value=round(cfg.T * n_tokens / dt, 3), unit=UNIT, cores=threads, kind="oracle",
                    sample="%d layer calls of T=%d (full routing, every touched expert: %.1f per call on average, "
                           "fp64 oracle), weights pre-generated" % (n_tokens, cfg.T, float(np.mean(touched))),
                    seconds=round(dt, 2), ys=ys, ids=routed)
    # prefill sizes: routing of the whole chunk, expert work for a token sample; per-token cost =
    # routing time / T + expert time / sample size
    (xb, tokens), = parity_inputs(cfg, n_tokens)
    t0 = time.perf_counter()
    ids, _ = O.topk_softmax(O.router_logits(xb, W_r, b), cfg.k)
    t_route = time.perf_counter() - t0
    for e in np.unique(ids[tokens]):
        weights(int(e))
    t0 = time.perf_counter()
    y_tok = O.moe_layer(xb[tokens], W_r, b, cfg.k, weights, act, expert_norm_eps=eps)["y"]
    t_exp = time.perf_counter() - t0
    per_tok = t_route / cfg.T + t_exp / len(tokens)
    return dict(value=round(1.0 / per_tok, 3), unit=UNIT, cores=threads, kind="oracle",
                sample="routing of all %d tokens (%.2f s) + expert FFNs and sum for %d sampled tokens (%.2f s), "
                       "fp64 oracle, weights pre-generated; tokens/s = 1 / (route/T + experts/sample)"
                       % (cfg.T, t_route, len(tokens), t_exp), seconds=round(t_route + t_exp, 2), ys=[y_tok],
                ids=[ids])


def run_reference(args, cfg, rank, world):
    if rank != 0:
        return None
    os.environ.setdefault("OMP_NUM_THREADS", str(len(os.sched_getaffinity(0))))
    from oracle import oracle as O
    O.build()
    # each step: one layer call of the workload on the CPU oracle; bounded so the run ends in
    # a few minutes (at most args.ref_budget seconds of timed oracle work)
    probe = oracle_sample(args, cfg, 1)
    per_step = cfg.T / max(probe["value"], 1e-9)
    n = max(1, min(args.steps, int(args.ref_budget / max(per_step, 1e-6))))
    res = oracle_sample(args, cfg, n)
    out = {"metric": METRIC, "value": res["value"], "unit": UNIT, "n_gpus": world, "steps": n,
           "warmup": 1, "ms_per_step": round(1e3 * cfg.T / res["value"], 3), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)", "data": "synthetic",
           "config": {"workload": workload_name(args, cfg),
                      "T": cfg.T, "d": cfg.d, "E": cfg.E, "k": cfg.k, "I": cfg.I, "act": args.fmt,
                      "weights": args.weights, "expert_norm_eps": norm_eps(args),
                      "latent_width": args.latent or None},
           "impl": "reference",
           "cpu_baseline": {"value": res["value"], "unit": UNIT, "cores": res["cores"], "kind": "oracle",
                            "sample": res["sample"] + "; %d of the %d requested steps" % (n, args.steps)},
           "e2e": {"value": res["value"], "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    return out


PREFILL_LAYER_COPIES = 2  # a prefill step reads ~3.4 GB of expert weights: far more than L2 already
SUB_KEYS = ("value", "unit", "ms_per_step", "steps", "warmup", "dtype", "config", "layer_roofline", "roofline",
            "e2e", "gpu_launches", "clocks", "wall_s_timed", "cpu_baseline", "parity")


# extra workload name -> (configuration, activation format)
EXTRA_WORKLOADS = {"spec_verify": ("spec_verify", "bf16"), "prefill": ("prefill", "mxfp4"),
                   "long_prefill": ("long_prefill", "mxfp4"), "prefill_mxfp8": ("prefill", "mxfp8")}


def extra_workloads(args):
    """Workloads timed after the headline one in the same run: speculative verification (four
    tokens), the prefill chunk, one chunk of the long prefill, and the prefill chunk with 8-bit
    activations, when the headline is the plain decode workload (no variant options)."""
    if args.extra == "none":
        return []
    if args.extra != "auto":
        return [n for n in args.extra.split(",") if n]
    plain = (args.config == "decode" and not args.latent and not args.expert_norm and args.weights == "mxfp4"
             and args.fmt == "bf16")
    return ["spec_verify", "prefill", "long_prefill", "prefill_mxfp8"] if plain else []


def run_workload(args, cfg, rank, world, local):
    """One workload: the GPU timing, then (rank 0, one GPU) the oracle sample, its time as the
    CPU baseline and the parity gate of the same rows (and routing) through the GPU layer."""
    out = run_gpu(args, cfg, rank, world, local)
    parity_y = out.pop("_parity_y", None)
    parity_ids = out.pop("_parity_ids", None)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res = oracle_sample(args, cfg, args.cpu_sample_tokens)
        out["cpu_baseline"] = {k: res[k] for k in ("value", "unit", "cores", "kind", "sample")}
        if cfg.T <= 8:  # a one-thread sample of the same kind (prefill sizes: tens of seconds, skipped)
            one = oracle_sample(args, cfg, 1, threads=1)
            out["cpu_baseline"]["single_thread"] = {k: one[k] for k in ("value", "cores", "sample")}
        # the same rows on the GPU (layer copy sample_layer_index) against the oracle
        out["parity"] = parity_gate(parity_y, res["ys"], parity_ids, res["ids"])
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="decode")
    ap.add_argument("--extra", default="auto",
                    help="workloads timed after the headline one ('auto': prefill and one long-prefill chunk "
                         "when the headline is the plain decode workload; 'none'; or a comma list)")
    ap.add_argument("--fmt", choices=["bf16", "mxfp4", "mxfp8"], default=None)
    ap.add_argument("--layers", type=int, default=N_LAYER_COPIES)
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--latent", type=int, default=0,
                    help="latent width: narrow x with a shared MXFP4 matrix before the router, run the layer "
                         "at that width and widen the weighted sum back (0 = off)")
    ap.add_argument("--expert-norm", action="store_true",
                    help="normalise each expert output (RMSNorm over d, eps 1e-6) before the weighted sum")
    ap.add_argument("--weights", choices=["mxfp4", "nvfp4"], default="mxfp4",
                    help="expert weight format (nvfp4: E4M3 scale per 16 values; bf16 activations only)")
    ap.add_argument("--experts", type=int, default=0,
                    help="number of experts E (0 = the workload's); profiling captures use a smaller E so that "
                         "few GB stay resident (per-expert shapes, T and k unchanged)")
    ap.add_argument("--cpu-sample-tokens", type=int, default=4)
    ap.add_argument("--ref-budget", type=float, default=90.0)
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    from bit_expert_ffn_moe_gb300 import inputs as IN
    cfg = IN.CONFIGS[args.config]
    if args.experts:
        import dataclasses
        cfg = dataclasses.replace(cfg, E=args.experts, note=cfg.note + " (E=%d for profiling)" % args.experts)
    if args.fmt is None:
        args.fmt = "bf16" if cfg.T <= 8 or args.weights == "nvfp4" else "mxfp4"
    if args.weights == "nvfp4" and args.fmt == "mxfp8":
        ap.error("NVFP4 expert weights are read by the bf16 and MXFP4 activation paths")
    rank, world, local = dist_env()

    if args.impl == "reference":
        out = run_reference(args, cfg, rank, world)
        if out is not None:
            print(json.dumps(out), flush=True)
        return

    os.environ.setdefault("OMP_NUM_THREADS", str(len(os.sched_getaffinity(0))))
    out = run_workload(args, cfg, rank, world, local)
    # With the default workload the same process also times speculative verification (the HBM
    # roofline at four tokens), the prefill chunk and one chunk of the long prefill (the other half
    # of the metric: the FP4 tensor roofline) and the prefill chunk with MXFP8 activations (the FP8
    # tensor roofline), each in a sub-object.
    for name in extra_workloads(args):
        import gc

        import torch
        gc.collect()
        torch.cuda.empty_cache()
        sub_args = argparse.Namespace(**vars(args))
        conf, act = EXTRA_WORKLOADS[name]
        sub_args.config, sub_args.fmt, sub_args.layers = conf, act, PREFILL_LAYER_COPIES
        sub = run_workload(sub_args, IN.CONFIGS[conf], rank, world, local)
        out[name] = {k: sub[k] for k in SUB_KEYS if k in sub}
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
