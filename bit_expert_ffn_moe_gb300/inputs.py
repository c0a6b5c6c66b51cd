"""Seeded synthetic inputs for the MoE expert-FFN layer.

This module holds input generation only -- none of the layer's arithmetic.  Both the CUDA
path (tests, benchmark) and the CPU oracle receive their inputs from here.

Two generators are used:

* numpy's ``default_rng`` (PCG64) for the host-side tensors: activations ``x`` (bf16),
  router weights ``W_r``, router bias ``b``, outlier rows and token samples.
* SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number generators",
  OOPSLA 2014), used as a counter-based generator, for the expert weight matrices.  The
  library's ``moe_synth_weights`` implements the same definition on the device, so a
  3.4 GB weight layer never has to be created on the host; the oracle regenerates only
  the experts it needs, here, from the same counters.  Each value is
  ``float32(2*(u0+u1+u2+u3) - 4*65535) * c`` where ``u0..u3`` are the four 16-bit fields
  of one SplitMix64 output and ``c = float32(std / SIGMA_V)``: a zero-mean Irwin-Hall(4)
  variate with standard deviation ``std`` (a close, bounded stand-in for N(0, std^2)).
  Integer work and one IEEE fp32 multiply make it bit-identical on both sides.

The five workloads (shapes, value distributions, routing skew) are those of the MoE layer
described in the Muse Spark Open explainer (sections 8-14) and the decode / speculative
verify regimes of the DGX Spark news item (section 3).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
SIGMA_V = 2.0 * math.sqrt((65536.0 ** 2 - 1.0) / 3.0)  # std of 2*(u0+u1+u2+u3) - 4*65535

TENSOR_GATE, TENSOR_UP, TENSOR_DOWN = 0, 1, 2


def splitmix64_mix(z: np.ndarray) -> np.ndarray:
    """The SplitMix64 output function applied to uint64 state values (wrapping arithmetic)."""
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def stream_key(seed: int, tensor_id: int, expert: int) -> np.uint64:
    """Key of the counter stream for one expert matrix (seed < 2^32, tensor_id < 256, expert < 2^24)."""
    assert 0 <= seed < 2 ** 32 and 0 <= tensor_id < 256 and 0 <= expert < 2 ** 24
    k = (np.uint64(seed) << np.uint64(32)) | (np.uint64(tensor_id) << np.uint64(24)) | np.uint64(expert)
    return splitmix64_mix(np.array([k], dtype=np.uint64))[0]


def weight_scale(std: float) -> np.float32:
    return np.float32(std / SIGMA_V)


_host_lib = None


def _host():
    """The C implementation of the same generator (inputs_host.c), built on first use; None if
    no C compiler is available (the numpy definition below is then used)."""
    global _host_lib
    if _host_lib is None:
        import ctypes
        import os
        import platform
        import subprocess
        here = os.path.dirname(os.path.abspath(__file__))
        src = os.path.join(here, "inputs_host.c")
        lib = os.path.join(here, "_build", "libinputs_%s.so" % platform.machine())
        try:
            if not os.path.exists(lib) or os.path.getmtime(lib) < os.path.getmtime(src):
                os.makedirs(os.path.dirname(lib), exist_ok=True)
                tmp = lib + ".tmp.%d" % os.getpid()
                subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared",
                                src, "-o", tmp], check=True)
                os.replace(tmp, lib)
            h = ctypes.CDLL(lib)
            h.inputs_stream_key.restype = ctypes.c_uint64
            h.inputs_stream_key.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32]
            h.inputs_synth.restype = None
            h.inputs_synth.argtypes = [ctypes.c_uint64, ctypes.c_int64, ctypes.c_int64, ctypes.c_float,
                                       ctypes.c_void_p]
            _host_lib = h
        except (OSError, subprocess.CalledProcessError):
            _host_lib = False
    return _host_lib or None


def synth_weights(seed: int, tensor_id: int, expert: int, rows: int, K: int, std: float,
                  row_start: int = 0, row_count: Optional[int] = None, use_c: bool = True) -> np.ndarray:
    """fp32 [row_count][K] rows ``row_start ..`` of one synthetic expert matrix [rows][K]."""
    if row_count is None:
        row_count = rows - row_start
    h = _host() if use_c else None
    if h is not None:
        out = np.empty((row_count, K), dtype=np.float32)
        key = h.inputs_stream_key(seed, tensor_id, expert)
        h.inputs_synth(key, row_start * K, row_count * K, float(weight_scale(std)), out.ctypes.data)
        return out
    key = stream_key(seed, tensor_id, expert)
    n = np.arange(row_start * K, (row_start + row_count) * K, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = splitmix64_mix(key + (n + np.uint64(1)) * GOLDEN)
    mask = np.uint64(0xFFFF)
    s = ((z & mask) + ((z >> np.uint64(16)) & mask) + ((z >> np.uint64(32)) & mask)
         + ((z >> np.uint64(48)) & mask)).astype(np.int64)
    v = (2 * s - 4 * 65535).astype(np.float32)
    return (v * weight_scale(std)).reshape(row_count, K)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (round to nearest even) and return the uint16 bit patterns."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclass(frozen=True)
class Config:
    name: str
    index: int          # 1-based workload number
    T: int              # tokens per layer call
    d: int              # hidden size
    E: int              # experts
    k: int              # experts per token
    I: int              # expert intermediate size
    calls: int = 1      # back-to-back layer calls (decode steps / prefill chunks)
    zipf_s: float = 0.0  # 0 = uniform expert prior (b = 0)
    outlier_frac: float = 0.0
    outlier_scale: float = 20.0
    weight_std: float = 0.02
    sample_tokens: int = 0   # 0 = oracle checks every token
    sample_seed: int = 0
    note: str = field(default="", compare=False)

    @property
    def seed(self) -> int:
        return 1000 + self.index

    @property
    def P(self) -> int:
        return self.T * self.k


CONFIGS = {
    "tiny": Config("tiny", 1, T=16, d=256, E=8, k=2, I=512,
                   note="tiny MoE layer: T=16, d=256, E=8, top-2, I=512"),
    "decode": Config("decode", 2, T=1, d=8192, E=128, k=8, I=2048, calls=1000,
                     note="decode, batch 1: T=1, d=8192, E=128, top-8, I=2048, uniform prior"),
    "spec_verify": Config("spec_verify", 3, T=4, d=8192, E=128, k=8, I=2048, calls=500,
                          note="speculative verify: T=4 (3 drafts + 1), d=8192, E=128, top-8, I=2048"),
    "prefill": Config("prefill", 4, T=4096, d=8192, E=128, k=8, I=2048, zipf_s=1.1,
                      sample_tokens=256, sample_seed=4,
                      note="prefill chunk: T=4096, d=8192, E=128, top-8, I=2048, Zipf(1.1) load"),
    "long_prefill": Config("long_prefill", 5, T=8192, d=4096, E=256, k=8, I=1536, calls=4, zipf_s=1.3,
                           outlier_frac=0.01, sample_tokens=512, sample_seed=5,
                           note="long prefill: 32768 tokens in 4 chunks of 8192, d=4096, E=256, top-8, "
                                "I=1536, Zipf(1.3) load, 1% outlier rows x20"),
}

_SUB = {"x": 1, "W_r": 2, "b": 3, "outliers": 4, "samples": 5}


def _rng(cfg: Config, name: str, extra: int = 0) -> np.random.Generator:
    return np.random.default_rng([cfg.seed, _SUB[name], extra])


def make_x(cfg: Config, call: int = 0, T: Optional[int] = None) -> np.ndarray:
    """bf16 bits [T][d] of layer call ``call``: N(0,1); for workloads with outliers, exactly
    round(frac*T) rows (seeded sample) multiplied by the outlier scale in fp32 before the one
    bf16 rounding."""
    T = cfg.T if T is None else T
    x = _rng(cfg, "x", call).standard_normal((T, cfg.d), dtype=np.float32)
    if cfg.outlier_frac > 0:
        n_out = int(round(cfg.outlier_frac * T))
        rows = _rng(cfg, "outliers", call).choice(T, size=n_out, replace=False)
        x[rows] *= np.float32(cfg.outlier_scale)
    return to_bf16_bits(x)


def make_router(cfg: Config):
    """W_r fp32 [E][d] ~ N(0, 1/d); b fp32 [E]: zeros for a uniform prior, else
    b_e = ln p_e with p_e proportional to rho(e)^(-s), rho a seeded permutation of 1..E."""
    W_r = (_rng(cfg, "W_r").standard_normal((cfg.E, cfg.d)) / math.sqrt(cfg.d)).astype(np.float32)
    if cfg.zipf_s > 0:
        ranks = _rng(cfg, "b").permutation(cfg.E).astype(np.float64) + 1.0
        p = ranks ** (-cfg.zipf_s)
        p /= p.sum()
        b = np.log(p).astype(np.float32)
    else:
        b = np.zeros(cfg.E, dtype=np.float32)
    return W_r, b


def sample_tokens(cfg: Config, total_tokens: int) -> np.ndarray:
    """Seeded sample (without replacement, sorted) of token indices the oracle checks."""
    if cfg.sample_tokens <= 0 or cfg.sample_tokens >= total_tokens:
        return np.arange(total_tokens, dtype=np.int64)
    rng = np.random.default_rng(cfg.sample_seed)
    return np.sort(rng.choice(total_tokens, size=cfg.sample_tokens, replace=False)).astype(np.int64)


def expert_matrix_shapes(cfg: Config):
    """(rows, K) of the gate, up and down matrices of one expert."""
    return {TENSOR_GATE: (cfg.I, cfg.d), TENSOR_UP: (cfg.I, cfg.d), TENSOR_DOWN: (cfg.d, cfg.I)}


def small_config(name: str, T: int, d: int, E: int, k: int, I: int, index: int = 90, **kw) -> Config:
    """An ad-hoc workload (tests): same generators, its own seed."""
    return Config(name, index, T=T, d=d, E=E, k=k, I=I, **kw)
