"""CPU oracle for the MoE expert-FFN layer -- ctypes wrapper around ``moe_oracle.c``.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this module.  It shares no code with the CUDA
library and never imports it; inputs come from the seeded generators and are passed in
as numpy arrays.

Each function follows one step of the layer as the sources state it (see the header of
``moe_oracle.c`` for the citations and the readings R1-R9 taken where they are silent):

* ``router_logits``  -- Muse Spark Open explainer, section 8 (one FP32 matrix product)
* ``topk_softmax``   -- section 8 (best k of E, a set) and section 9 (weights sum to 1)
* ``permute``        -- section 12 (tokens gathered per expert, one batch per expert)
* ``expert_ffn``     -- section 9 (gate / up / down) on MXFP4 weights (section 11, and the
                        DGX Spark news item, section 2)
* ``combine``        -- section 9 (weighted sum over the chosen experts)
* ``expert_norm``    -- section 9 (each chosen expert's output is normalised before the sum;
                        reading R8: RMSNorm over d, no learned scale)
* ``dense_linear``   -- section 9 (the shared latent projections around the experts; reading R9)
* ``nvfp4_pack``     -- section 11 (16 values share a small scale, about 4.5 bits each; reading
                        R10: E4M3 block scales after OCP OFP8, one fp32 global scale per matrix)
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess
from typing import Callable, Dict, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle_%s.so" % platform.machine())

ACT_BF16 = 0
ACT_MXFP4 = 1
ACT_EXACT = 2
ACT_MXFP8 = 3   # reading R11: E4M3 elements, one E8M0 scale per 32 (x and h)

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (ISO C, no FP contraction, OpenMP)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
           "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    P = ctypes.c_void_p
    i32, i64 = ctypes.c_int, ctypes.c_int64
    sig = {
        "oracle_e2m1_value": (ctypes.c_double, [i32]),
        "oracle_e8m0_value": (ctypes.c_double, [i32]),
        "oracle_e2m1_encode_magnitude": (i32, [ctypes.c_double]),
        "oracle_mx_block_quantize": (None, [P, i32, P, P]),
        "oracle_mxfp4_pack": (i32, [P, i64, i64, P, P]),
        "oracle_mxfp4_unpack": (i32, [P, P, i64, i64, P]),
        "oracle_router_logits": (None, [P, P, P, i32, i32, i32, P]),
        "oracle_topk_softmax": (None, [P, i32, i32, i32, P, P]),
        "oracle_permute": (i32, [P, i32, i32, i32, P, P, P, P]),
        "oracle_activation_row": (None, [P, i32, i32, P, P, P]),
        "oracle_expert_ffn": (None, [P, i32, i32, i32, P, P, P, P, P, P, i32, P, P, P, P]),
        "oracle_combine": (None, [P, P, P, i32, P, i32, i32, P]),
        "oracle_expert_norm": (None, [P, i64, i32, ctypes.c_double, P]),
        "oracle_dense_linear": (None, [P, i32, i32, i32, P, P, P]),
        "oracle_e4m3_value": (ctypes.c_double, [i32]),
        "oracle_mx8_block_quantize": (None, [P, i32, P, P]),
        "oracle_e4m3_encode_nonneg": (i32, [ctypes.c_double]),
        "oracle_nvfp4_global_scale": (ctypes.c_float, [ctypes.c_float]),
        "oracle_nv_block_quantize": (None, [P, i32, ctypes.c_float, P, P]),
        "oracle_nvfp4_pack": (i32, [P, i64, i64, i64, P, P, P]),
        "oracle_nvfp4_unpack": (i32, [P, P, P, i64, i64, i64, P]),
        "oracle_expert_ffn_nvfp4": (None, [P, i32, i32, i32, P, P, P, P, P, P, ctypes.c_float, ctypes.c_float,
                                           ctypes.c_float, i32, P, P, P, P]),
        "oracle_set_threads": (None, [i32]),
        "oracle_max_threads": (i32, []),
        "oracle_float_to_bf16_bits": (ctypes.c_uint16, [ctypes.c_float]),
        "oracle_bf16_bits_to_float": (ctypes.c_float, [ctypes.c_uint16]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def _ptr(a: Optional[np.ndarray]):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def set_threads(n: int) -> None:
    """Thread count of the OpenMP loops for later calls."""
    _load().oracle_set_threads(int(n))


def max_threads() -> int:
    return int(_load().oracle_max_threads())


# ------------------------------------------------------------------ scalar formats

def e2m1_value(code: int) -> float:
    return _load().oracle_e2m1_value(int(code))


def e8m0_value(s: int) -> float:
    return _load().oracle_e8m0_value(int(s))


def e2m1_encode_magnitude(a: float) -> int:
    return _load().oracle_e2m1_encode_magnitude(float(a))


def float_to_bf16_bits(f: float) -> int:
    return int(_load().oracle_float_to_bf16_bits(float(f)))


def mx_block_quantize(v: np.ndarray):
    """Quantise one block (any length) with a shared scale: returns (codes uint8[n], scale byte)."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    codes = np.zeros(v.shape[0], dtype=np.uint8)
    sb = np.zeros(1, dtype=np.uint8)
    _load().oracle_mx_block_quantize(_ptr(v), v.shape[0], _ptr(codes), _ptr(sb))
    return codes, int(sb[0])


# ------------------------------------------------------------------ MXFP4 tensors

def mxfp4_pack(w: np.ndarray):
    """fp32 [rows][K] -> (q uint8 [rows][K/2], s uint8 [rows][K/32])."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    rows, K = w.shape
    q = np.empty((rows, K // 2), dtype=np.uint8)
    s = np.empty((rows, K // 32), dtype=np.uint8)
    rc = _load().oracle_mxfp4_pack(_ptr(w), rows, K, _ptr(q), _ptr(s))
    if rc != 0:
        raise ValueError("K must be a multiple of 32")
    return q, s


def mxfp4_unpack(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.uint8)
    s = np.ascontiguousarray(s, dtype=np.uint8)
    rows, K = q.shape[0], q.shape[1] * 2
    w = np.empty((rows, K), dtype=np.float32)
    rc = _load().oracle_mxfp4_unpack(_ptr(q), _ptr(s), rows, K, _ptr(w))
    if rc != 0:
        raise ValueError("NaN scale byte (0xFF) in MXFP4 tensor")
    return w


def mx8_block_quantize(v: np.ndarray):
    """MXFP8 (reading R11) of one block: (E4M3 code bytes uint8[n], E8M0 scale byte)."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    codes = np.zeros(v.shape[0], dtype=np.uint8)
    sb = np.zeros(1, dtype=np.uint8)
    _load().oracle_mx8_block_quantize(_ptr(v), v.shape[0], _ptr(codes), _ptr(sb))
    return codes, int(sb[0])


# ------------------------------------------------------------------ NVFP4 tensors (reading R10)

def e4m3_value(code: int) -> float:
    return _load().oracle_e4m3_value(int(code))


def e4m3_encode(a: float) -> int:
    """Nearest finite non-negative E4M3 code to a >= 0 (ties even, saturating at 448)."""
    return _load().oracle_e4m3_encode_nonneg(float(a))


def nvfp4_global_scale(amax: float) -> float:
    return float(_load().oracle_nvfp4_global_scale(float(amax)))


def nv_block_quantize(v: np.ndarray, gs: float):
    """Quantise one block (fp32 values) with the global scale gs: (codes uint8[n], scale byte)."""
    v = np.ascontiguousarray(v, dtype=np.float32)
    codes = np.zeros(v.shape[0], dtype=np.uint8)
    sb = np.zeros(1, dtype=np.uint8)
    _load().oracle_nv_block_quantize(_ptr(v), v.shape[0], float(gs), _ptr(codes), _ptr(sb))
    return codes, int(sb[0])


def nvfp4_pack(w: np.ndarray):
    """fp32 [rows][K] (one matrix) or [n][rows][K] -> (q uint8 [.., rows, K/2],
    s uint8 [.., rows, K/16], gs fp32 (a scalar array for one matrix, [n] otherwise))."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    one = w.ndim == 2
    w3 = w[None] if one else w
    n, rows, K = w3.shape
    q = np.empty((n, rows, K // 2), dtype=np.uint8)
    s = np.empty((n, rows, K // 16), dtype=np.uint8)
    gs = np.empty(n, dtype=np.float32)
    rc = _load().oracle_nvfp4_pack(_ptr(w3), n, rows, K, _ptr(q), _ptr(s), _ptr(gs))
    if rc != 0:
        raise ValueError("K must be a multiple of 16")
    if one:
        return q[0], s[0], np.float32(gs[0])
    return q, s, gs


def nvfp4_unpack(q: np.ndarray, s: np.ndarray, gs) -> np.ndarray:
    """Exact fp64 values of one NVFP4 matrix (q [rows][K/2], s [rows][K/16], gs scalar) or of
    n matrices (leading axis n, gs [n])."""
    q = np.ascontiguousarray(q, dtype=np.uint8)
    s = np.ascontiguousarray(s, dtype=np.uint8)
    gs = np.ascontiguousarray(np.atleast_1d(np.asarray(gs, dtype=np.float32)))
    one = q.ndim == 2
    q3, s3 = (q[None], s[None]) if one else (q, s)
    n, rows, K = q3.shape[0], q3.shape[1], q3.shape[2] * 2
    w = np.empty((n, rows, K), dtype=np.float64)
    rc = _load().oracle_nvfp4_unpack(_ptr(q3), _ptr(s3), _ptr(gs), n, rows, K, _ptr(w))
    if rc != 0:
        raise ValueError("NaN scale byte in NVFP4 tensor")
    return w[0] if one else w


# ------------------------------------------------------------------ router / permute

def router_logits(x_bits: np.ndarray, W_r: np.ndarray, b: Optional[np.ndarray]) -> np.ndarray:
    """x_bits uint16 bf16 [T][d]; W_r fp32 [E][d]; b fp32 [E] or None -> fp32 [T][E]."""
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    W_r = np.ascontiguousarray(W_r, dtype=np.float32)
    T, d = x_bits.shape
    E = W_r.shape[0]
    out = np.empty((T, E), dtype=np.float32)
    bb = None if b is None else np.ascontiguousarray(b, dtype=np.float32)
    _load().oracle_router_logits(_ptr(x_bits), _ptr(W_r), _ptr(bb), T, d, E, _ptr(out))
    return out


def topk_softmax(logits: np.ndarray, k: int):
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    T, E = logits.shape
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float32)
    _load().oracle_topk_softmax(_ptr(logits), T, E, k, _ptr(ids), _ptr(w))
    return ids, w


def permute(ids: np.ndarray, E: int):
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    T, k = ids.shape
    counts = np.empty(E, dtype=np.int32)
    offsets = np.empty(E + 1, dtype=np.int32)
    perm_token = np.empty(T * k, dtype=np.int32)
    inv_pos = np.empty(T * k, dtype=np.int32)
    rc = _load().oracle_permute(_ptr(ids), T, E, k, _ptr(counts), _ptr(offsets), _ptr(perm_token), _ptr(inv_pos))
    if rc != 0:
        raise ValueError("expert id out of range")
    return counts, offsets, perm_token, inv_pos


# ------------------------------------------------------------------ activations / experts

def activation_rows(x_bits: np.ndarray, act_fmt: int, want_codes: bool = False):
    """Activation operand values of token rows (fp32 [n][d]); with want_codes also the
    codes/scales (ACT_MXFP4: packed nibbles [n][d/2]; ACT_MXFP8: E4M3 bytes [n][d])."""
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    n, d = x_bits.shape
    out = np.empty((n, d), dtype=np.float32)
    q = np.zeros((n, d if act_fmt == ACT_MXFP8 else d // 2), dtype=np.uint8) if want_codes else None
    s = np.zeros((n, d // 32), dtype=np.uint8) if want_codes else None
    lib = _load()
    for r in range(n):
        lib.oracle_activation_row(_ptr(x_bits[r]), d, act_fmt, _ptr(out[r]),
                                  None if q is None else _ptr(q[r]), None if s is None else _ptr(s[r]))
    if want_codes:
        return out, q, s
    return out


def expert_ffn(a: np.ndarray, wg, wu, wd, act_fmt: int, want_h: bool = False):
    """One expert on n activation rows.  wg/wu/wd are MXFP4 pairs (q, s), or NVFP4 triples
    (q, s, global scale) (reading R10), with wg/wu of shape [I][d] and wd of shape [d][I].
    Returns y [n][d] (bf16 values as fp32) and optionally (h [n][I], hq, hs)."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    n, d = a.shape
    I = wg[0].shape[0]
    assert wg[0].shape == (I, d // 2) and wu[0].shape == (I, d // 2) and wd[0].shape == (d, I // 2)
    nv = len(wg) == 3
    assert len(wu) == len(wg) and len(wd) == len(wg), "one weight format per expert"
    y = np.empty((n, d), dtype=np.float32)
    h = np.empty((n, I), dtype=np.float32) if want_h else None
    hq = np.zeros((n, I if act_fmt == ACT_MXFP8 else I // 2), dtype=np.uint8) if want_h else None
    hs = np.zeros((n, I // 32), dtype=np.uint8) if want_h else None
    ws = [np.ascontiguousarray(m[i], dtype=np.uint8) for m in (wg, wu, wd) for i in (0, 1)]
    if nv:
        _load().oracle_expert_ffn_nvfp4(_ptr(a), n, d, I, *[_ptr(m) for m in ws], float(wg[2]), float(wu[2]),
                                        float(wd[2]), act_fmt, _ptr(h), _ptr(hq), _ptr(hs), _ptr(y))
    else:
        _load().oracle_expert_ffn(_ptr(a), n, d, I, *[_ptr(m) for m in ws], act_fmt,
                                  _ptr(h), _ptr(hq), _ptr(hs), _ptr(y))
    if want_h:
        return y, (h, hq, hs)
    return y


def combine(y_perm: np.ndarray, rows: np.ndarray, w: np.ndarray, tokens: np.ndarray) -> np.ndarray:
    y_perm = np.ascontiguousarray(y_perm, dtype=np.float32)
    rows = np.ascontiguousarray(rows, dtype=np.int32)
    w = np.ascontiguousarray(w, dtype=np.float32)
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    k = w.shape[1]
    d = y_perm.shape[1]
    y = np.empty((tokens.shape[0], d), dtype=np.float32)
    _load().oracle_combine(_ptr(y_perm), _ptr(rows.reshape(-1)), _ptr(w), tokens.shape[0], _ptr(tokens), k, d, _ptr(y))
    return y


EXPERT_NORM_EPS = 1e-6


def dense_linear(x_bits: np.ndarray, W: tuple, act_fmt: int) -> np.ndarray:
    """out = a(x) W^T for bf16 rows x [n][K] and W MXFP4 (q [N][K/2], s [N][K/32]) (reading R9):
    a(x) the activation operand of R7, fp64 accumulation, rounded to fp32 then bf16."""
    q, s = W
    n, K = x_bits.shape
    N = q.shape[0]
    a = np.ascontiguousarray(activation_rows(x_bits, act_fmt), dtype=np.float32)
    out = np.empty((n, N), dtype=np.float32)
    if n:
        _load().oracle_dense_linear(_ptr(a), n, K, N, _ptr(np.ascontiguousarray(q)), _ptr(np.ascontiguousarray(s)),
                                    _ptr(out))
    return out


def expert_norm(y: np.ndarray, eps: float = EXPERT_NORM_EPS) -> np.ndarray:
    """Each row divided by its RMS over the columns, sqrt(mean(v^2) + eps) (reading R8)."""
    y = np.ascontiguousarray(y, dtype=np.float32)
    out = np.empty_like(y)
    if y.size:
        _load().oracle_expert_norm(_ptr(y), y.shape[0], y.shape[1], float(eps), _ptr(out))
    return out


# ------------------------------------------------------------------ the layer

def moe_layer(x_bits: np.ndarray, W_r: np.ndarray, b: Optional[np.ndarray], k: int,
              expert_weights: Callable[[int], Dict[str, tuple]], act_fmt: int,
              tokens: Optional[Sequence[int]] = None, want_intermediates: bool = False,
              expert_norm_eps: Optional[float] = None) -> Dict:
    """The whole layer: routing and permutation for every token, expert outputs and the
    weighted sum for ``tokens`` (all tokens when None).  With ``expert_norm_eps`` each expert
    output row is normalised (``expert_norm``) before the weighted sum.

    ``expert_weights(e)`` returns {"gate": (q, s), "up": (q, s), "down": (q, s)} for expert e
    (MXFP4 packed by this oracle's own packer; (q, s, global scale) triples for NVFP4), so only
    the experts the sampled tokens touch need to exist on the host.
    """
    T, d = x_bits.shape
    E = W_r.shape[0]
    logits = router_logits(x_bits, W_r, b)
    ids, w = topk_softmax(logits, k)
    counts, offsets, perm_token, inv_pos = permute(ids, E)
    tok = np.arange(T, dtype=np.int32) if tokens is None else np.asarray(tokens, dtype=np.int32)
    a_tok = activation_rows(x_bits[tok], act_fmt)
    # expert outputs of the sampled pairs, grouped by expert
    pair_rows = {}  # (t, j) -> row in y_sel
    y_sel_rows = []
    h_rows = {}
    by_expert: Dict[int, list] = {}
    tok_index = {int(t): n for n, t in enumerate(tok)}
    for t in tok:
        for j in range(k):
            by_expert.setdefault(int(ids[t, j]), []).append((int(t), j))
    n_rows = 0
    y_blocks = []
    for e in sorted(by_expert):
        pairs = by_expert[e]
        a = np.stack([a_tok[tok_index[t]] for (t, _) in pairs])
        wts = expert_weights(e)
        if want_intermediates:
            y_e, (h_e, hq_e, hs_e) = expert_ffn(a, wts["gate"], wts["up"], wts["down"], act_fmt, want_h=True)
        else:
            y_e = expert_ffn(a, wts["gate"], wts["up"], wts["down"], act_fmt)
        for n, (t, j) in enumerate(pairs):
            pair_rows[(t, j)] = n_rows + n
            if want_intermediates:
                h_rows[(t, j)] = (h_e[n], hq_e[n], hs_e[n])
        n_rows += len(pairs)
        y_blocks.append(y_e)
    y_perm_sel = np.concatenate(y_blocks, axis=0) if y_blocks else np.zeros((0, d), np.float32)
    rows_full = np.zeros((T, k), dtype=np.int32)
    for (t, j), r in pair_rows.items():
        rows_full[t, j] = r
    y_in = y_perm_sel if expert_norm_eps is None else expert_norm(y_perm_sel, expert_norm_eps)
    y = combine(y_in, rows_full, w, tok)
    out = dict(logits=logits, ids=ids, w=w, counts=counts, offsets=offsets, perm_token=perm_token,
               inv_pos=inv_pos, tokens=tok, y=y)
    if want_intermediates:
        out["y_perm"] = {pair: y_perm_sel[r] for pair, r in pair_rows.items()}
        out["h"] = h_rows
        out["a"] = a_tok
    return out
