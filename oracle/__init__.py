"""Python access to the CPU oracle (``gqmm_oracle.c``).

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the benchmark's
CPU-baseline / reference leg are the only callers.  The product package never imports
this module.  The oracle follows the pages' statement of the quantized MoE gather matmul;
the C file's header lists each step and the passage it follows.

Arrays cross the boundary as numpy arrays: bfloat16 tensors as their raw uint16 bit
patterns, indices as uint32, results as float64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gqmm_oracle.c")
_LIB = os.path.join(_HERE, "libgqmm_oracle.so")
_lock = threading.Lock()
_lib = None

# -O2 for speed, but no fast-math and no floating-point contraction, so every operation
# is the IEEE operation the C source spells out.
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off", "-fno-fast-math"]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (a second of work); returns the library path."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            I64 = ctypes.c_int64
            I = ctypes.c_int
            lib.oracle_nthreads_default.restype = I
            lib.oracle_quantize.argtypes = [P, I64, I64, I, I, P, P, P, I]
            lib.oracle_quantize.restype = I
            lib.oracle_dequantize.argtypes = [P, P, P, I64, I64, I, I, P]
            lib.oracle_dequantize.restype = I
            lib.oracle_quantize_fp.argtypes = [P, I64, I64, I, I64, P, P, P]
            lib.oracle_quantize_fp.restype = I
            lib.oracle_dequantize_fp.argtypes = [P, P, P, I64, I64, I, I64, P]
            lib.oracle_dequantize_fp.restype = I
            lib.oracle_gather_qmm_fp.argtypes = [P, P, P, P, P, I64, I64, I64, I64, I, P, I64, P, I]
            lib.oracle_gather_qmm_fp.restype = I
            lib.oracle_route_sort.argtypes = [P, I64, I, P, P]
            lib.oracle_route_sort.restype = I64
            lib.oracle_gather_qmm.argtypes = [P, P, P, P, P, I64, I64, I64, I64, I, I, P, I]
            lib.oracle_gather_qmm.restype = I
            lib.oracle_gather_qmm_rows.argtypes = [P, P, P, P, P, I64, I64, I64, I, I, P, I64, P, I]
            lib.oracle_gather_qmm_rows.restype = I
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _u16(a) -> np.ndarray:
    """Accepts a uint16 numpy array or a bfloat16 torch CPU tensor."""
    if isinstance(a, np.ndarray):
        assert a.dtype == np.uint16
        return np.ascontiguousarray(a)
    import torch  # only for the dtype view

    assert a.dtype == torch.bfloat16
    return a.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def nthreads_default() -> int:
    return int(_load().oracle_nthreads_default())


# the block-scaled floating-point modes of oracle_quantize_fp (the affine format is mode 0)
MODES = {"affine": 0, "mxfp4": 1, "nvfp4": 2, "mxfp8": 3}
# weights per shared scale, and code bytes per weight, of each floating-point mode
MODE_BLOCK = {"mxfp4": 32, "nvfp4": 16, "mxfp8": 32}
MODE_CODE_BYTES = {"mxfp4": 0.5, "nvfp4": 0.5, "mxfp8": 1.0}


def quantize(w, group_size: int = 64, bits: int = 4, nthreads: int = 0):
    """w: bf16 [..., H] -> (wq u8 [..., H*bits/8], scales u16 [..., H/gs], biases u16 [..., H/gs])."""
    w16 = _u16(w)
    H = w16.shape[-1]
    lead = w16.shape[:-1]
    rows = int(np.prod(lead)) if lead else 1
    if H % group_size or group_size % 8:
        raise ValueError("H must be a multiple of group_size")
    wq = np.empty(lead + (H * bits // 8,), np.uint8)
    sc = np.empty(lead + (H // group_size,), np.uint16)
    bs = np.empty(lead + (H // group_size,), np.uint16)
    rc = _load().oracle_quantize(_ptr(w16), rows, H, group_size, bits, _ptr(wq), _ptr(sc), _ptr(bs), nthreads)
    if rc != 0:
        raise ValueError("oracle_quantize rejected its arguments")
    return wq, sc, bs


def dequantize(wq: np.ndarray, scales: np.ndarray, biases: np.ndarray, group_size: int = 64,
               bits: int = 4) -> np.ndarray:
    """-> float64 [..., H] with H = wq.shape[-1] * 8 / bits."""
    wq = np.ascontiguousarray(wq, np.uint8)
    scales = _u16(scales)
    biases = _u16(biases)
    H = wq.shape[-1] * 8 // bits
    rows = int(np.prod(wq.shape[:-1])) if wq.ndim > 1 else 1
    out = np.empty(wq.shape[:-1] + (H,), np.float64)
    rc = _load().oracle_dequantize(_ptr(wq), _ptr(scales), _ptr(biases), rows, H, group_size, bits, _ptr(out))
    if rc != 0:
        raise ValueError("oracle_dequantize rejected its arguments")
    return out


def quantize_fp(w, mode: str):
    """Block-scaled floating-point quantization of w: bf16 [..., H] (an [E, F, H] stack: each
    expert is one nvfp4 tensor; a 2-D [F, H] weight is one tensor).  Returns (wq u8 [..., H/2]
    (mxfp4, nvfp4) or [..., H] (mxfp8), scales u8 [..., H/32] or [..., H/16] (nvfp4), tensor
    scales float32 [E] (nvfp4; None otherwise))."""
    w16 = _u16(w)
    H = w16.shape[-1]
    lead = w16.shape[:-1]
    rows = int(np.prod(lead)) if lead else 1
    per_tensor = int(lead[-1]) if len(lead) >= 2 else rows
    nb = MODE_BLOCK[mode]
    wq = np.empty(lead + (int(H * MODE_CODE_BYTES[mode]),), np.uint8)
    sc = np.empty(lead + (H // nb,), np.uint8)
    ts = np.empty(max(rows // max(per_tensor, 1), 1), np.float32) if mode == "nvfp4" else None
    rc = _load().oracle_quantize_fp(_ptr(w16), rows, H, MODES[mode], per_tensor, _ptr(wq), _ptr(sc),
                                    None if ts is None else _ptr(ts))
    if rc != 0:
        raise ValueError("oracle_quantize_fp rejected its arguments")
    return wq, sc, ts


def dequantize_fp(wq: np.ndarray, scales: np.ndarray, tscale, mode: str) -> np.ndarray:
    """-> float64 [..., H]; the nvfp4 tensor scales apply per expert (per leading-dimension
    slice of an [E, F, ...] stack)."""
    wq = np.ascontiguousarray(wq, np.uint8)
    scales = np.ascontiguousarray(scales, np.uint8)
    H = int(wq.shape[-1] / MODE_CODE_BYTES[mode])
    lead = wq.shape[:-1]
    rows = int(np.prod(lead)) if lead else 1
    per_tensor = int(lead[-1]) if len(lead) >= 2 else rows
    out = np.empty(lead + (H,), np.float64)
    ts = None if tscale is None else np.ascontiguousarray(tscale, np.float32)
    rc = _load().oracle_dequantize_fp(_ptr(wq), _ptr(scales), None if ts is None else _ptr(ts), rows, H, MODES[mode],
                                      per_tensor, _ptr(out))
    if rc != 0:
        raise ValueError("oracle_dequantize_fp rejected its arguments")
    return out


def gather_qmm_fp(x, wq, scales, tscale, idx, E: int, mode: str, nthreads: int = 0, rows=None):
    """gather_qmm on weights in a floating-point mode (as quantize_fp writes them for [E, F, H]),
    float64.  Returns [n, F] (or [len(rows), F])."""
    x16 = _u16(x)
    H = x16.shape[-1]
    x16 = x16.reshape(-1, H)
    n = x16.shape[0]
    wq = np.ascontiguousarray(wq, np.uint8)
    scales = np.ascontiguousarray(scales, np.uint8)
    F = wq.shape[-2]
    if int(wq.shape[-1] / MODE_CODE_BYTES[mode]) != H:
        raise ValueError("wq does not match H")
    ts = None if tscale is None else np.ascontiguousarray(tscale, np.float32)
    idx_p = None
    if idx is not None:
        flat = np.ascontiguousarray(np.asarray(idx, np.uint32).reshape(-1))
        if flat.size != n:
            raise ValueError("idx must have one entry per row of x")
        idx_p = _ptr(flat)
    r = None if rows is None else np.ascontiguousarray(np.asarray(rows, np.int64))
    y = np.empty(((n if r is None else r.size), F), np.float64)
    used = _load().oracle_gather_qmm_fp(_ptr(x16), _ptr(wq), _ptr(scales), None if ts is None else _ptr(ts), idx_p, n,
                                        H, F, E, MODES[mode], None if r is None else _ptr(r),
                                        0 if r is None else r.size, _ptr(y), nthreads)
    if used < 0:
        raise ValueError("oracle_gather_qmm_fp rejected its arguments")
    return y


def route_sort(idx: np.ndarray, E: int):
    """idx: uint32 [...] -> (perm int32 [n], offsets int32 [E+1], n_bad)."""
    flat = np.ascontiguousarray(np.asarray(idx, np.uint32).reshape(-1))
    n = flat.size
    perm = np.empty(n, np.int32)
    offsets = np.empty(E + 1, np.int32)
    bad = _load().oracle_route_sort(_ptr(flat), n, E, _ptr(perm), _ptr(offsets))
    if bad < 0:
        raise ValueError("oracle_route_sort rejected its arguments")
    return perm, offsets, int(bad)


def gather_qmm(x, wq, scales, biases, idx, E: int, group_size: int = 64, bits: int = 4,
               nthreads: int = 0, rows=None):
    """x: bf16 [..., H] (flattened to n rows); wq u8 [E, F, H/2]; scales/biases [E, F, H/gs];
    idx: uint32 [...] with n entries, or None for the dense case (E == 1).
    Returns float64 [n, F] (or [len(rows), F] when ``rows`` lists flat rows)."""
    x16 = _u16(x)
    H = x16.shape[-1]
    x16 = x16.reshape(-1, H)
    n = x16.shape[0]
    wq = np.ascontiguousarray(wq, np.uint8)
    scales = _u16(scales)
    biases = _u16(biases)
    F = wq.shape[-2]
    if wq.shape[-1] * 8 != H * bits:
        raise ValueError("wq last dim must be H*bits/8")
    idx_p = None
    if idx is not None:
        flat = np.ascontiguousarray(np.asarray(idx, np.uint32).reshape(-1))
        if flat.size != n:
            raise ValueError("idx must have one entry per row of x")
        idx_p = _ptr(flat)
    lib = _load()
    if rows is None:
        y = np.empty((n, F), np.float64)
        used = lib.oracle_gather_qmm(_ptr(x16), _ptr(wq), _ptr(scales), _ptr(biases), idx_p,
                                     n, H, F, E, group_size, bits, _ptr(y), nthreads)
    else:
        r = np.ascontiguousarray(np.asarray(rows, np.int64))
        y = np.empty((r.size, F), np.float64)
        used = lib.oracle_gather_qmm_rows(_ptr(x16), _ptr(wq), _ptr(scales), _ptr(biases), idx_p,
                                          H, F, E, group_size, bits, _ptr(r), r.size, _ptr(y), nthreads)
    if used < 0:
        raise ValueError("oracle_gather_qmm rejected its arguments")
    gather_qmm.last_threads = int(used)
    return y


gather_qmm.last_threads = 0


def gather_qmm_nn(x, wq, scales, biases, idx, E: int, group_size: int = 64, rows=None):
    """gather_qmm with transpose=False, in float64: y[i] = x[i] . deq(W[e]), e = idx[i], where W[e]
    is [K, N] quantized along N (the layout mx.quantize gives a [E, K, N] weight: wq u8
    [E, K, N/2], scales/biases [E, K, N/gs]).  x: bf16 [..., K] (n rows); idx None for E == 1.
    Rows whose index is >= E are zero.  Returns float64 [n, N] (or [len(rows), N])."""
    x16 = _u16(x)
    K = x16.shape[-1]
    xf = (x16.reshape(-1, K).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    n = xf.shape[0]
    r = np.arange(n) if rows is None else np.asarray(rows, np.int64)
    e = np.zeros(r.size, np.int64) if idx is None else np.asarray(idx, np.uint32).reshape(-1)[r].astype(np.int64)
    wq = np.asarray(wq)
    N = wq.shape[-1] * 2
    y = np.zeros((r.size, N), np.float64)
    for ex in np.unique(e):
        if ex >= E:
            continue
        w_hat = dequantize(wq[ex], _u16(scales)[ex], _u16(biases)[ex], group_size)  # [K, N]
        for i in np.nonzero(e == ex)[0]:  # one vector-matrix product per row
            y[i] = xf[r[i]] @ w_hat
    return y


def silu(v: np.ndarray) -> np.ndarray:
    """SiLU in float64: v / (1 + exp(-v))."""
    return v / (1.0 + np.exp(-v))


def gelu(v: np.ndarray) -> np.ndarray:
    """GELU in float64 by its definition v * Phi(v) = v/2 * (1 + erf(v / sqrt 2)) (Hendrycks and
    Gimpel, "Gaussian Error Linear Units"), the gate of GeGLU (Shazeer, "GLU Variants Improve
    Transformer")."""
    from scipy.special import erf

    return 0.5 * v * (1.0 + erf(v / np.sqrt(2.0)))


def gelu_tanh(v: np.ndarray) -> np.ndarray:
    """The tanh form of GELU from the same paper, in float64:
    v/2 * (1 + tanh(sqrt(2/pi) * (v + 0.044715 v^3)))."""
    return 0.5 * v * (1.0 + np.tanh(np.sqrt(2.0 / np.pi) * (v + 0.044715 * v ** 3)))


# gate activations of the expert MLP, by the name the binding uses
ACTIVATIONS = {"silu": silu, "gelu": gelu, "gelu_tanh": gelu_tanh}


def moe_mlp(x, q_gu, q_dn, idx, E: int, group_size: int = 64, bits: int = 4, nthreads: int = 0, rows=None,
            activation: str = "silu"):
    """The MoE expert MLP on the routed rows, in float64:
    y[i] = W_dn[e] (act(W_g[e] x[i]) * (W_u[e] x[i])), e = idx[i], with W_gu[e] = [W_g[e]; W_u[e]]
    (gate rows 0 .. I-1, up rows I .. 2I-1) and every weight dequantized from its 4-bit codes;
    act is SiLU (SwiGLU), GELU (GeGLU) or GELU's tanh form, by ``activation``.
    q_gu = (wq, scales, biases) for W_gu [E, 2I, H]; q_dn the same for W_dn [E, H, I].
    Rows whose index is >= E are zero.  Returns float64 [n, H] (or [len(rows), H])."""
    wq_gu, sc_gu, bs_gu = q_gu
    wq_dn, sc_dn, bs_dn = q_dn
    I2 = np.asarray(wq_gu).shape[-2]
    I = I2 // 2
    gu = gather_qmm(x, wq_gu, sc_gu, bs_gu, idx, E, group_size, bits, nthreads, rows)  # [m, 2I]
    h = ACTIVATIONS[activation](gu[:, :I]) * gu[:, I:]
    x16 = _u16(x)
    n = x16.reshape(-1, x16.shape[-1]).shape[0]
    r = np.arange(n) if rows is None else np.asarray(rows, np.int64)
    e = np.zeros(r.size, np.int64) if idx is None else np.asarray(idx, np.uint32).reshape(-1)[r].astype(np.int64)
    H_out = np.asarray(wq_dn).shape[-2]
    y = np.zeros((r.size, H_out), np.float64)
    for ex in np.unique(e):
        if ex >= E:
            continue
        sel = np.nonzero(e == ex)[0]
        w_dn = dequantize(np.asarray(wq_dn)[ex], _u16(sc_dn)[ex], _u16(bs_dn)[ex], group_size)  # [H, I]
        for i in sel:  # one matrix-vector product per row: a row's result depends on that row only
            y[i] = w_dn @ h[i]
    return y
