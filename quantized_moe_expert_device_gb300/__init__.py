"""Thin Python binding of libgqmm, the GB300 (sm_103a) quantized MoE gather matmul.

Every function here marshals torch tensors into the C ABI declared in include/gqmm.h
(device pointers, sizes, the current CUDA stream) and raises on a non-zero return code.
All arithmetic runs in the library's CUDA kernels; there is no fallback of any kind.  The
shared library is loaded on first use and its absence is an error.

Names follow the C ABI: gqmm_quantize, gqmm_route_sort, gqmm_gather_qmm, gqmm_moe_mlp, ...
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Tuple

import torch

__all__ = [
    "GqmmError", "library_path", "load_library", "gqmm_quantize", "gqmm_workspace_size",
    "new_workspace", "gqmm_route_sort", "gqmm_gather_qmm", "gqmm_gather_qmm_simt",
    "gqmm_moe_mlp_workspace_size", "new_mlp_workspace", "gqmm_moe_mlp", "gqmm_gather_qmm_nn", "gqmm_gather_qmm_nn_simt",
    "gqmm_device_status", "gqmm_status_string", "launch_count", "kernel_timer",
    "kernel_timer_read", "dispatch_count", "test_stall_next", "STATUS_BAD_INDEX", "STATUS_NOT_SORTED",
    "STATUS_TIMEOUT", "VARIANTS", "MAX_EXPERTS", "ACTIVATIONS", "MODES", "gqmm_quantize_fp", "gqmm_gather_qmm_fp",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libgqmm.so")
_lock = threading.Lock()
_lib = None

ERR_NAMES = {0: "OK", 1: "ERR_NULL", 2: "ERR_SHAPE", 3: "ERR_UNSUPPORTED", 4: "ERR_ALIGN",
             5: "ERR_WORKSPACE", 6: "ERR_CUDA", 7: "ERR_DEVICE"}
STATUS_BAD_INDEX = 0x100
STATUS_NOT_SORTED = 0x200
STATUS_TIMEOUT = 0x400
MAX_EXPERTS = 1024
ACTIVATIONS = {"silu": 0, "gelu": 1, "gelu_tanh": 2}  # GQMM_ACT_* of gqmm_moe_mlp
MODES = {"mxfp4": 1, "nvfp4": 2, "mxfp8": 3}  # GQMM_MODE_* of gqmm_quantize_fp / gqmm_gather_qmm_fp
MODE_BLOCK = {"mxfp4": 32, "nvfp4": 16, "mxfp8": 32}  # weights per scale byte
VARIANTS = {"route_unsorted": 0, "route_sorted": 1, "route_dense": 2, "gemm_tc": 3, "gemm_narrow": 4,
            "split_k": 5, "gemv": 6, "gemv_mma": 7, "nn": 8, "route_fused": 9}


class GqmmError(RuntimeError):
    def __init__(self, code: int, where: str, message: str):
        self.code = code
        super().__init__(f"{where}: {ERR_NAMES.get(code, code)}: {message}")


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Loads libgqmm.so (built by quantized_moe_expert_device_gb300.build)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"libgqmm.so is missing ({_LIB_PATH}); build it with "
                "`python -m quantized_moe_expert_device_gb300.build` (needs nvcc for sm_103a)")
        lib = ctypes.CDLL(_LIB_PATH)
        P, I, I64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
        sig = {
            "gqmm_quantize": ([P, I64, I64, I, I, P, P, P, P], I),
            "gqmm_workspace_size": ([I64, I, I], SZ),
            "gqmm_route_sort": ([P, I64, I, P, P, P, SZ, P], I),
            "gqmm_gather_qmm": ([P, P, P, P, P, I64, I, I, I, I, I, I, I, I, P, P, SZ, P], I),
            "gqmm_quantize_fp": ([P, I64, I64, I64, I, P, P, P, P], I),
            "gqmm_gather_qmm_fp": ([P, P, P, P, P, I64, I, I, I, I, I, I, I, P, P, SZ, P], I),
            "gqmm_gather_qmm_simt": ([P, P, P, P, P, I64, I, I, I, I, I, I, I, P, P], I),
            "gqmm_gather_qmm_nn": ([P, P, P, P, P, I64, I, I, I, I, I, I, I, I, P, P, SZ, P], I),
            "gqmm_gather_qmm_nn_simt": ([P, P, P, P, P, I64, I, I, I, I, I, I, I, P, P], I),
            "gqmm_moe_mlp_workspace_size": ([I64, I, I, I], SZ),
            "gqmm_moe_mlp": ([P, P, P, P, P, P, P, P, I64, I, I, I, I, I, I, I, I, I, P, P, SZ, P], I),
            "gqmm_device_status": ([P, P], I),
            "gqmm_status_string": ([I], ctypes.c_char_p),
            "gqmm_last_error": ([], ctypes.c_char_p),
            "gqmm_launch_count": ([], I64),
            "gqmm_kernel_timer": ([I], None),
            "gqmm_kernel_timer_read": ([ctypes.POINTER(I64), ctypes.POINTER(ctypes.c_double)], I),
            "gqmm_dispatch_count": ([I], I64),
            "gqmm_test_stall_next": ([I], None),
        }
        for name, (args, res) in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


def _check(rc: int, where: str):
    if rc != 0:
        lib = load_library()
        raise GqmmError(rc, where, lib.gqmm_last_error().decode())


def _stream(stream, device) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need(t: torch.Tensor, name: str, dtype):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must have dtype {dtype} (got {t.dtype})")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def gqmm_quantize(w: torch.Tensor, group_size: int = 64, bits: int = 4, stream=None
                  ) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """w bf16 [..., H] -> (wq uint8 [..., H*bits/8], scales bf16 [..., H/gs], biases bf16 [..., H/gs])."""
    _need(w, "w", torch.bfloat16)
    H = w.shape[-1]
    lead = tuple(w.shape[:-1])
    rows = 1
    for s in lead:
        rows *= s
    wq = torch.empty(lead + (H * bits // 8,), dtype=torch.uint8, device=w.device)
    sc = torch.empty(lead + (max(H // max(group_size, 1), 0),), dtype=torch.bfloat16, device=w.device)
    bs = torch.empty_like(sc)
    lib = load_library()
    _check(lib.gqmm_quantize(_ptr(w), rows, H, group_size, bits, _ptr(wq), _ptr(sc), _ptr(bs),
                             _stream(stream, w.device)), "gqmm_quantize")
    return wq, sc, bs


def gqmm_quantize_fp(w: torch.Tensor, mode: str, stream=None):
    """Block-scaled floating-point quantization of w bf16 [E, F, H] (or [F, H]): mode "mxfp4",
    "nvfp4" or "mxfp8".  Returns (wq uint8 [..., H/2] or [..., H] (mxfp8), scales uint8
    [..., H/32] or [..., H/16] (nvfp4), tscale float32 [E] for nvfp4 (one per expert) or None)."""
    _need(w, "w", torch.bfloat16)
    if mode not in MODES:
        raise ValueError(f"mode must be one of {sorted(MODES)}, got {mode!r}")
    H = w.shape[-1]
    lead = tuple(w.shape[:-1])
    rows = 1
    for s_ in lead:
        rows *= s_
    per_tensor = lead[-1] if len(lead) >= 2 else rows
    wq = torch.empty(lead + ((H if mode == "mxfp8" else H // 2),), dtype=torch.uint8, device=w.device)
    sc = torch.empty(lead + (H // MODE_BLOCK[mode],), dtype=torch.uint8, device=w.device)
    ts = torch.empty(max(rows // max(per_tensor, 1), 1), dtype=torch.float32, device=w.device) if mode == "nvfp4" else None
    lib = load_library()
    _check(lib.gqmm_quantize_fp(_ptr(w), rows, H, per_tensor, MODES[mode], _ptr(wq), _ptr(sc), _ptr(ts),
                                _stream(stream, w.device)), "gqmm_quantize_fp")
    return wq, sc, ts


def gqmm_gather_qmm_fp(x: torch.Tensor, wq: torch.Tensor, scales: torch.Tensor, tscale: Optional[torch.Tensor],
                       idx: Optional[torch.Tensor], mode: str, sorted_indices: bool = False,
                       y: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """gqmm_gather_qmm on weights quantized by gqmm_quantize_fp (mode "mxfp4", "nvfp4" or "mxfp8");
    x, idx and the result as for gqmm_gather_qmm."""
    _need(x, "x", torch.bfloat16)
    _need(wq, "wq", torch.uint8)
    _need(scales, "scales", torch.uint8)
    if mode not in MODES:
        raise ValueError(f"mode must be one of {sorted(MODES)}, got {mode!r}")
    if tscale is not None:
        _need(tscale, "tscale", torch.float32)
    if idx is not None and (not idx.is_cuda or not idx.is_contiguous() or idx.element_size() != 4):
        raise ValueError("idx must be a contiguous 32-bit CUDA tensor")
    T, A, H, F, E = _gather_shapes(x, idx, wq)
    if y is None:
        y = torch.empty(_out_shape(x, T, A, F), dtype=torch.bfloat16, device=x.device)
    else:
        _need(y, "y", torch.bfloat16)
    if ws is None:
        ws = new_workspace(T * A, F, E, x.device)
    lib = load_library()
    _check(lib.gqmm_gather_qmm_fp(_ptr(x), _ptr(wq), _ptr(scales), _ptr(tscale), _ptr(idx), T, A, H, F, E, MODES[mode],
                                  1 if sorted_indices else 0, _x_shared(x, T, A, H), _ptr(y), _ptr(ws), ws.numel(),
                                  _stream(stream, x.device)), "gqmm_gather_qmm_fp")
    return y


def gqmm_workspace_size(n: int, F: int, E: int) -> int:
    return int(load_library().gqmm_workspace_size(n, F, E))


def new_workspace(n, F: int, E: int, device="cuda") -> torch.Tensor:
    """A zero-filled workspace of the size gqmm_workspace_size asks for.  n may be a list of
    row counts the workspace will serve; it is then sized for the largest need among them
    (the size is not monotone in n: decode-sized calls add split-K partial-sum planes)."""
    ns = list(n) if isinstance(n, (list, tuple)) else [n]
    sizes = [gqmm_workspace_size(int(k), F, E) for k in ns]
    size = max(sizes) if sizes else 0
    if not sizes or min(sizes) == 0:
        raise ValueError(f"no workspace size for n={n}, F={F}, E={E}")
    return torch.zeros(size, dtype=torch.uint8, device=device)


def gqmm_route_sort(idx: torch.Tensor, E: int, ws: Optional[torch.Tensor] = None, stream=None
                    ) -> Tuple[torch.Tensor, torch.Tensor]:
    """idx uint32 (or int32 holding the same bits) [...] -> (perm int32 [n], offsets int32 [E+1])."""
    if idx.dtype not in (torch.int32, getattr(torch, "uint32", torch.int32)):
        raise TypeError("idx must be int32/uint32")
    if not idx.is_cuda or not idx.is_contiguous():
        raise ValueError("idx must be a contiguous CUDA tensor")
    n = idx.numel()
    if ws is None:
        ws = new_workspace(n, 1, E, idx.device)
    perm = torch.empty(max(n, 1), dtype=torch.int32, device=idx.device)[:n]
    offsets = torch.empty(E + 1, dtype=torch.int32, device=idx.device)
    lib = load_library()
    _check(lib.gqmm_route_sort(_ptr(idx), n, E, _ptr(perm) if n else _ptr(offsets), _ptr(offsets), _ptr(ws),
                               ws.numel(), _stream(stream, idx.device)), "gqmm_route_sort")
    return perm, offsets


def _check_groups(scales: torch.Tensor, K: int, group_size: int, name: str):
    if group_size <= 0 or scales.shape[-1] * group_size != K:
        raise ValueError(f"{name} has {scales.shape[-1]} groups per row; K={K} with group_size={group_size} "
                         f"needs {K // max(group_size, 1)}")


def _gather_shapes(x: torch.Tensor, idx: Optional[torch.Tensor], wq: torch.Tensor):
    H = x.shape[-1]
    if idx is None:
        T, A = x.numel() // H, 1
    elif idx.dim() >= 2:
        T, A = idx.shape[0], idx.numel() // idx.shape[0]
    else:
        T, A = idx.numel(), 1
    if T * A * H != x.numel() and not (idx is not None and T * H == x.numel()):
        raise ValueError(f"x has {x.numel()} elements, expected T*A*H = {T}*{A}*{H} (or T*H, shared by the A rows)")
    E, F = wq.shape[0], wq.shape[1]
    return T, A, H, F, E


def _x_shared(x: torch.Tensor, T: int, A: int, H: int) -> int:
    """1 when x holds one row per token for its A routed rows ([T, H] or [T, 1, H])."""
    return 1 if A > 1 and x.numel() == T * H else 0


def _out_shape(x: torch.Tensor, T: int, A: int, cols: int):
    return (T, A, cols) if _x_shared(x, T, A, x.shape[-1]) else tuple(x.shape[:-1]) + (cols,)


def gqmm_gather_qmm(x: torch.Tensor, wq: torch.Tensor, scales: torch.Tensor, biases: torch.Tensor,
                    idx: Optional[torch.Tensor], group_size: int = 64, bits: int = 4,
                    sorted_indices: bool = False, y: Optional[torch.Tensor] = None,
                    ws: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """y[t, a, :] = x[t, a, :] . deq(W[idx[t, a]])^T.

    x bf16 [T, A, H] (or [T, A, 1, H], or [n, H]); wq uint8 [E, F, H*bits/8]; scales/biases bf16
    [E, F, H/group_size] (4-bit codes with group_size 32, 64 or 128; 2-, 3-, 5-, 6- or 8-bit codes with
    group_size 64); idx uint32/int32 [T, A] or None (dense, E == 1).  Returns y bf16 with x's leading
    shape and last dimension F.
    """
    _need(x, "x", torch.bfloat16)
    _need(wq, "wq", torch.uint8)
    _need(scales, "scales", torch.bfloat16)
    _need(biases, "biases", torch.bfloat16)
    if idx is not None and (not idx.is_cuda or not idx.is_contiguous() or idx.element_size() != 4):
        raise ValueError("idx must be a contiguous 32-bit CUDA tensor")
    T, A, H, F, E = _gather_shapes(x, idx, wq)
    _check_groups(scales, H, group_size, "scales")
    if y is None:
        y = torch.empty(_out_shape(x, T, A, F), dtype=torch.bfloat16, device=x.device)
    else:
        _need(y, "y", torch.bfloat16)
    if ws is None:
        ws = new_workspace(T * A, F, E, x.device)
    lib = load_library()
    _check(lib.gqmm_gather_qmm(_ptr(x), _ptr(wq), _ptr(scales), _ptr(biases), _ptr(idx), T, A, H, F, E,
                               group_size, bits, 1 if sorted_indices else 0, _x_shared(x, T, A, H), _ptr(y), _ptr(ws),
                               ws.numel(),
                               _stream(stream, x.device)), "gqmm_gather_qmm")
    return y


def gqmm_gather_qmm_simt(x, wq, scales, biases, idx, group_size: int = 64, bits: int = 4,
                         y: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """CUDA-core cross-check of gqmm_gather_qmm (same arguments, no workspace)."""
    _need(x, "x", torch.bfloat16)
    T, A, H, F, E = _gather_shapes(x, idx, wq)
    _check_groups(scales, H, group_size, "scales")
    if y is None:
        y = torch.empty(_out_shape(x, T, A, F), dtype=torch.bfloat16, device=x.device)
    lib = load_library()
    _check(lib.gqmm_gather_qmm_simt(_ptr(x), _ptr(wq), _ptr(scales), _ptr(biases), _ptr(idx), T, A, H, F, E,
                                    group_size, bits, _x_shared(x, T, A, H), _ptr(y), _stream(stream, x.device)),
           "gqmm_gather_qmm_simt")
    return y


def _nn_shapes(x: torch.Tensor, wq: torch.Tensor, scales: torch.Tensor, idx: Optional[torch.Tensor],
               group_size: int):
    _need(x, "x", torch.bfloat16)
    if idx is not None and (not idx.is_cuda or not idx.is_contiguous() or idx.element_size() != 4):
        raise ValueError("idx must be a contiguous 32-bit CUDA tensor")
    K = x.shape[-1]
    if wq.dim() != 3 or wq.shape[1] != K:
        raise ValueError(f"wq must be [E, K, N/2] with K = {K}, got {tuple(wq.shape)}")
    E, N = wq.shape[0], wq.shape[2] * 2
    _check_groups(scales, N, group_size, "scales")
    T, A, _, _, _ = _gather_shapes(x, idx, wq)
    return T, A, K, N, E


def gqmm_gather_qmm_nn(x: torch.Tensor, wq: torch.Tensor, scales: torch.Tensor, biases: torch.Tensor,
                       idx: Optional[torch.Tensor], group_size: int = 64, bits: int = 4,
                       sorted_indices: bool = False, y: Optional[torch.Tensor] = None,
                       ws: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """gather_qmm with transpose=False: y[t, a, :] = x[t, a, :] . deq(W[idx[t, a]]), W[e] [K, N]
    quantized along N.  x bf16 [T, A, K] (or [T, K], shared by the A rows, or [n, K]); wq uint8
    [E, K, N/2] and scales/biases [E, K, N/group_size], as gqmm_quantize writes for an [E, K, N]
    weight; idx, sorted_indices and ws as for gqmm_gather_qmm (the workspace sized for N output
    columns).  Returns y bf16 [..., N]."""
    T, A, K, N, E = _nn_shapes(x, wq, scales, idx, group_size)
    _need(wq, "wq", torch.uint8)
    _need(scales, "scales", torch.bfloat16)
    _need(biases, "biases", torch.bfloat16)
    if y is None:
        y = torch.empty(_out_shape(x, T, A, N), dtype=torch.bfloat16, device=x.device)
    else:
        _need(y, "y", torch.bfloat16)
    if ws is None:
        ws = new_workspace(T * A, N, E, x.device)
    lib = load_library()
    _check(lib.gqmm_gather_qmm_nn(_ptr(x), _ptr(wq), _ptr(scales), _ptr(biases), _ptr(idx), T, A, K, N, E,
                                  group_size, bits, 1 if sorted_indices else 0, _x_shared(x, T, A, K), _ptr(y),
                                  _ptr(ws), ws.numel(), _stream(stream, x.device)), "gqmm_gather_qmm_nn")
    return y


def gqmm_gather_qmm_nn_simt(x: torch.Tensor, wq: torch.Tensor, scales: torch.Tensor, biases: torch.Tensor,
                            idx: Optional[torch.Tensor], group_size: int = 64, bits: int = 4,
                            y: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """CUDA-core cross-check of gqmm_gather_qmm_nn (same arguments, no workspace; any K >= 1)."""
    T, A, K, N, E = _nn_shapes(x, wq, scales, idx, group_size)
    if y is None:
        y = torch.empty(_out_shape(x, T, A, N), dtype=torch.bfloat16, device=x.device)
    lib = load_library()
    _check(lib.gqmm_gather_qmm_nn_simt(_ptr(x), _ptr(wq), _ptr(scales), _ptr(biases), _ptr(idx), T, A, K, N, E,
                                       group_size, bits, _x_shared(x, T, A, K), _ptr(y), _stream(stream, x.device)),
           "gqmm_gather_qmm_nn_simt")
    return y


def gqmm_moe_mlp_workspace_size(n: int, H: int, I: int, E: int) -> int:
    return int(load_library().gqmm_moe_mlp_workspace_size(n, H, I, E))


def new_mlp_workspace(n: int, H: int, I: int, E: int, device="cuda") -> torch.Tensor:
    """A zero-filled workspace of the size gqmm_moe_mlp_workspace_size asks for."""
    size = gqmm_moe_mlp_workspace_size(int(n), H, I, E)
    if size == 0:
        raise ValueError(f"no MLP workspace size for n={n}, H={H}, I={I}, E={E}")
    return torch.zeros(size, dtype=torch.uint8, device=device)


def gqmm_moe_mlp(x: torch.Tensor, q_gu, q_dn, idx: Optional[torch.Tensor], group_size: int = 64, bits: int = 4,
                 sorted_indices: bool = False, y: Optional[torch.Tensor] = None,
                 ws: Optional[torch.Tensor] = None, stream=None, activation: str = "silu") -> torch.Tensor:
    """The MoE expert MLP: y[t, a] = W_dn[e] (act(W_g[e] x[t, a]) * (W_u[e] x[t, a])), e = idx[t, a],
    act one of ACTIVATIONS: "silu" (SwiGLU), "gelu" (GeGLU) or "gelu_tanh" (GeGLU, tanh form).

    x bf16 [T, A, H] (or [n, H]); q_gu = (wq, scales, biases) of W_gu = [W_gate; W_up]
    [E, 2I, H]; q_dn the same for W_dn [E, H, I]; idx as for gqmm_gather_qmm.  Returns y
    bf16 with x's shape.
    """
    if activation not in ACTIVATIONS:
        raise ValueError(f"activation must be one of {sorted(ACTIVATIONS)}, got {activation!r}")
    wq_gu, sc_gu, bs_gu = q_gu
    wq_dn, sc_dn, bs_dn = q_dn
    _need(x, "x", torch.bfloat16)
    for t, name, dt in ((wq_gu, "wq_gu", torch.uint8), (sc_gu, "sc_gu", torch.bfloat16), (bs_gu, "bs_gu", torch.bfloat16),
                        (wq_dn, "wq_dn", torch.uint8), (sc_dn, "sc_dn", torch.bfloat16), (bs_dn, "bs_dn", torch.bfloat16)):
        _need(t, name, dt)
    if idx is not None and (not idx.is_cuda or not idx.is_contiguous() or idx.element_size() != 4):
        raise ValueError("idx must be a contiguous 32-bit CUDA tensor")
    T, A, H, I2, E = _gather_shapes(x, idx, wq_gu)
    I = I2 // 2
    if tuple(wq_dn.shape[:2]) != (E, H) or wq_dn.shape[2] * 2 != I:
        raise ValueError(f"wq_dn must be [E, H, I/2] = [{E}, {H}, {I // 2}], got {tuple(wq_dn.shape)}")
    _check_groups(sc_gu, H, group_size, "sc_gu")
    _check_groups(sc_dn, I, group_size, "sc_dn")
    if y is None:
        y = torch.empty(_out_shape(x, T, A, H), dtype=torch.bfloat16, device=x.device)
    else:
        _need(y, "y", torch.bfloat16)
    if ws is None:
        ws = new_mlp_workspace(T * A, H, I, E, x.device)
    lib = load_library()
    _check(lib.gqmm_moe_mlp(_ptr(x), _ptr(wq_gu), _ptr(sc_gu), _ptr(bs_gu), _ptr(wq_dn), _ptr(sc_dn), _ptr(bs_dn),
                            _ptr(idx), T, A, H, I, E, group_size, bits, ACTIVATIONS[activation],
                            1 if sorted_indices else 0, _x_shared(x, T, A, H), _ptr(y), _ptr(ws),
                            ws.numel(), _stream(stream, x.device)), "gqmm_moe_mlp")
    return y


def gqmm_device_status(ws: torch.Tensor, stream=None) -> int:
    """Synchronizes the stream, returns and clears the device status bits in ws."""
    lib = load_library()
    rc = lib.gqmm_device_status(_ptr(ws), _stream(stream, ws.device))
    if rc < 0:
        _check(-rc, "gqmm_device_status")
    return rc


def gqmm_status_string(code: int) -> str:
    return load_library().gqmm_status_string(code).decode()


def launch_count() -> int:
    return int(load_library().gqmm_launch_count())


def kernel_timer(capacity: int) -> None:
    """capacity > 0: time the next `capacity` grouped-GEMM launches; 0: stop."""
    load_library().gqmm_kernel_timer(int(capacity))


def kernel_timer_read() -> Tuple[int, float]:
    n = ctypes.c_int64(0)
    ms = ctypes.c_double(0.0)
    _check(load_library().gqmm_kernel_timer_read(ctypes.byref(n), ctypes.byref(ms)), "gqmm_kernel_timer_read")
    return int(n.value), float(ms.value)


def test_stall_next(n: int) -> None:
    """Failure-path test hook: the next n tensor-core GEMM launches time out (GQMM_STATUS_TIMEOUT)
    and unwind instead of computing."""
    load_library().gqmm_test_stall_next(int(n))


def dispatch_count(variant: str) -> int:
    return int(load_library().gqmm_dispatch_count(VARIANTS[variant]))
