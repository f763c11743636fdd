"""Shared test utilities: moving seeded inputs to the GPU and the parity criteria.

Parity criteria for y (bfloat16 GPU result vs the float64 oracle):
  * relative Frobenius error  ||y - y_ref|| / ||y_ref|| <= 5e-3
  * every element             |y - y_ref| <= 2e-2 * max|y_ref|
Derivation: the GPU rounds each dequantized weight to bfloat16 (relative 2^-9) and the output
to bfloat16 (relative 2^-9); with independent rounding errors the expected relative Frobenius
error is about 2^-9 * sqrt(1 + 1) / sqrt(3) ~ 1.6e-3 for N(0, 1) data, well inside 5e-3;
float32 accumulation over H <= 4096 adds < 1e-5.
Integer and byte outputs (codes, scales/biases bits, perm, offsets) must match exactly.
"""
import numpy as np
import torch

import workloads as wl

REL_FRO_TOL = 5e-3
ELEM_TOL = 2e-2


def to_dev_idx(idx: np.ndarray) -> torch.Tensor:
    """uint32 numpy -> int32 CUDA tensor with the same bit patterns."""
    return torch.from_numpy(np.ascontiguousarray(idx).view(np.int32)).cuda()


def parity_stats(y_gpu: torch.Tensor, y_ref: np.ndarray):
    y = y_gpu.detach().float().cpu().double().numpy().reshape(y_ref.shape)
    err = y - y_ref
    ref_norm = np.linalg.norm(y_ref)
    rel = np.linalg.norm(err) / ref_norm if ref_norm > 0 else np.linalg.norm(err)
    scale = np.abs(y_ref).max() if y_ref.size else 0.0
    elem = np.abs(err).max() / scale if scale > 0 else (np.abs(err).max() if err.size else 0.0)
    return float(rel), float(elem)


def assert_parity(y_gpu: torch.Tensor, y_ref: np.ndarray, what: str = ""):
    rel, elem = parity_stats(y_gpu, y_ref)
    assert rel <= REL_FRO_TOL, f"{what}: relative Frobenius error {rel:.3e} > {REL_FRO_TOL}"
    assert elem <= ELEM_TOL, f"{what}: max element error {elem:.3e} * max|y_ref| > {ELEM_TOL}"
    return rel, elem


def quantized_on_gpu(w_cpu_bf16: torch.Tensor):
    import quantized_moe_expert_device_gb300 as g

    return g.gqmm_quantize(w_cpu_bf16.cuda())


def np_of(t: torch.Tensor) -> np.ndarray:
    """bf16 tensors -> uint16 bit patterns; other tensors -> numpy."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return wl.bf16_bits(t)
    return t.numpy()
