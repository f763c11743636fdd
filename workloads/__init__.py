"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle checks.

This module draws random numbers and lays them out in the shapes of the
workloads the gather_qmm pages describe; it contains none of the method's
arithmetic (no quantization, no sorting, no matmul).  Every array is produced
from numpy's PCG64 generator with a fixed seed per tensor (x: 1, W: 2, idx: 3
unless a caller asks otherwise), drawn in float32 and rounded once to bfloat16
(round-to-nearest-even, through torch's dtype conversion).

Shapes follow the pages:
  * "[CUDA] gather_qmm ~24x slower ..." (ml-explore/mlx issue 4339), kernel
    microbenchmark: T=2048 tokens, A=8 active experts, H=2048, F=768, E=64,
    x of shape (T, A, 1, H), W of shape (E, F, H), idx uniform in [0, E).
  * "Pick BM from rows per expert in gather_qmm_rhs_nax" (mlx PR 4023),
    measurement paragraph: E=256, K=2048, N=512, 4 to 128 rows per expert.
  * "perf(cuda/moe): fix MoE prefill collapse" (lablup/mlxcel issue 629),
    implementation plan item 1: mixtral-8x7b at a 2048-token prompt (expert
    shape 8 x 14336 x 4096, top-2 routing).
  * "perf(cuda/quant): amortizing small-M quantized GEMM" (lablup/mlxcel issue
    725), the gap: batched decode with B in [1, 8] rows.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional

import numpy as np
import torch

SEED_X = 1
SEED_W = 2
SEED_IDX = 3


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def to_bf16(a_f32: np.ndarray) -> torch.Tensor:
    """float32 numpy array -> bfloat16 torch CPU tensor (round to nearest even)."""
    return torch.from_numpy(np.ascontiguousarray(a_f32, dtype=np.float32)).to(torch.bfloat16)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """The raw 16-bit patterns of a bfloat16 CPU tensor as a uint16 numpy array."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def normal_bf16(shape, seed: int, std: float = 1.0, chunk_rows: Optional[int] = None) -> torch.Tensor:
    """N(0, std^2) samples drawn in float32 and rounded to bfloat16.

    For large tensors the draw is made ``chunk_rows`` leading-dimension slices at a
    time from one generator stream, which keeps host memory bounded.
    """
    shape = tuple(int(s) for s in shape)
    g = _rng(seed)
    if chunk_rows is None or shape[0] <= chunk_rows:
        a = g.standard_normal(shape, dtype=np.float32)
        if std != 1.0:
            a *= np.float32(std)
        return to_bf16(a)
    out = torch.empty(shape, dtype=torch.bfloat16)
    for r0 in range(0, shape[0], chunk_rows):
        r1 = min(shape[0], r0 + chunk_rows)
        a = g.standard_normal((r1 - r0,) + shape[1:], dtype=np.float32)
        if std != 1.0:
            a *= np.float32(std)
        out[r0:r1] = to_bf16(a)
    return out


# ----------------------------------------------------------------------------------------------
# Routing index generators.  idx has shape (T, A), dtype uint32, values in [0, E).
# ----------------------------------------------------------------------------------------------

def idx_uniform(T: int, A: int, E: int, seed: int = SEED_IDX) -> np.ndarray:
    """Independent uniform draws in [0, E); duplicates within a token are allowed,
    as with the issue script's ``mx.random.randint(0, E, (T, A))``."""
    return _rng(seed).integers(0, E, size=(T, A), dtype=np.uint32)


def idx_balanced(r: int, E: int, A: int, seed: int = SEED_IDX) -> np.ndarray:
    """Exactly r rows per expert: each expert id repeated r times, shuffled, reshaped (r*E/A, A)."""
    n = r * E
    assert n % A == 0
    flat = np.repeat(np.arange(E, dtype=np.uint32), r)
    _rng(seed).shuffle(flat)
    return flat.reshape(n // A, A)


def idx_topk_distinct_uniform(T: int, A: int, E: int, seed: int = SEED_IDX) -> np.ndarray:
    """Per token, A distinct experts drawn uniformly without replacement."""
    g = _rng(seed)
    out = np.empty((T, A), dtype=np.uint32)
    for t in range(T):
        out[t] = g.choice(E, size=A, replace=False).astype(np.uint32)
    return out


def idx_zipf_topk(T: int, A: int, E: int, s: float = 1.1, seed: int = SEED_IDX) -> np.ndarray:
    """Per token, A distinct experts drawn without replacement with probability
    proportional to rank^-s, where ranks are assigned to experts by a seeded
    random permutation (unbalanced segments)."""
    g = _rng(seed)
    ranks = g.permutation(E)  # expert e has popularity rank ranks[e] (0 = most popular)
    p = (ranks + 1.0) ** (-s)
    p = p / p.sum()
    out = np.empty((T, A), dtype=np.uint32)
    for t in range(T):
        out[t] = g.choice(E, size=A, replace=False, p=p).astype(np.uint32)
    return out


# ----------------------------------------------------------------------------------------------
# Workload table.
# ----------------------------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    A: int
    H: int
    F: int
    E: int
    routing: str            # "uniform" | "balanced" | "zipf" | "topk_distinct" | "dense"
    w_std: float = 1.0
    r: int = 0              # rows per expert for "balanced"
    note: str = ""
    group_size: int = 64    # quantization group along the reduction dimension (32, 64 or 128)
    bits: int = 4           # affine code width (2, 3, 4, 5, 6 or 8)
    mode: str = "affine"    # weight format: "affine", or a block-scaled mode "mxfp4", "nvfp4", "mxfp8"
    kind: str = "gather"    # "gather": one projection, F output columns; "nn": transpose=False, W [E, H, F]
                            # quantized along F (K = H, N = F);
                            # "mlp": the expert MLP, F = intermediate width I (gate/up 2F rows, down H rows)

    @property
    def n(self) -> int:
        return self.T * self.A

    @property
    def flops(self) -> int:
        per = 6 if self.kind == "mlp" else 2  # mlp: 2*n*H*2I (gate/up) + 2*n*I*H (down)
        return per * self.T * self.A * self.H * self.F

    @property
    def out_cols(self) -> int:
        return self.H if self.kind == "mlp" else self.F


def workloads() -> Dict[str, Workload]:
    w = {}
    w["tiny"] = Workload("tiny", T=16, A=2, H=256, F=128, E=8, routing="uniform",
                         note="correctness case, sorted and unsorted")
    w["prefill_e64"] = Workload("prefill_e64", T=2048, A=8, H=2048, F=768, E=64, routing="uniform",
                                note="MoE prefill microbenchmark shape (rows/expert avg 256)")
    for gs in (32, 128):
        w[f"prefill_e64_g{gs}"] = Workload(f"prefill_e64_g{gs}", T=2048, A=8, H=2048, F=768, E=64, routing="uniform",
                                           group_size=gs, note=f"MoE prefill microbenchmark shape, {gs}-wide groups")
    for b in (2, 3, 8):
        w[f"prefill_e64_b{b}"] = Workload(f"prefill_e64_b{b}", T=2048, A=8, H=2048, F=768, E=64, routing="uniform",
                                          bits=b, note=f"MoE prefill microbenchmark shape, {b}-bit affine codes")
    for m in ("mxfp4", "nvfp4", "mxfp8"):
        w[f"prefill_e64_{m}"] = Workload(f"prefill_e64_{m}", T=2048, A=8, H=2048, F=768, E=64, routing="uniform",
                                         mode=m, group_size=16 if m == "nvfp4" else 32,
                                         note=f"MoE prefill microbenchmark shape, {m} weights")
    w["nn_e64"] = Workload("nn_e64", T=2048, A=8, H=2048, F=768, E=64, routing="uniform", kind="nn",
                           note="transpose=False gather_qmm on the MoE prefill microbenchmark shape (W[e] is [K=2048, N=768])")
    w["nn_e4"] = Workload("nn_e4", T=1024, A=1, H=512, F=512, E=4, routing="uniform", kind="nn",
                          note="transpose=False gather_qmm, E=4, K=N=512, 1024 rows (the mlx PR #4023 follow-up timing)")
    w["prefill_dense"] = Workload("prefill_dense", T=16384, A=1, H=2048, F=768, E=1, routing="dense",
                                  note="equal-FLOPs dense control x[16384,2048] x W[768,2048]^T")
    for r in (4, 8, 16, 32, 64, 128):
        w[f"sweep_r{r}"] = Workload(f"sweep_r{r}", T=32 * r, A=8, H=2048, F=512, E=256,
                                    routing="balanced", r=r,
                                    note=f"rows-per-expert sweep, exactly {r} rows per expert")
    w["mixtral"] = Workload("mixtral", T=2048, A=2, H=4096, F=14336, E=8, routing="zipf", w_std=0.02,
                            note="Mixtral-like expert shape, Zipf(1.1)-skewed top-2 routing")
    w["mlp_tiny"] = Workload("mlp_tiny", T=16, A=2, H=256, F=128, E=8, routing="uniform", kind="mlp",
                             note="expert MLP correctness case")
    w["mlp_e64"] = Workload("mlp_e64", T=2048, A=8, H=2048, F=768, E=64, routing="uniform", kind="mlp",
                            note="expert MLP (gate/up + SiLU + down) on the MoE prefill microbenchmark shape")
    w["mlp_decode_m8"] = Workload("mlp_decode_m8", T=8, A=8, H=2048, F=768, E=128, routing="topk_distinct",
                                  kind="mlp", note="expert MLP, MoE decode, 8 tokens, top-8")
    for m in (1, 2, 4, 8):
        w[f"decode_dense_m{m}"] = Workload(f"decode_dense_m{m}", T=m, A=1, H=4096, F=14336, E=1,
                                           routing="dense", note="dense decode, M rows")
        w[f"decode_moe_m{m}"] = Workload(f"decode_moe_m{m}", T=m, A=8, H=2048, F=768, E=128,
                                         routing="topk_distinct", note="MoE decode, M tokens, top-8")
    return w


def make_idx(wl: Workload, seed: int = SEED_IDX) -> Optional[np.ndarray]:
    if wl.routing == "dense":
        return None
    if wl.routing == "uniform":
        return idx_uniform(wl.T, wl.A, wl.E, seed)
    if wl.routing == "balanced":
        return idx_balanced(wl.r, wl.E, wl.A, seed)
    if wl.routing == "zipf":
        return idx_zipf_topk(wl.T, wl.A, wl.E, 1.1, seed)
    if wl.routing == "topk_distinct":
        return idx_topk_distinct_uniform(wl.T, wl.A, wl.E, seed)
    raise ValueError(wl.routing)


def make_inputs(wl: Workload, seed_x: int = SEED_X, seed_w: int = SEED_W, seed_idx: int = SEED_IDX,
                cache: Optional[dict] = None):
    """Returns dict(x=bf16 [T, A, H], w=bf16 [E, F, H], idx=uint32 [T, A] or None); for an
    "mlp" workload w_gu=bf16 [E, 2F, H] ~ N(0, 1/H) and w_dn=bf16 [E, H, F] ~ N(0, 1/F) in place
    of w, scaled so the gate pre-activations are about N(0, 1).  ``cache`` (a dict the caller
    keeps) reuses weight draws of the same shape, seed and scale across workloads."""
    def weights(shape, seed, std):
        key = (tuple(shape), seed, std)
        if cache is not None and key in cache:
            return cache[key]
        t = normal_bf16(shape, seed, std=std, chunk_rows=1)
        if cache is not None:
            cache[key] = t
        return t

    x = normal_bf16((wl.T, wl.A, wl.H), seed_x)
    if wl.kind == "nn":
        w = weights((wl.E, wl.H, wl.F), seed_w, wl.w_std)
        return dict(x=x, w=w, idx=make_idx(wl, seed_idx))
    if wl.kind == "mlp":
        w_gu = weights((wl.E, 2 * wl.F, wl.H), seed_w, wl.H ** -0.5)
        w_dn = weights((wl.E, wl.H, wl.F), seed_w + 1, wl.F ** -0.5)
        return dict(x=x, w_gu=w_gu, w_dn=w_dn, idx=make_idx(wl, seed_idx))
    w = weights((wl.E, wl.F, wl.H), seed_w, wl.w_std)
    return dict(x=x, w=w, idx=make_idx(wl, seed_idx))


def sorted_by_expert(x: torch.Tensor, idx: np.ndarray):
    """Rows of (x, idx) reordered so idx is nondecreasing (the caller-side order a
    sorted_indices=True call promises).  Returns (x_sorted [n, H], idx_sorted [n], order)
    where order[j] is the original flat row of sorted row j.  Uses numpy's stable argsort;
    this is input preparation, not the method's routing step."""
    flat = idx.reshape(-1)
    order = np.argsort(flat, kind="stable")
    xs = x.reshape(-1, x.shape[-1])[torch.from_numpy(order)]
    return xs.contiguous(), flat[order].copy(), order
