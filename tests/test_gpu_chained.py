"""Calls chained on one stream: a call must see every result the calls before it on the stream
wrote, even though the library's kernels start early (programmatic dependent launch) and
overlap their predecessors' tails.

Each case runs its chain many times on fresh, zero-filled buffers, so a kernel that copied its
input before the previous kernel had written it would read zeros and show up as a result that
differs between iterations or from the oracle.  Every iteration must give the same bits (the
kernels are deterministic), and the result must match the float64 oracle within the parity
tolerances.  The oracle's inputs are its own: where a chained call reads the output of an earlier
call, the oracle reads its own float64 result of that earlier call, rounded to bfloat16.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import assert_parity, to_dev_idx

pytestmark = pytest.mark.gpu

ITERS = 50


def _dev_q(q):
    wq, sc, bs = q
    return (torch.from_numpy(wq).cuda(), torch.from_numpy(sc.view(np.int16)).cuda().view(torch.bfloat16),
            torch.from_numpy(bs.view(np.int16)).cuda().view(torch.bfloat16))


def _bf16_of(y_ref: np.ndarray) -> torch.Tensor:
    """float64 oracle result -> bfloat16 (float32 first: exact for every value that the float64 -> bfloat16
    rounding would not also round, and the test tolerances cover the rest)."""
    return wl.to_bf16(y_ref.astype(np.float32))


@pytest.mark.parametrize("M", [1, 4, 8])
def test_routed_gemm_then_dense_decode(M):
    """A routed call on the tensor-core GEMM writes y1; right behind it on the stream a dense
    decode call (weight-streaming kernels: M = 1 on the CUDA-core kernel, 4 and 8 on the MMA
    kernel) reads y1's first M rows as its x."""
    import quantized_moe_expert_device_gb300 as g

    T, A, E, H1, F1, F2 = 128, 4, 8, 1024, 1024, 2048  # 64 rows per expert: the wide GEMM
    x1 = wl.normal_bf16((T, A, H1), 101)
    q1 = oracle.quantize(wl.normal_bf16((E, F1, H1), 102, chunk_rows=1))
    q2 = oracle.quantize(wl.normal_bf16((1, F2, F1), 103, std=F1 ** -0.5))
    idx = wl.idx_uniform(T, A, E, seed=104)
    d_x1, d_idx, d_q1, d_q2 = x1.cuda(), to_dev_idx(idx), _dev_q(q1), _dev_q(q2)
    ws1, ws2 = g.new_workspace(T * A, F1, E), g.new_workspace(M, F2, 1)
    before = {v: g.dispatch_count(v) for v in ("gemm_tc", "gemv", "gemv_mma")}
    outs = []
    for _ in range(ITERS):
        y1 = torch.zeros((T * A, F1), dtype=torch.bfloat16, device="cuda")
        y2 = torch.zeros((M, F2), dtype=torch.bfloat16, device="cuda")
        g.gqmm_gather_qmm(d_x1, *d_q1, d_idx, y=y1.view(T, A, F1), ws=ws1)
        g.gqmm_gather_qmm(y1[:M], *d_q2, None, y=y2, ws=ws2)
        outs.append((y1, y2))
    torch.cuda.synchronize()
    assert g.gqmm_device_status(ws1) == 0 and g.gqmm_device_status(ws2) == 0
    assert g.dispatch_count("gemm_tc") - before["gemm_tc"] == ITERS
    decode = "gemv" if M == 1 else "gemv_mma"
    assert g.dispatch_count(decode) - before[decode] == ITERS
    y1_ref = oracle.gather_qmm(x1, *q1, idx, E)
    y2_ref = oracle.gather_qmm(_bf16_of(y1_ref[:M]), *q2, None, 1)
    assert_parity(outs[0][0], y1_ref, "routed y1")
    assert_parity(outs[0][1], y2_ref, f"dense decode of y1, M={M}")
    for i, (y1, y2) in enumerate(outs[1:], 1):
        assert torch.equal(y1, outs[0][0]), f"iteration {i}: y1 differs"
        assert torch.equal(y2, outs[0][1]), f"iteration {i}: decode of y1 differs"


@pytest.mark.parametrize("n", [1, 4])
def test_dense_mlp_streaming_down_projection(n):
    """The dense expert MLP with I = 1024: both projections run on the weight-streaming kernels,
    the down projection right behind the gating kernel that writes its input."""
    import quantized_moe_expert_device_gb300 as g

    H, I = 2048, 1024
    q_gu = oracle.quantize(wl.normal_bf16((1, 2 * I, H), 111, std=H ** -0.5, chunk_rows=1))
    q_dn = oracle.quantize(wl.normal_bf16((1, H, I), 112, std=I ** -0.5, chunk_rows=1))
    x = wl.normal_bf16((n, H), 113)
    d_x, d_gu, d_dn = x.cuda(), _dev_q(q_gu), _dev_q(q_dn)
    kind = "gemv" if n == 1 else "gemv_mma"
    before = g.dispatch_count(kind)
    outs = []
    for _ in range(ITERS):
        ws = g.new_mlp_workspace(n, H, I, 1)
        y = torch.zeros((n, H), dtype=torch.bfloat16, device="cuda")
        g.gqmm_moe_mlp(d_x, d_gu, d_dn, None, y=y, ws=ws)
        outs.append((y, ws))
    torch.cuda.synchronize()
    assert g.dispatch_count(kind) - before == 2 * ITERS, "both projections on the streaming kernel"
    for _, ws in outs:
        assert g.gqmm_device_status(ws) == 0
    y_ref = oracle.moe_mlp(x, q_gu, q_dn, None, 1)
    assert_parity(outs[0][0], y_ref, f"dense mlp n={n}")
    for i, (y, _) in enumerate(outs[1:], 1):
        assert torch.equal(y, outs[0][0]), f"iteration {i}: y differs"


@pytest.mark.parametrize("M", [1, 8])
def test_quantize_then_dense_decode(M):
    """gqmm_quantize writes fresh codes, scales and biases; a dense decode call right behind it
    on the stream reads them."""
    import quantized_moe_expert_device_gb300 as g

    F, H = 4096, 2048
    w = wl.normal_bf16((1, F, H), 121, chunk_rows=1)
    x = wl.normal_bf16((M, H), 122)
    d_w, d_x = w.cuda(), x.cuda()
    ws = g.new_workspace(M, F, 1)
    kind = "gemv" if M == 1 else "gemv_mma"
    before = g.dispatch_count(kind)
    outs = []
    lib = g.load_library()
    stream = torch.cuda.current_stream()
    for _ in range(ITERS):
        wq = torch.zeros((1, F, H // 2), dtype=torch.uint8, device="cuda")
        sc = torch.zeros((1, F, H // 64), dtype=torch.bfloat16, device="cuda")
        bs = torch.zeros_like(sc)
        y = torch.zeros((M, F), dtype=torch.bfloat16, device="cuda")
        rc = lib.gqmm_quantize(d_w.data_ptr(), F, H, 64, 4, wq.data_ptr(), sc.data_ptr(), bs.data_ptr(),
                               stream.cuda_stream)
        assert rc == 0
        g.gqmm_gather_qmm(d_x, wq, sc, bs, None, y=y, ws=ws)
        outs.append(y)
    torch.cuda.synchronize()
    assert g.gqmm_device_status(ws) == 0
    assert g.dispatch_count(kind) - before == ITERS
    q = oracle.quantize(w)
    y_ref = oracle.gather_qmm(x, *q, None, 1)
    assert_parity(outs[0], y_ref, f"decode on fresh codes, M={M}")
    for i, y in enumerate(outs[1:], 1):
        assert torch.equal(y, outs[0]), f"iteration {i}: y differs"
