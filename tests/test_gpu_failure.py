"""The failure path of the tensor-core GEMM: every wait inside it is bounded, and a launch whose
wait runs out reports GQMM_STATUS_TIMEOUT, unwinds and frees its tensor memory, so that the context
and the next calls on the same stream stay usable.  The wait is made to run out with the library's
test hook (gqmm_test_stall_next: the launch leaves one stage of weight codes uncopied, a copy that
nothing then completes); no fault, trap or unbounded wait is involved."""
import time

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import assert_parity, to_dev_idx

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T,A,E,F,H", [(64, 8, 4, 512, 1024),   # wide variant (128 rows per expert)
                                       (16, 2, 8, 256, 512)])   # narrow variant (4 rows per expert)
def test_bounded_wait_runs_out_and_the_next_calls_work(T, A, E, F, H):
    import quantized_moe_expert_device_gb300 as g

    w = wl.normal_bf16((E, F, H), 31, chunk_rows=1)
    q = oracle.quantize(w)
    dev = g.gqmm_quantize(w.cuda())
    x = wl.normal_bf16((T, A, H), 32)
    idx = wl.idx_uniform(T, A, E, seed=33)
    d_x, d_idx = x.cuda(), to_dev_idx(idx)
    ws = g.new_workspace(T * A, F, E)
    torch.cuda.synchronize()

    g.test_stall_next(1)
    t0 = time.time()
    g.gqmm_gather_qmm(d_x, *dev, d_idx, ws=ws)
    status = g.gqmm_device_status(ws)
    elapsed = time.time() - t0
    g.test_stall_next(0)
    assert status & g.STATUS_TIMEOUT, f"status {status:#x}"
    assert elapsed < 30, f"the stalled launch took {elapsed:.1f} s"

    ref = oracle.gather_qmm(x, *q, idx, E)
    for _ in range(3):  # the same stream and workspace keep working (tensor memory was freed)
        y = g.gqmm_gather_qmm(d_x, *dev, d_idx, ws=ws)
        assert g.gqmm_device_status(ws) == 0
        assert_parity(y.reshape(-1, F), ref, f"after a timed-out launch T={T} A={A} E={E}")
