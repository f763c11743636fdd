"""gqmm_gather_qmm_noalloc: the entry point for callers that cannot allocate device memory.

It must give the same results as gqmm_gather_qmm (which takes a caller workspace) when called
through the C ABI, on consecutive calls that share its built-in scratch, and it must refuse
sizes its scratch cannot hold.  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import workloads as wl
from helpers import assert_parity, to_dev_idx

pytestmark = pytest.mark.gpu

P, I, I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64


def _lib():
    import quantized_moe_expert_device_gb300 as g

    lib = g.load_library()
    fn = lib.gqmm_gather_qmm_noalloc
    fn.argtypes = [P, P, P, P, P, I64, I, I, I, I, I, I, I, P, P]
    fn.restype = I
    return g, lib, fn


def _call_noalloc(fn, x, wq, sc, bs, idx, T, A, H, F, E, sorted_flag):
    y = torch.empty(T, A, F, dtype=torch.bfloat16, device="cuda")
    stream = P(torch.cuda.current_stream().cuda_stream)
    rc = fn(P(x.data_ptr()), P(wq.data_ptr()), P(sc.data_ptr()), P(bs.data_ptr()),
            None if idx is None else P(idx.data_ptr()), T, A, H, F, E, 64, 4, sorted_flag,
            P(y.data_ptr()), stream)
    return rc, y


def test_noalloc_matches_gather_qmm_on_two_consecutive_calls():
    g, lib, fn = _lib()
    E, F, H = 16, 384, 1024
    wq, sc, bs = g.gqmm_quantize(wl.normal_bf16((E, F, H), wl.SEED_W, chunk_rows=1).cuda())
    # call 1: unsorted routing; call 2: a different, smaller, caller-sorted batch that reuses
    # the same built-in scratch right after call 1
    T1, A1 = 512, 4
    x1 = wl.normal_bf16((T1, A1, H), 11).cuda()
    i1 = wl.idx_uniform(T1, A1, E, seed=12)
    T2, A2 = 97, 2
    x2c = wl.normal_bf16((T2, A2, H), 13)
    x2s, i2s, _ = wl.sorted_by_expert(x2c, wl.idx_uniform(T2, A2, E, seed=14))
    x2 = x2s.reshape(T2, A2, H).cuda()
    i2 = i2s.reshape(T2, A2)

    rc1, y1 = _call_noalloc(fn, x1, wq, sc, bs, to_dev_idx(i1), T1, A1, H, F, E, 0)
    assert rc1 == 0, lib.gqmm_last_error()
    rc2, y2 = _call_noalloc(fn, x2, wq, sc, bs, to_dev_idx(i2), T2, A2, H, F, E, 1)
    assert rc2 == 0, lib.gqmm_last_error()
    torch.cuda.synchronize()

    r1 = g.gqmm_gather_qmm(x1, wq, sc, bs, to_dev_idx(i1))
    r2 = g.gqmm_gather_qmm(x2, wq, sc, bs, to_dev_idx(i2), sorted_indices=True)
    torch.cuda.synchronize()
    assert_parity(y1.reshape(-1, F), r1.reshape(-1, F).double().cpu().numpy(), "noalloc call 1")
    assert_parity(y2.reshape(-1, F), r2.reshape(-1, F).double().cpu().numpy(), "noalloc call 2")


def test_noalloc_dense_and_rejects_sizes_beyond_its_scratch():
    g, lib, fn = _lib()
    E, F, H = 1, 256, 512
    wq, sc, bs = g.gqmm_quantize(wl.normal_bf16((E, F, H), 3).cuda())
    x = wl.normal_bf16((40, 1, H), 4).cuda()
    rc, y = _call_noalloc(fn, x, wq, sc, bs, None, 40, 1, H, F, E, 0)
    assert rc == 0, lib.gqmm_last_error()
    ref = g.gqmm_gather_qmm(x, wq, sc, bs, None)
    torch.cuda.synchronize()
    assert_parity(y.reshape(-1, F), ref.reshape(-1, F).double().cpu().numpy(), "noalloc dense")

    # 131072 rows always fit; far more rows than the scratch holds are refused, no launch
    assert g.gqmm_workspace_size(131072, F, g.MAX_EXPERTS) <= (1 << 20)
    lib.gqmm_last_error.restype = ctypes.c_char_p
    too_many = 1 << 19
    rc = fn(P(x.data_ptr()), P(wq.data_ptr()), P(sc.data_ptr()), P(bs.data_ptr()), P(x.data_ptr()),
            too_many, 1, H, F, 64, 64, 4, 0, P(y.data_ptr()), None)
    assert rc == 5  # GQMM_ERR_WORKSPACE
    assert b"scratch" in lib.gqmm_last_error()
    # the entry point stays usable after a refusal
    rc, y3 = _call_noalloc(fn, x, wq, sc, bs, None, 40, 1, H, F, E, 0)
    assert rc == 0
    torch.cuda.synchronize()
    assert torch.equal(y3, y)
