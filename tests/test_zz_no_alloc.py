"""gqmm_gather_qmm_noalloc: the entry point for callers that cannot allocate device memory
(a plugin whose host framework owns all device memory, a path that must not block in
cudaMalloc).  It keeps its scratch in a fixed array inside the library.

Its results must equal those of gqmm_gather_qmm (which takes a caller workspace) bit for bit
wherever the two split the work the same way (they run the same kernels on the same inputs),
and within the parity tolerance where gqmm_gather_qmm splits K into partial-sum planes that the
built-in scratch cannot hold.  This must hold through the C ABI, on consecutive calls that share
the built-in scratch, on a decode-sized call that splits K inside the scratch, and at the largest
call the scratch is documented to hold.  The entry point must refuse larger calls with a clear
error.  Two calls are also checked against the float64 oracle.  This file is collected last on
purpose."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
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


def _call_noalloc(fn, x, wq, sc, bs, idx, T, A, H, F, E, sorted_flag, y=None):
    if y is None:
        y = torch.empty(T, A, F, dtype=torch.bfloat16, device="cuda")
    stream = P(torch.cuda.current_stream().cuda_stream)
    rc = fn(P(x.data_ptr()), P(wq.data_ptr()), P(sc.data_ptr()), P(bs.data_ptr()),
            None if idx is None else P(idx.data_ptr()), T, A, H, F, E, 64, 4, sorted_flag,
            P(y.data_ptr()), stream)
    return rc, y


def test_noalloc_matches_gather_qmm_on_two_consecutive_calls():
    g, lib, fn = _lib()
    E, F, H = 16, 384, 1024
    w = wl.normal_bf16((E, F, H), wl.SEED_W, chunk_rows=1)
    wq, sc, bs = g.gqmm_quantize(w.cuda())
    # call 1: unsorted routing; call 2: a different, smaller, caller-sorted batch that reuses
    # the same built-in scratch right after call 1
    T1, A1 = 512, 4
    x1h = wl.normal_bf16((T1, A1, H), 11)
    x1 = x1h.cuda()
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
    assert torch.equal(y1, r1), "noalloc call 1 differs from gqmm_gather_qmm"
    # Call 2 has few work units, so gqmm_gather_qmm splits K into float32 partial-sum planes;
    # those planes (14 x 194 x 384 floats) do not fit the built-in scratch, so the no-allocation
    # call runs unsplit.  Only the float32 summation order differs: equal within the parity
    # tolerance, not bit for bit.
    q = oracle.quantize(w)
    assert_parity(y2.reshape(-1, F), r2.reshape(-1, F).double().cpu().numpy(), "noalloc call 2 vs gqmm_gather_qmm")
    assert_parity(y2.reshape(-1, F), oracle.gather_qmm(x2s, *q, i2, E), "noalloc call 2 against the oracle")
    assert_parity(y1.reshape(-1, F), oracle.gather_qmm(x1h, *q, i1, E), "noalloc call 1 against the oracle")


def test_noalloc_split_k_decode_call_inside_the_scratch():
    """A routed decode-sized call (16 rows over 4 experts, K = 1024): gqmm_gather_qmm splits K
    into float32 partial-sum planes, and those planes fit in the built-in scratch too."""
    g, lib, fn = _lib()
    E, F, H, T, A = 4, 256, 1024, 2, 8
    wq, sc, bs = g.gqmm_quantize(wl.normal_bf16((E, F, H), 21, chunk_rows=1).cuda())
    x = wl.normal_bf16((T, A, H), 22).cuda()
    idx = to_dev_idx(wl.idx_uniform(T, A, E, seed=23))
    before = g.dispatch_count("split_k")
    outs = [_call_noalloc(fn, x, wq, sc, bs, idx, T, A, H, F, E, 0) for _ in range(2)]
    assert g.dispatch_count("split_k") - before == 2, "the call splits K"
    ref = g.gqmm_gather_qmm(x, wq, sc, bs, idx)
    torch.cuda.synchronize()
    for rc, y in outs:
        assert rc == 0, lib.gqmm_last_error()
        assert torch.equal(y, ref)


def test_noalloc_dense_and_rejects_sizes_beyond_its_scratch():
    g, lib, fn = _lib()
    E, F, H = 1, 256, 512
    wq, sc, bs = g.gqmm_quantize(wl.normal_bf16((E, F, H), 3).cuda())
    x = wl.normal_bf16((40, 1, H), 4).cuda()
    rc, y = _call_noalloc(fn, x, wq, sc, bs, None, 40, 1, H, F, E, 0)
    assert rc == 0, lib.gqmm_last_error()
    ref = g.gqmm_gather_qmm(x, wq, sc, bs, None)
    torch.cuda.synchronize()
    assert torch.equal(y, ref)

    # far more rows than the scratch holds are refused, with a message, and nothing runs
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


def test_noalloc_at_its_documented_limit():
    """T*A = 131072 rows with E = GQMM_MAX_EXPERTS (1024) is the largest call the scratch is
    documented to hold: it must run and match gqmm_gather_qmm."""
    g, lib, fn = _lib()
    E, F, H, T, A = g.MAX_EXPERTS, 16, 64, 16384, 8
    assert g.gqmm_workspace_size(T * A, F, E) <= (1 << 20)
    wq, sc, bs = g.gqmm_quantize(wl.normal_bf16((E, F, H), 31, chunk_rows=64).cuda())
    x = wl.normal_bf16((T, A, H), 32, chunk_rows=4096).cuda()
    idx = to_dev_idx(wl.idx_uniform(T, A, E, seed=33))
    rc, y = _call_noalloc(fn, x, wq, sc, bs, idx, T, A, H, F, E, 0)
    assert rc == 0, lib.gqmm_last_error()
    ref = g.gqmm_gather_qmm(x, wq, sc, bs, idx)
    torch.cuda.synchronize()
    assert torch.equal(y, ref)


def test_noalloc_false_sorted_promise_gives_zeros():
    """The status word is not readable through this entry point, so a broken sorted = 1
    promise must leave a defined result: y all zeros."""
    g, lib, fn = _lib()
    E, F, H, T, A = 8, 128, 256, 16, 2
    wq, sc, bs = g.gqmm_quantize(wl.normal_bf16((E, F, H), 41).cuda())
    x = wl.normal_bf16((T, A, H), 42).cuda()
    idx = np.arange(T * A, dtype=np.uint32)[::-1].copy() % E  # decreasing somewhere: not sorted
    y = torch.full((T, A, F), 7.0, dtype=torch.bfloat16, device="cuda")
    rc, y = _call_noalloc(fn, x, wq, sc, bs, to_dev_idx(idx.reshape(T, A)), T, A, H, F, E, 1, y=y)
    assert rc == 0, lib.gqmm_last_error()
    torch.cuda.synchronize()
    assert torch.count_nonzero(y).item() == 0
