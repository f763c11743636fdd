"""gqmm_gather_qmm (tcgen05 grouped GEMM) on the GPU vs the CPU oracle.

Inputs: seeded workloads (x, W ~ N(0, 1) bf16, quantized by the oracle; idx per case).
Criteria: relative Frobenius error <= 5e-3 and every element within 2e-2 * max|y_ref|
(tests/helpers.py states the derivation)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import assert_parity, to_dev_idx

pytestmark = pytest.mark.gpu


def _weights(E, F, H, seed=wl.SEED_W, std=1.0):
    w = wl.normal_bf16((E, F, H), seed, std=std, chunk_rows=1)
    wq, sc, bs = oracle.quantize(w)
    dev = (torch.from_numpy(wq).cuda(), torch.from_numpy(sc.view(np.int16)).cuda().view(torch.bfloat16),
           torch.from_numpy(bs.view(np.int16)).cuda().view(torch.bfloat16))
    return (wq, sc, bs), dev


def _run(x_cpu, idx, E, host_w, dev_w, sorted_indices=False, simt=False):
    import quantized_moe_expert_device_gb300 as g

    x = x_cpu.cuda()
    d_idx = None if idx is None else to_dev_idx(idx)
    if simt:
        y = g.gqmm_gather_qmm_simt(x, *dev_w, d_idx)
        status = 0
    else:
        F = dev_w[0].shape[1]
        ws = g.new_workspace(x.numel() // x.shape[-1], F, E)
        y = g.gqmm_gather_qmm(x, *dev_w, d_idx, sorted_indices=sorted_indices, ws=ws)
        status = g.gqmm_device_status(ws)
    torch.cuda.synchronize()
    y_ref = oracle.gather_qmm(x_cpu, *host_w, idx, E)
    return y, y_ref, status


@pytest.mark.parametrize("simt", [False, True])
@pytest.mark.parametrize("sorted_indices", [False, True])
def test_tiny_config(sorted_indices, simt):
    w = wl.workloads()["tiny"]
    host_w, dev_w = _weights(w.E, w.F, w.H)
    inp = wl.make_inputs(w)
    x, idx = inp["x"], inp["idx"]
    if sorted_indices:
        x, idx, _ = wl.sorted_by_expert(x, idx)
    y, y_ref, status = _run(x, idx, w.E, host_w, dev_w, sorted_indices, simt)
    assert status == 0
    assert_parity(y.reshape(-1, w.F), y_ref, f"tiny sorted={sorted_indices} simt={simt}")


@pytest.mark.parametrize("rows_per_expert", [1, 2, 3, 4, 5, 8, 16, 17, 64, 255, 256, 257, 300, 513])
def test_rows_per_expert_regimes(rows_per_expert):
    # The pages' test regimes (mlx PR #4023 coverage discussion: 16 and 64 rows per expert and
    # a 78-row unaligned batch) plus the small-M decode range and chunk boundaries at 256.
    E, F, H = 4, 256, 512
    host_w, dev_w = _weights(E, F, H)
    n = rows_per_expert * E
    idx = wl.idx_balanced(rows_per_expert, E, 1).reshape(-1)
    x = wl.normal_bf16((n, H), wl.SEED_X)
    y, y_ref, status = _run(x, idx, E, host_w, dev_w)
    assert status == 0
    assert_parity(y, y_ref, f"r={rows_per_expert}")


@pytest.mark.parametrize("gs", [32, 64, 128])
def test_mid_variant_uneven_experts(gs):
    """33-64 routed rows per expert on average run on the mid variant (operands swapped: the chunk's
    tokens are the MMA's M rows, 256 weight rows its N; chunks of up to 128 tokens).  Experts of 150
    down to 2 rows (so one chunk splits at 128), F = 400 (a partial second 256-row unit), every group
    size, against the oracle; caller-sorted indices give the same bits as the unsorted call."""
    import quantized_moe_expert_device_gb300 as g

    E, F, H = 6, 400, 1024
    sizes = [150, 100, 40, 30, 10, 2]  # 332 rows: 56 per expert on average
    w = wl.normal_bf16((E, F, H), wl.SEED_W, chunk_rows=1)
    host_w = oracle.quantize(w, group_size=gs)
    dev_w = g.gqmm_quantize(w.cuda(), group_size=gs)
    idx = np.random.default_rng(gs).permutation(np.repeat(np.arange(E, dtype=np.uint32), sizes)).reshape(-1, 1)
    n = idx.shape[0]
    x = wl.normal_bf16((n, 1, H), wl.SEED_X)
    ws = g.new_workspace(n, F, E)
    y = g.gqmm_gather_qmm(x.cuda(), *dev_w, to_dev_idx(idx), group_size=gs, ws=ws)
    assert g.gqmm_device_status(ws) == 0
    assert_parity(y.reshape(n, F), oracle.gather_qmm(x, *host_w, idx, E, group_size=gs), f"mid gs={gs}")
    idx_s = np.sort(idx.reshape(-1)).reshape(-1, 1)
    y_s = g.gqmm_gather_qmm(x.cuda(), *dev_w, to_dev_idx(idx_s), group_size=gs, sorted_indices=True)
    y_u = g.gqmm_gather_qmm(x.cuda(), *dev_w, to_dev_idx(idx_s), group_size=gs, sorted_indices=False)
    torch.cuda.synchronize()
    assert torch.equal(y_s, y_u)


@pytest.mark.parametrize("H", [1024, 384])
@pytest.mark.parametrize("gs", [32, 64, 128])
def test_pair_variant_uneven_experts(gs, H):
    """More than 256 routed rows per expert on average run on CTA pairs (chunks of up to 512 tokens,
    each CTA of the pair dequantizing 128 of the unit's 256 weight rows).  Experts of 600, 300 and 10
    rows (one chunk splits at 512), F = 384 (the second unit has 128 weight rows, so the odd CTA of
    its pair has none), every group size, H/gs a multiple of 8 (one 16-byte scale load covers eight
    groups) and not (H = 384), against the oracle; caller-sorted indices give the same bits as the
    unsorted call."""
    import quantized_moe_expert_device_gb300 as g

    E, F = 3, 384
    sizes = [600, 300, 10]  # 910 rows: 303 per expert on average
    w = wl.normal_bf16((E, F, H), wl.SEED_W, chunk_rows=1)
    host_w = oracle.quantize(w, group_size=gs)
    dev_w = g.gqmm_quantize(w.cuda(), group_size=gs)
    idx = np.random.default_rng(gs + H).permutation(np.repeat(np.arange(E, dtype=np.uint32), sizes)).reshape(-1, 1)
    n = idx.shape[0]
    x = wl.normal_bf16((n, 1, H), wl.SEED_X)
    ws = g.new_workspace(n, F, E)
    y = g.gqmm_gather_qmm(x.cuda(), *dev_w, to_dev_idx(idx), group_size=gs, ws=ws)
    assert g.gqmm_device_status(ws) == 0
    assert_parity(y.reshape(n, F), oracle.gather_qmm(x, *host_w, idx, E, group_size=gs), f"pair gs={gs} H={H}")
    idx_s = np.sort(idx.reshape(-1)).reshape(-1, 1)
    y_s = g.gqmm_gather_qmm(x.cuda(), *dev_w, to_dev_idx(idx_s), group_size=gs, sorted_indices=True)
    y_u = g.gqmm_gather_qmm(x.cuda(), *dev_w, to_dev_idx(idx_s), group_size=gs, sorted_indices=False)
    torch.cuda.synchronize()
    assert torch.equal(y_s, y_u)


def test_unaligned_78_row_batch_sorted_and_unsorted():
    E, F, H = 4, 128, 1024
    host_w, dev_w = _weights(E, F, H)
    idx = np.random.default_rng(78).integers(0, E, size=78, dtype=np.uint32)
    x = wl.normal_bf16((78, H), wl.SEED_X)
    y, y_ref, _ = _run(x, idx, E, host_w, dev_w)
    assert_parity(y, y_ref, "78 unsorted")
    xs, idx_s, _ = wl.sorted_by_expert(x.reshape(78, 1, H), idx.reshape(78, 1))
    ys, ys_ref, _ = _run(xs, idx_s, E, host_w, dev_w, sorted_indices=True)
    assert_parity(ys, ys_ref, "78 sorted")


@pytest.mark.parametrize("F", [16, 144, 400])
def test_f_not_a_multiple_of_the_tile(F):
    E, H = 3, 256
    host_w, dev_w = _weights(E, F, H)
    idx = np.random.default_rng(F).integers(0, E, size=100, dtype=np.uint32)
    x = wl.normal_bf16((100, H), wl.SEED_X)
    y, y_ref, _ = _run(x, idx, E, host_w, dev_w)
    assert_parity(y, y_ref, f"F={F}")


@pytest.mark.parametrize("H", [64, 192, 448, 4096])
def test_h_sizes_scalar_and_vector_scale_paths(H):
    # H % 512 != 0 takes the per-group scale fetch, H % 512 == 0 the 8-group one
    E, F = 2, 128
    host_w, dev_w = _weights(E, F, H)
    idx = np.random.default_rng(H).integers(0, E, size=40, dtype=np.uint32)
    x = wl.normal_bf16((40, H), wl.SEED_X)
    y, y_ref, _ = _run(x, idx, E, host_w, dev_w)
    assert_parity(y, y_ref, f"H={H}")


def test_dense_e1_matches_gather_with_zero_index_bitwise():
    E, F, H = 1, 256, 1024
    host_w, dev_w = _weights(E, F, H)
    x = wl.normal_bf16((300, H), wl.SEED_X)
    yd, y_ref, _ = _run(x, None, 1, host_w, dev_w)
    assert_parity(yd, y_ref, "dense")
    y0, _, _ = _run(x, np.zeros(300, np.uint32), 1, host_w, dev_w)
    assert torch.equal(yd, y0)


def test_sorted_equals_unsorted_bitwise():
    w = wl.workloads()["tiny"]
    E, F, H = 16, 256, 512
    host_w, dev_w = _weights(E, F, H)
    idx = wl.idx_uniform(200, 4, E)
    x = wl.normal_bf16((200, 4, H), wl.SEED_X)
    y, y_ref, _ = _run(x, idx, E, host_w, dev_w)
    assert_parity(y.reshape(-1, F), y_ref, "unsorted")
    xs, idx_s, order = wl.sorted_by_expert(x, idx)
    ys, _, _ = _run(xs, idx_s, E, host_w, dev_w, sorted_indices=True)
    assert torch.equal(ys.cpu(), y.reshape(-1, F).cpu()[torch.from_numpy(order)])
    del w


def test_invalid_index_rows_are_zero_and_flagged():
    import quantized_moe_expert_device_gb300 as g

    E, F, H = 4, 128, 256
    host_w, dev_w = _weights(E, F, H)
    idx = np.random.default_rng(3).integers(0, E, size=64, dtype=np.uint32)
    idx[5] = E
    idx[40] = 2**32 - 1
    x = wl.normal_bf16((64, H), wl.SEED_X)
    for sorted_indices in (False, True):
        xi, ii = x, idx
        if sorted_indices:
            xi, ii, _ = wl.sorted_by_expert(x.reshape(64, 1, H), idx.reshape(64, 1))
        y, y_ref, status = _run(xi, ii, E, host_w, dev_w, sorted_indices)
        assert status & g.STATUS_BAD_INDEX
        assert_parity(y.reshape(64, F), y_ref, f"bad index sorted={sorted_indices}")
        bad_rows = np.nonzero(np.asarray(ii).reshape(-1) >= E)[0]
        assert (y.reshape(64, F)[torch.from_numpy(bad_rows).cuda()] == 0).all()


def test_false_sorted_promise_is_flagged():
    import quantized_moe_expert_device_gb300 as g

    E, F, H = 4, 128, 256
    _, dev_w = _weights(E, F, H)
    idx = to_dev_idx(np.array([3, 2, 1, 0] * 8, np.uint32))
    x = wl.normal_bf16((32, H), wl.SEED_X).cuda()
    ws = g.new_workspace(32, F, E)
    g.gqmm_gather_qmm(x, *dev_w, idx, sorted_indices=True, ws=ws)
    assert g.gqmm_device_status(ws) & g.STATUS_NOT_SORTED
    assert g.gqmm_device_status(ws) == 0  # reading clears


def test_workspace_reuse_across_shapes_and_calls():
    import quantized_moe_expert_device_gb300 as g

    E, F, H = 8, 256, 512
    host_w, dev_w = _weights(E, F, H)
    shapes = (1000, 17, 4096, 256)
    ws = g.new_workspace(list(shapes), F, E)
    for n in shapes:
        idx = np.random.default_rng(n).integers(0, E, size=n, dtype=np.uint32)
        x = wl.normal_bf16((n, H), n)
        y = g.gqmm_gather_qmm(x.cuda(), *dev_w, to_dev_idx(idx), ws=ws)
        assert_parity(y, oracle.gather_qmm(x, *host_w, idx, E), f"n={n}")
    assert g.gqmm_device_status(ws) == 0


def test_repeated_calls_many_units_per_cta_match_oracle_every_time():
    """Regression test for cross-stage races: with T*A=16384, E=64, F=768 every CTA runs
    several work units, and each call starts with a cold pipeline.  Every one of 30 calls
    (with a device synchronization before each) must match the oracle."""
    import quantized_moe_expert_device_gb300 as g

    w = wl.workloads()["prefill_e64"]
    host_w, dev_w = _weights(w.E, w.F, w.H)
    inp = wl.make_inputs(w)
    x_cpu, idx = inp["x"], inp["idx"]
    y_ref = oracle.gather_qmm(x_cpu, *host_w, idx, w.E)
    x = x_cpu.cuda()
    d_idx = to_dev_idx(idx)
    ws = g.new_workspace(w.n, w.F, w.E)
    first = None
    for rep in range(30):
        torch.cuda.synchronize()
        y = g.gqmm_gather_qmm(x, *dev_w, d_idx, ws=ws).reshape(w.n, w.F)
        assert_parity(y, y_ref, f"rep {rep}")
        if first is None:
            first = y.clone()
        else:
            assert torch.equal(y, first), f"rep {rep} differs from rep 0"
    assert g.gqmm_device_status(ws) == 0


def test_dispatch_coverage_every_variant_runs_and_matches():
    """Each internal variant (wide and narrow GEMM, split-K, weight streaming, the three routing paths) is
    exercised and checked here, in the manner of the pages' coverage check (mlx PR #4023:
    log each dispatched kernel while running the suite, count the distinct ones)."""
    import quantized_moe_expert_device_gb300 as g

    before = {k: g.dispatch_count(k) for k in g.VARIANTS}
    E, F, H = 8, 512, 1024
    host_w, dev_w = _weights(E, F, H)
    cases = [
        (wl.idx_uniform(512, 8, E), False),            # 512 rows/expert: wide, no split
        (wl.idx_uniform(16, 4, E), False),             # 8 rows/expert, few units: narrow + split-K
        (wl.idx_uniform(4, 2, E), False),              # 1 row/expert: weight streaming
        (np.sort(wl.idx_uniform(64, 4, E).reshape(-1)).reshape(64, 4), True),  # caller-sorted
    ]
    for idx, srt in cases:
        x = wl.normal_bf16(idx.shape + (H,), wl.SEED_X)
        y, y_ref, status = _run(x, idx, E, host_w, dev_w, sorted_indices=srt)
        assert status == 0
        assert_parity(y.reshape(-1, F), y_ref, f"coverage {idx.shape} sorted={srt}")
    host1, dev1 = _weights(1, F, H)
    for rows in (2, 3):                              # dense decode: CUDA-core and MMA streaming
        x = wl.normal_bf16((rows, H), wl.SEED_X)
        yd, yd_ref, _ = _run(x, None, 1, host1, dev1)
        assert_parity(yd, yd_ref, f"coverage dense {rows} rows")
    # transpose=False: W [E, K = H, N = 256] quantized along N
    w_nn = wl.normal_bf16((E, H, 256), 91, chunk_rows=1)
    q_nn_host, q_nn_dev = oracle.quantize(w_nn), g.gqmm_quantize(w_nn.cuda())
    idx_nn = wl.idx_uniform(8, 2, E)
    x_nn = wl.normal_bf16((8, 2, H), 92)
    y_nn = g.gqmm_gather_qmm_nn(x_nn.cuda(), *q_nn_dev, to_dev_idx(idx_nn))
    torch.cuda.synchronize()
    assert_parity(y_nn, oracle.gather_qmm_nn(x_nn, *q_nn_host, idx_nn, E), "coverage transpose=False")
    after = {k: g.dispatch_count(k) for k in g.VARIANTS}
    for k in g.VARIANTS:
        assert after[k] > before[k], f"variant {k} never dispatched"


@pytest.mark.parametrize("M", [1, 2, 3, 5, 8, 9])
@pytest.mark.parametrize("H", [1024, 4096])
def test_weight_streaming_dense_matches_oracle(M, H):
    """Dense decode shapes: 1 row runs on the CUDA-core weight-streaming kernel, 2 to 8 on the
    MMA one, 9 on the narrow tensor-core kernel; F is not a multiple of any row batch."""
    import quantized_moe_expert_device_gb300 as g

    F = 400
    host_w, dev_w = _weights(1, F, H)
    before = g.dispatch_count("gemv"), g.dispatch_count("gemv_mma")
    x = wl.normal_bf16((M, H), wl.SEED_X + M)
    y, y_ref, status = _run(x, None, 1, host_w, dev_w)
    assert status == 0
    assert (g.dispatch_count("gemv") > before[0]) == (M == 1)
    assert (g.dispatch_count("gemv_mma") > before[1]) == (2 <= M <= 8)
    assert_parity(y, y_ref, f"stream dense M={M} H={H}")


@pytest.mark.parametrize("M,H", [(1, 768), (2, 768), (3, 768), (1, 640), (2, 1536), (1, 8192)])
def test_weight_streaming_dense_k_not_a_multiple_of_1024(M, H):
    """K a multiple of 128 but not of 1024 (the CUDA-core streaming kernel pads a row's threads to a
    power of two, the extra threads adding zeros): 1 and 2 rows stream on the CUDA-core kernel, the
    MMA streaming kernel does not take these K, so 3 rows go to the narrow tensor-core kernel."""
    import quantized_moe_expert_device_gb300 as g

    F = 400
    host_w, dev_w = _weights(1, F, H)
    before = g.dispatch_count("gemv"), g.dispatch_count("gemv_mma")
    x = wl.normal_bf16((M, H), wl.SEED_X + M)
    y, y_ref, status = _run(x, None, 1, host_w, dev_w)
    assert status == 0
    assert (g.dispatch_count("gemv") > before[0]) == (M <= 2)
    assert g.dispatch_count("gemv_mma") == before[1]
    assert_parity(y, y_ref, f"stream dense M={M} H={H}")


@pytest.mark.parametrize("T,A,E,H,hot", [(1, 8, 128, 2048, 1), (8, 8, 128, 2048, 1), (5, 3, 16, 1024, 1),
                                         (32, 8, 256, 2048, 1), (32, 8, 256, 2048, 3),
                                         (4, 8, 64, 768, 1), (3, 8, 32, 1536, 1), (2, 8, 16, 640, 1)])
def test_weight_streaming_moe_matches_oracle(T, A, E, H, hot):
    """MoE decode shapes with at most 1.5 rows per hit expert on average run on the
    weight-streaming kernel in chunks of 2 rows; an expert with more rows gets several chunks
    (`hot` tokens send all their A rows to expert 3)."""
    import quantized_moe_expert_device_gb300 as g

    F = 272
    host_w, dev_w = _weights(E, F, H)
    idx = np.random.default_rng(T * 1000 + E).integers(0, E, size=(T, A), dtype=np.uint32)
    idx[:hot, :] = 3
    before = g.dispatch_count("gemv")
    x = wl.normal_bf16((T, A, H), wl.SEED_X)
    y, y_ref, status = _run(x, idx, E, host_w, dev_w)
    assert status == 0
    assert g.dispatch_count("gemv") > before
    assert_parity(y.reshape(-1, F), y_ref, f"stream moe T={T} A={A} E={E}")


def test_weight_streaming_one_item_chunks():
    """F = 16 makes every chunk a single work item, so each block of the streaming kernel
    moves through a new chunk (and a new copy of x) at every item."""
    import quantized_moe_expert_device_gb300 as g

    E, F, H = 512, 16, 1024
    host_w, dev_w = _weights(E, F, H)
    idx = np.random.default_rng(5).integers(0, E, size=(64, 8), dtype=np.uint32)
    before = g.dispatch_count("gemv")
    x = wl.normal_bf16((64, 8, H), wl.SEED_X)
    y, y_ref, status = _run(x, idx, E, host_w, dev_w)
    assert status == 0
    assert g.dispatch_count("gemv") > before
    assert_parity(y.reshape(-1, F), y_ref, "stream one-item chunks")


def test_weight_streaming_invalid_indices_and_unsupported_h():
    """Invalid indices give zero rows on the streaming path; an H the streaming kernel does
    not take (192: not a multiple of the kernel's k slices) runs the narrow tensor-core kernel
    with the same small chunks."""
    import quantized_moe_expert_device_gb300 as g

    E, F = 16, 144
    for H, expect_stream in ((1024, True), (4096, True), (768, True), (192, False)):
        host_w, dev_w = _weights(E, F, H)
        idx = np.random.default_rng(H).integers(0, E, size=(6, 2), dtype=np.uint32)
        idx[2, 1] = E + 5
        before = g.dispatch_count("gemv")
        x = wl.normal_bf16((6, 2, H), wl.SEED_X)
        y, y_ref, status = _run(x, idx, E, host_w, dev_w)
        assert status & g.STATUS_BAD_INDEX
        assert (g.dispatch_count("gemv") > before) == expect_stream
        assert_parity(y.reshape(-1, F), y_ref, f"stream invalid H={H}")


@pytest.mark.parametrize("T,A", [(8, 8), (12, 5), (65, 1), (64, 1)])
def test_in_kernel_plan_matches_route_kernel_bitwise(T, A):
    """Unsorted routed decode calls of at most 64 rows are planned inside the streaming kernel
    (no route kernel); 65 rows go through the route kernel.  Either way the result equals, bit
    for bit, the same rows run caller-sorted through the sorted-route plan, and meets the oracle.
    Expert 3 is sent five rows (chunks of 2, 2 and 1) and one row has an invalid index."""
    import quantized_moe_expert_device_gb300 as g

    E, F, H = 96, 272, 2048
    host_w, dev_w = _weights(E, F, H)
    idx = np.random.default_rng(T * 7 + A).permutation(E)[np.arange(T * A) % E].astype(np.uint32).reshape(T, A)
    idx.reshape(-1)[[1, 4, 6, 9, 12]] = 3
    idx.reshape(-1)[2] = E + 1
    x = wl.normal_bf16((T, A, H), wl.SEED_X)
    before = {k: g.dispatch_count(k) for k in ("route_fused", "route_unsorted", "gemv")}
    y, y_ref, status = _run(x, idx, E, host_w, dev_w)
    assert status & g.STATUS_BAD_INDEX
    fused = T * A <= 64
    assert (g.dispatch_count("route_fused") > before["route_fused"]) == fused
    assert (g.dispatch_count("route_unsorted") > before["route_unsorted"]) == (not fused)
    assert g.dispatch_count("gemv") > before["gemv"]
    assert_parity(y.reshape(-1, F), y_ref, f"in-kernel plan T={T} A={A}")
    xs, idx_s, order = wl.sorted_by_expert(x, idx)
    ys, _, _ = _run(xs, idx_s.reshape(-1, 1), E, host_w, dev_w, sorted_indices=True)
    y_back = torch.empty_like(ys.reshape(-1, F))
    y_back[torch.from_numpy(order).cuda()] = ys.reshape(-1, F)
    assert torch.equal(y.reshape(-1, F), y_back), "in-kernel plan and sorted-route plan differ"


def test_in_kernel_plan_with_shared_x():
    """The in-kernel plan with x shared by a token's A rows ([T, H]) equals the call on x repeated
    A times, bit for bit."""
    import quantized_moe_expert_device_gb300 as g

    T, A, E, F, H = 6, 8, 128, 256, 2048
    host_w, dev_w = _weights(E, F, H)
    idx = wl.idx_topk_distinct_uniform(T, A, E, seed=17)
    x_tok = wl.normal_bf16((T, H), 18)
    before = g.dispatch_count("route_fused")
    y_shared = g.gqmm_gather_qmm(x_tok.cuda(), *dev_w, to_dev_idx(idx))
    y_rep = g.gqmm_gather_qmm(x_tok.cuda().unsqueeze(1).expand(T, A, H).contiguous(), *dev_w, to_dev_idx(idx))
    torch.cuda.synchronize()
    assert g.dispatch_count("route_fused") - before == 2
    assert torch.equal(y_shared, y_rep)
