"""gqmm_gather_qmm_nn (transpose=False: W[e] = [K, N] quantized along N) on the GPU against the
oracle's float64 gather_qmm_nn, on the GPU's own quantized weights (bit-equal to the oracle's).

The tensor-core path: the shape of the pages' transpose=False timing (E=4, K=N=512, 1024 rows),
every group size on both GEMM variants (wide chunks of up to 256 rows, whose A operand is MN-major,
and narrow ones of up to 32, whose A is K-major in tensor memory), N not a multiple of the
256-column unit or of 64, a decode-sized call that splits K, dense E=1, invalid indices, a shared x,
and caller-sorted indices equal to the unsorted call bit for bit on both variants.  The
CUDA-core cross-check gqmm_gather_qmm_nn_simt takes any K; it is checked on K that are not
multiples of 64 as well.  Tolerances are the gather's (relative Frobenius error <= 5e-3, every
element within 2e-2 * max|y_ref|): weights are decoded exactly and rounded once to bfloat16."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import assert_parity, np_of, to_dev_idx

pytestmark = pytest.mark.gpu


def _weights(E, K, N, gs, seed):
    import quantized_moe_expert_device_gb300 as g

    w = wl.normal_bf16((E, K, N), seed, chunk_rows=1)
    host = oracle.quantize(w, group_size=gs)
    dev = g.gqmm_quantize(w.cuda(), group_size=gs)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(np_of(dev[0]), host[0])
    return host, dev


NN_CASES = [(1024, 1, 512, 512, 4, 64),     # the pages' transpose=False shape (wide chunks)
            (16, 2, 256, 256, 8, 32),       # narrow chunks
            (7, 3, 3072, 1152, 5, 128),     # N = 4.5 units of 256 columns
            (4, 8, 2048, 768, 64, 64),
            (2, 4, 4096, 512, 4, 64),       # decode-sized: K split into slices
            (5, 1, 320, 96, 1, 32),         # dense (idx None), N below one unit
            (300, 2, 192, 32, 3, 32),       # the smallest N, ragged chunk tails (wide)
            (512, 2, 1024, 640, 4, 128),    # wide, 128-wide groups, N = 2.5 units
            (600, 1, 512, 800, 1, 32)]      # dense wide, N % 64 == 32 (a 64-column chunk half past N)


@pytest.mark.parametrize("T,A,K,N,E,gs", NN_CASES)
def test_nn_matches_oracle(T, A, K, N, E, gs):
    import quantized_moe_expert_device_gb300 as g

    host, dev = _weights(E, K, N, gs, seed=81)
    x = wl.normal_bf16((T, A, K) if E > 1 else (T, K), 82)
    idx = None if E == 1 else np.random.default_rng(T + K).integers(0, E, size=(T, A)).astype(np.uint32)
    ws = g.new_workspace(T * A, N, E)
    y = g.gqmm_gather_qmm_nn(x.cuda(), *dev, None if idx is None else to_dev_idx(idx), group_size=gs, ws=ws)
    assert g.gqmm_device_status(ws) == 0
    assert y.shape[-1] == N
    assert_parity(y, oracle.gather_qmm_nn(x, *host, idx, E, group_size=gs), f"nn T={T} A={A} K={K} N={N} E={E}")


def test_nn_invalid_indices_shared_x_and_sorted():
    import quantized_moe_expert_device_gb300 as g

    T, A, K, N, E = 12, 4, 512, 256, 6
    host, dev = _weights(E, K, N, 64, seed=83)
    x = wl.normal_bf16((T, K), 84)
    idx = np.random.default_rng(8).integers(0, E, size=(T, A)).astype(np.uint32)
    idx[::3, 2] = E + 1
    ws = g.new_workspace(T * A, N, E)
    y = g.gqmm_gather_qmm_nn(x.cuda(), *dev, to_dev_idx(idx), ws=ws)          # x [T, K] shared by the A rows
    assert g.gqmm_device_status(ws) & g.STATUS_BAD_INDEX
    x_rep = x.repeat_interleave(A, dim=0).reshape(T, A, K)
    y_rep = g.gqmm_gather_qmm_nn(x_rep.cuda(), *dev, to_dev_idx(idx))
    torch.cuda.synchronize()
    assert y.shape == (T, A, N) and torch.equal(y, y_rep)
    assert not y[::3, 2].float().abs().sum().item()
    assert_parity(y, oracle.gather_qmm_nn(x_rep, *host, idx, E), "nn invalid + shared")
    # caller-sorted indices through the sorted-route plan equal the unsorted call bit for bit
    idx_s = np.sort(np.random.default_rng(9).integers(0, E, size=T * A)).astype(np.uint32).reshape(-1, 1)
    xs = wl.normal_bf16((T * A, 1, K), 85).cuda()
    y_s = g.gqmm_gather_qmm_nn(xs, *dev, to_dev_idx(idx_s), sorted_indices=True)
    y_u = g.gqmm_gather_qmm_nn(xs, *dev, to_dev_idx(idx_s), sorted_indices=False)
    torch.cuda.synchronize()
    assert torch.equal(y_s, y_u)


def test_nn_wide_sorted_equals_unsorted_and_invalid_index():
    """The wide variant (MN-major A): caller-sorted indices equal the unsorted call bit for bit,
    and an invalid index gives a zero row and the status bit."""
    import quantized_moe_expert_device_gb300 as g

    T, K, N, E = 1200, 768, 576, 4
    host, dev = _weights(E, K, N, 64, seed=90)
    idx_s = np.sort(np.random.default_rng(10).integers(0, E, size=T)).astype(np.uint32).reshape(-1, 1)
    x = wl.normal_bf16((T, 1, K), 91)
    xs = x.cuda()
    y_s = g.gqmm_gather_qmm_nn(xs, *dev, to_dev_idx(idx_s), sorted_indices=True)
    y_u = g.gqmm_gather_qmm_nn(xs, *dev, to_dev_idx(idx_s), sorted_indices=False)
    torch.cuda.synchronize()
    assert torch.equal(y_s, y_u)
    rows = np.arange(0, T, 5)
    assert_parity(y_u.reshape(T, N)[torch.from_numpy(rows).cuda()],
                  oracle.gather_qmm_nn(x, *host, idx_s, E, rows=rows), "nn wide sorted")
    idx_b = idx_s.copy()
    idx_b[7, 0] = E + 3
    ws = g.new_workspace(T, N, E)
    y_b = g.gqmm_gather_qmm_nn(xs, *dev, to_dev_idx(idx_b), ws=ws)
    assert g.gqmm_device_status(ws) & g.STATUS_BAD_INDEX
    assert torch.count_nonzero(y_b.reshape(T, N)[7]).item() == 0
    assert torch.equal(y_b.reshape(T, N)[8:], y_u.reshape(T, N)[8:])


@pytest.mark.parametrize("T,A,K,N,E,gs", [(16, 2, 256, 256, 8, 32),
                                          (7, 3, 3000, 1152, 5, 128),   # K not a multiple of 64
                                          (5, 1, 300, 96, 1, 32)])
def test_nn_simt_cross_check_matches_oracle(T, A, K, N, E, gs):
    import quantized_moe_expert_device_gb300 as g

    host, dev = _weights(E, K, N, gs, seed=86)
    x = wl.normal_bf16((T, A, K) if E > 1 else (T, K), 87)
    idx = None if E == 1 else np.random.default_rng(T + K).integers(0, E, size=(T, A)).astype(np.uint32)
    y = g.gqmm_gather_qmm_nn_simt(x.cuda(), *dev, None if idx is None else to_dev_idx(idx), group_size=gs)
    torch.cuda.synchronize()
    assert_parity(y, oracle.gather_qmm_nn(x, *host, idx, E, group_size=gs), f"nn simt T={T} A={A} K={K} N={N}")


def test_nn_rejects_k_not_a_multiple_of_64():
    import quantized_moe_expert_device_gb300 as g

    _, dev = _weights(2, 320 - 32, 128, 64, seed=88)
    x = wl.normal_bf16((4, 288), 89).cuda()
    idx = to_dev_idx(np.zeros((4, 1), np.uint32))
    with pytest.raises(g.GqmmError) as ei:
        g.gqmm_gather_qmm_nn(x, *dev, idx)
    assert ei.value.code == 2


def test_nn_full_size_prefill_shape_sampled_rows():
    """The benchmark's transpose=False workload at full size (E=64, K=2048, N=768, 16384 routed
    rows, unsorted), in the launch configuration the benchmark times: quantized weights bit-equal
    to the oracle's, and a seeded sample of rows (plus one row of every expert) within the
    parity criteria."""
    import quantized_moe_expert_device_gb300 as g

    w = wl.workloads()["nn_e64"]
    host, dev = _weights(w.E, w.H, w.F, w.group_size, seed=wl.SEED_W)
    x = wl.normal_bf16((w.T, w.A, w.H), wl.SEED_X)
    idx = wl.make_idx(w)
    ws = g.new_workspace(w.n, w.F, w.E)
    y = g.gqmm_gather_qmm_nn(x.cuda(), *dev, to_dev_idx(idx), ws=ws)
    assert g.gqmm_device_status(ws) == 0
    rng = np.random.default_rng(3)
    _, first = np.unique(idx.reshape(-1), return_index=True)
    rows = np.array(sorted(set(rng.choice(w.n, size=160, replace=False).tolist()) | set(first.tolist()) | {0, w.n - 1}))
    ref = oracle.gather_qmm_nn(x, *host, idx, w.E, rows=rows)
    assert_parity(y.reshape(w.n, w.F)[torch.from_numpy(rows).cuda()], ref, "nn_e64 full size")
    assert torch.isfinite(y.float()).all()
