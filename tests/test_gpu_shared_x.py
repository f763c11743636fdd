"""x shared by a token's A experts (x [T, H], the x of an MoE layer): every path must give the
result of the same call on x repeated A times ([T, A, H]) bit for bit (the same weights and
kernels, only the x row each routed row reads differs), and match the oracle on the repeated
x.  Paths: wide, narrow, split K, weight streaming, sorted indices, the CUDA-core cross-check,
and the expert MLP."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import assert_parity, to_dev_idx

pytestmark = pytest.mark.gpu


def _weights(shape, gs, seed, std=1.0):
    import quantized_moe_expert_device_gb300 as g

    w = wl.normal_bf16(shape, seed, std=std, chunk_rows=1)
    return oracle.quantize(w, group_size=gs), g.gqmm_quantize(w.cuda(), group_size=gs)


@pytest.mark.parametrize("T,A,H,F,E,gs", [(256, 8, 1024, 512, 16, 64),   # wide
                                          (16, 4, 512, 256, 8, 64),      # narrow
                                          (4, 8, 2048, 768, 64, 64),     # weight streaming (chunks of 2 rows)
                                          (4, 2, 2048, 768, 16, 32),     # narrow with split K
                                          (130, 2, 512, 256, 4, 128),    # wide, ragged
                                          (160, 8, 1024, 384, 4, 64)])   # CTA pairs (320 rows per expert)
def test_shared_x_equals_repeated_x(T, A, H, F, E, gs):
    import quantized_moe_expert_device_gb300 as g

    host, dev = _weights((E, F, H), gs, seed=61)
    x = wl.normal_bf16((T, H), 62)
    x_rep = x.repeat_interleave(A, dim=0).reshape(T, A, H)
    idx = np.random.default_rng(T * A + E).integers(0, E, size=(T, A)).astype(np.uint32)
    d_idx = to_dev_idx(idx)
    ws = g.new_workspace(T * A, F, E)
    y_shared = g.gqmm_gather_qmm(x.cuda(), *dev, d_idx, group_size=gs, ws=ws)
    assert g.gqmm_device_status(ws) == 0
    y_rep = g.gqmm_gather_qmm(x_rep.cuda(), *dev, d_idx, group_size=gs, ws=ws)
    torch.cuda.synchronize()
    assert y_shared.shape == (T, A, F)
    assert torch.equal(y_shared, y_rep)
    assert_parity(y_shared, oracle.gather_qmm(x_rep, *host, idx, E, group_size=gs), f"shared x T={T} A={A} E={E}")
    y_simt = g.gqmm_gather_qmm_simt(x.cuda(), *dev, d_idx, group_size=gs)
    y_simt_rep = g.gqmm_gather_qmm_simt(x_rep.cuda(), *dev, d_idx, group_size=gs)
    torch.cuda.synchronize()
    assert torch.equal(y_simt, y_simt_rep)


def test_shared_x_sorted_indices():
    import quantized_moe_expert_device_gb300 as g

    T, A, H, F, E = 64, 4, 512, 256, 8
    _, dev = _weights((E, F, H), 64, seed=63)
    x = wl.normal_bf16((T, H), 64).cuda()
    idx = np.sort(np.random.default_rng(6).integers(0, E, size=T * A).astype(np.uint32)).reshape(T, A)
    y0 = g.gqmm_gather_qmm(x, *dev, to_dev_idx(idx))
    y1 = g.gqmm_gather_qmm(x, *dev, to_dev_idx(idx), sorted_indices=True)
    y2 = g.gqmm_gather_qmm(x.repeat_interleave(A, dim=0).reshape(T, A, H), *dev, to_dev_idx(idx))
    torch.cuda.synchronize()
    assert torch.equal(y0, y1) and torch.equal(y0, y2)


@pytest.mark.parametrize("T,A,E", [(128, 8, 16), (2, 8, 64)])
def test_moe_mlp_shared_x(T, A, E):
    import quantized_moe_expert_device_gb300 as g

    H, I = 512, 256
    hgu, dgu = _weights((E, 2 * I, H), 64, seed=65, std=H ** -0.5)
    hdn, ddn = _weights((E, H, I), 64, seed=66, std=I ** -0.5)
    x = wl.normal_bf16((T, H), 67)
    x_rep = x.repeat_interleave(A, dim=0).reshape(T, A, H)
    idx = np.random.default_rng(T + E).integers(0, E, size=(T, A)).astype(np.uint32)
    y = g.gqmm_moe_mlp(x.cuda(), dgu, ddn, to_dev_idx(idx))
    y_rep = g.gqmm_moe_mlp(x_rep.cuda(), dgu, ddn, to_dev_idx(idx))
    torch.cuda.synchronize()
    assert y.shape == (T, A, H) and torch.equal(y, y_rep)
    assert_parity(y, oracle.moe_mlp(x_rep, hgu, hdn, idx, E), f"moe_mlp shared x T={T} A={A} E={E}")
