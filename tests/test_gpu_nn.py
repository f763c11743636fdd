"""gqmm_gather_qmm_nn (transpose=False: W[e] = [K, N] quantized along N) on the GPU against the
oracle's float64 gather_qmm_nn, on the GPU's own quantized weights (bit-equal to the oracle's):
the shape of the pages' transpose=False timing (E=4, K=N=512, 1024 rows), every group size, K
over several 1024-wide x chunks with a ragged tail, N not a multiple of the 1024-column block,
dense E=1, invalid indices and a shared x."""
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


@pytest.mark.parametrize("T,A,K,N,E,gs", [(1024, 1, 512, 512, 4, 64),    # the pages' transpose=False shape
                                          (16, 2, 256, 256, 8, 32),
                                          (7, 3, 3000, 1152, 5, 128),    # K: three x chunks, ragged; N: 1.1 blocks
                                          (4, 8, 2048, 768, 64, 64),
                                          (5, 1, 300, 96, 1, 32)])       # dense (idx None)
def test_nn_matches_oracle(T, A, K, N, E, gs):
    import quantized_moe_expert_device_gb300 as g

    host, dev = _weights(E, K, N, gs, seed=81)
    x = wl.normal_bf16((T, A, K) if E > 1 else (T, K), 82)
    idx = None if E == 1 else np.random.default_rng(T + K).integers(0, E, size=(T, A)).astype(np.uint32)
    y = g.gqmm_gather_qmm_nn(x.cuda(), *dev, None if idx is None else to_dev_idx(idx), group_size=gs)
    torch.cuda.synchronize()
    assert y.shape[-1] == N
    assert_parity(y, oracle.gather_qmm_nn(x, *host, idx, E, group_size=gs), f"nn T={T} A={A} K={K} N={N} E={E}")


def test_nn_invalid_indices_and_shared_x():
    import quantized_moe_expert_device_gb300 as g

    T, A, K, N, E = 12, 4, 512, 256, 6
    host, dev = _weights(E, K, N, 64, seed=83)
    x = wl.normal_bf16((T, K), 84)
    idx = np.random.default_rng(8).integers(0, E, size=(T, A)).astype(np.uint32)
    idx[::3, 2] = E + 1
    y = g.gqmm_gather_qmm_nn(x.cuda(), *dev, to_dev_idx(idx))           # x [T, K] shared by the A rows
    x_rep = x.repeat_interleave(A, dim=0).reshape(T, A, K)
    y_rep = g.gqmm_gather_qmm_nn(x_rep.cuda(), *dev, to_dev_idx(idx))
    torch.cuda.synchronize()
    assert y.shape == (T, A, N) and torch.equal(y, y_rep)
    assert not y[::3, 2].float().abs().sum().item()
    assert_parity(y, oracle.gather_qmm_nn(x_rep, *host, idx, E), "nn invalid + shared")
