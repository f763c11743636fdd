"""32- and 128-wide quantization groups on the GPU: quantize bit for bit against the oracle,
and gqmm_gather_qmm / gqmm_moe_mlp within the parity criteria against the oracle's float64
results.  Cases cover the wide and narrow tensor-core variants, split K on decode-sized calls
(the weight-streaming kernels take only 64-wide groups, so those calls run on the narrow
variant), scale rows loaded eight groups at a time (H/gs a multiple of 8) and one at a time
(H/gs = 3 or 6), dense E=1, and the CUDA-core cross-check."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import assert_parity, np_of, to_dev_idx

pytestmark = pytest.mark.gpu


def _weights(shape, gs, seed, std=1.0):
    import quantized_moe_expert_device_gb300 as g

    w = wl.normal_bf16(shape, seed, std=std, chunk_rows=1)
    host = oracle.quantize(w, group_size=gs)
    dev = g.gqmm_quantize(w.cuda(), group_size=gs)
    torch.cuda.synchronize()
    for d, h in zip(dev, host):
        np.testing.assert_array_equal(np_of(d), h)  # the GPU's codes, scales and biases are the oracle's
    return host, dev


_GROUP_SHAPES = [(256, 8, 1024, 512, 8),    # wide, H/gs a multiple of 8
                 (32, 2, 1024, 256, 8),     # narrow
                 (4, 2, 2048, 768, 16),     # decode-sized: narrow with split K
                 (64, 2, 384, 128, 4),      # H/128 = 3 scale groups per row
                 (40, 1, 192, 128, 1),      # dense; H/32 = 6 (192 is no multiple of 128: 32 only)
                 (3, 1, 1024, 256, 1)]      # dense decode-sized


@pytest.mark.parametrize("gs,T,A,H,F,E", [(gs,) + s for gs in (32, 128) for s in _GROUP_SHAPES if s[2] % gs == 0])
def test_gather_group_sizes_match_oracle(gs, T, A, H, F, E):
    import quantized_moe_expert_device_gb300 as g

    host, dev = _weights((E, F, H), gs, seed=41 + gs)
    x = wl.normal_bf16((T, A, H) if E > 1 else (T, H), 43)
    idx = None if E == 1 else np.random.default_rng(T + gs).integers(0, E, size=(T, A)).astype(np.uint32)
    ws = g.new_workspace(T * A, F, E)
    y = g.gqmm_gather_qmm(x.cuda(), *dev, None if idx is None else to_dev_idx(idx), group_size=gs, ws=ws)
    assert g.gqmm_device_status(ws) == 0
    ref = oracle.gather_qmm(x, *host, idx, E, group_size=gs)
    assert_parity(y, ref, f"gs={gs} T={T} A={A} H={H} F={F} E={E}")
    y_simt = g.gqmm_gather_qmm_simt(x.cuda(), *dev, None if idx is None else to_dev_idx(idx), group_size=gs)
    torch.cuda.synchronize()
    assert_parity(y_simt, ref, f"simt gs={gs}")


@pytest.mark.parametrize("gs", [32, 128])
def test_group_sizes_sorted_equals_unsorted_bitwise(gs):
    import quantized_moe_expert_device_gb300 as g

    T, A, H, F, E = 96, 4, 512, 256, 6
    _, dev = _weights((E, F, H), gs, seed=47)
    idx = np.sort(np.random.default_rng(5).integers(0, E, size=T * A).astype(np.uint32)).reshape(T, A)
    x = wl.normal_bf16((T, A, H), 48).cuda()
    y0 = g.gqmm_gather_qmm(x, *dev, to_dev_idx(idx), group_size=gs)
    y1 = g.gqmm_gather_qmm(x, *dev, to_dev_idx(idx), group_size=gs, sorted_indices=True)
    torch.cuda.synchronize()
    assert torch.equal(y0, y1)


@pytest.mark.parametrize("gs", [32, 128])
@pytest.mark.parametrize("T,A,E", [(128, 4, 8), (2, 8, 64)])
def test_moe_mlp_group_sizes_match_oracle(gs, T, A, E):
    import quantized_moe_expert_device_gb300 as g

    H, I = 512, 256
    hgu, dgu = _weights((E, 2 * I, H), gs, seed=51, std=H ** -0.5)
    hdn, ddn = _weights((E, H, I), gs, seed=52, std=I ** -0.5)
    x = wl.normal_bf16((T, A, H), 53)
    idx = np.random.default_rng(T * E).integers(0, E, size=(T, A)).astype(np.uint32)
    ws = g.new_mlp_workspace(T * A, H, I, E)
    y = g.gqmm_moe_mlp(x.cuda(), dgu, ddn, to_dev_idx(idx), group_size=gs, ws=ws)
    assert g.gqmm_device_status(ws) == 0
    ref = oracle.moe_mlp(x, hgu, hdn, idx, E, group_size=gs)
    assert_parity(y, ref, f"moe_mlp gs={gs} T={T} A={A} E={E}")


def test_group_size_mismatch_is_rejected_by_the_binding():
    import quantized_moe_expert_device_gb300 as g

    _, dev = _weights((2, 64, 256), 64, seed=55)
    x = wl.normal_bf16((4, 256), 56).cuda()
    with pytest.raises(ValueError):
        g.gqmm_gather_qmm(x, *dev, to_dev_idx(np.zeros((4, 1), np.uint32)), group_size=128)
