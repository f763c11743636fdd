"""gqmm_quantize on the GPU vs the CPU oracle: packed codes, scales and biases bit-exact."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import np_of

pytestmark = pytest.mark.gpu


def _check(w_cpu):
    import quantized_moe_expert_device_gb300 as g

    wq, sc, bs = g.gqmm_quantize(w_cpu.cuda())
    torch.cuda.synchronize()
    rq, rs, rb = oracle.quantize(w_cpu)
    np.testing.assert_array_equal(np_of(wq), rq)
    np.testing.assert_array_equal(np_of(sc), rs)
    np.testing.assert_array_equal(np_of(bs), rb)


def test_quantize_tiny_config_bit_exact():
    w = wl.workloads()["tiny"]
    _check(wl.normal_bf16((w.E, w.F, w.H), wl.SEED_W))


@pytest.mark.parametrize("std", [1.0, 0.02, 300.0])
def test_quantize_random_scales_bit_exact(std):
    _check(wl.normal_bf16((37, 3, 512), seed=5, std=std))


def test_quantize_special_groups_bit_exact():
    rng = np.random.default_rng(0)
    rows = []
    rows.append(np.full(128, 1.5, np.float32))                     # constant groups
    rows.append(np.tile(np.arange(16, dtype=np.float32), 8))       # exact codes, scale 1
    r = np.zeros(128, np.float32)
    r[2:6] = [0.5, 1.5, 2.5, 3.5]
    r[1] = 15.0
    rows.append(r)                                                  # ties to even
    rows.append(rng.standard_normal(128).astype(np.float32) * 1e-30)  # tiny magnitudes
    rows.append(-np.abs(rng.standard_normal(128).astype(np.float32)) * 1e4)
    _check(wl.to_bf16(np.stack(rows)))


def test_quantize_prefill_shape_bit_exact():
    w = wl.workloads()["prefill_e64"]
    _check(wl.normal_bf16((w.E, w.F, w.H), wl.SEED_W, chunk_rows=1))


def test_quantize_rejects_unsupported():
    import quantized_moe_expert_device_gb300 as g

    w = torch.zeros(4, 96, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(g.GqmmError):
        g.gqmm_quantize(w)
    with pytest.raises(g.GqmmError):  # group sizes are 32, 64 and 128
        g.gqmm_quantize(torch.zeros(4, 128, dtype=torch.bfloat16, device="cuda"), group_size=96)
    with pytest.raises(g.GqmmError):  # H must be a multiple of the group size
        g.gqmm_quantize(torch.zeros(4, 192, dtype=torch.bfloat16, device="cuda"), group_size=128)
    with pytest.raises(g.GqmmError):  # code widths are 2, 3, 4, 5, 6 and 8
        g.gqmm_quantize(torch.zeros(4, 128, dtype=torch.bfloat16, device="cuda"), bits=7)
    with pytest.raises(g.GqmmError):  # widths other than 4 take 64-wide groups only
        g.gqmm_quantize(torch.zeros(4, 128, dtype=torch.bfloat16, device="cuda"), group_size=128, bits=8)
