"""gqmm_route_sort on the GPU vs the CPU oracle: perm and offsets bit-exact."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import to_dev_idx

pytestmark = pytest.mark.gpu


def _check(idx: np.ndarray, E: int, expect_bad: bool = False):
    import quantized_moe_expert_device_gb300 as g

    n = idx.size
    ws = g.new_workspace(n, 1, E)
    perm, offsets = g.gqmm_route_sort(to_dev_idx(idx.reshape(-1)), E, ws=ws)
    status = g.gqmm_device_status(ws)
    rp, ro, bad = oracle.route_sort(idx, E)
    np.testing.assert_array_equal(perm.cpu().numpy(), rp)
    np.testing.assert_array_equal(offsets.cpu().numpy(), ro)
    assert bool(status & g.STATUS_BAD_INDEX) == (bad > 0) == expect_bad


@pytest.mark.parametrize("name", ["tiny", "prefill_e64", "mixtral", "decode_moe_m1", "decode_moe_m8"]
                         + [f"sweep_r{r}" for r in (4, 16, 128)])
def test_route_sort_workloads(name):
    w = wl.workloads()[name]
    _check(wl.make_idx(w), w.E)


# sizes on both sides of the single-block route limits (256 and 4096 entries, E = 256), of the
# 1024-entry tiles of the two-kernel route and of its switch to 2048-entry tiles (n > 65536)
@pytest.mark.parametrize("n,E", [(1, 1), (77, 1), (78, 4), (2047, 3), (2048, 64), (2049, 64),
                                 (6000, 1024), (40000, 257), (5, 1024), (4096, 256), (4097, 256),
                                 (4096, 257), (16384, 256), (9999, 255), (33, 256), (1025, 300),
                                 (65536, 64), (65537, 64), (70001, 1000), (255, 256), (256, 256),
                                 (257, 256), (256, 257), (200, 3), (64, 128)])
def test_route_sort_sizes(n, E):
    idx = np.random.default_rng(n * 7 + E).integers(0, E, size=n, dtype=np.uint32)
    _check(idx, E)


def test_route_sort_all_rows_one_expert_and_empty_experts():
    _check(np.full(5000, 7, np.uint32), 64)
    idx = np.random.default_rng(1).integers(0, 4, size=3000, dtype=np.uint32) * 16
    _check(idx, 64)


@pytest.mark.parametrize("n", [200, 4100, 20000])
def test_route_sort_invalid_indices_go_last_and_flag(n):
    idx = np.random.default_rng(2).integers(0, 12, size=n, dtype=np.uint32)
    idx[::97] = 2**31 + 5
    idx[1] = 10  # == E: also invalid
    _check(idx, 10, expect_bad=True)


def test_route_sort_repeatable_on_reused_workspace():
    import quantized_moe_expert_device_gb300 as g

    idx = to_dev_idx(wl.idx_uniform(2048, 8, 64))
    ws = g.new_workspace(idx.numel(), 1, 64)
    p1, o1 = g.gqmm_route_sort(idx, 64, ws=ws)
    p2, o2 = g.gqmm_route_sort(idx, 64, ws=ws)
    assert torch.equal(p1, p2) and torch.equal(o1, o2)
    assert g.gqmm_device_status(ws) == 0
