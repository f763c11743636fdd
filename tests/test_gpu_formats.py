"""The other weight formats on the GPU against the oracle: affine codes of 2, 3, 5, 6 and 8 bits
(64-wide groups) and the block-scaled floating-point modes mxfp4, nvfp4 and mxfp8.

Quantization is bit-exact (codes, scales, biases, nvfp4 tensor scales).  The gather meets the
same tolerances as the 4-bit path (relative Frobenius error <= 5e-3, every element within
2e-2 * max|y_ref|): every format's weights are decoded exactly and rounded once to bfloat16 (the
nvfp4 product S * t, and element * (S * t), in float32 first), as the 4-bit affine weights are,
so the expected error is the same ~1.6e-3.  Cases cover the wide variant (128 rows per expert:
2-bit, mxfp4, nvfp4), the narrow one (16 rows per expert; every format), a decode-sized call with
K split, a dense call, an invalid index, and sorted == unsorted bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import assert_parity, np_of, to_dev_idx

pytestmark = pytest.mark.gpu

BITS = [2, 3, 5, 6, 8]
MODES = ["mxfp4", "nvfp4", "mxfp8"]


def _dev_affine(q):
    wq, sc, bs = q
    return (torch.from_numpy(wq).cuda(), torch.from_numpy(sc.view(np.int16)).cuda().view(torch.bfloat16),
            torch.from_numpy(bs.view(np.int16)).cuda().view(torch.bfloat16))


@pytest.mark.parametrize("bits", BITS)
def test_quantize_other_bit_widths_bit_exact(bits):
    import quantized_moe_expert_device_gb300 as g

    w = wl.normal_bf16((3, 80, 512), 60 + bits, chunk_rows=1)
    w[0, 0, :64] = 0.5  # a constant group: scale 0, codes 0
    wq, sc, bs = g.gqmm_quantize(w.cuda(), group_size=64, bits=bits)
    rq, rs, rb = oracle.quantize(w, group_size=64, bits=bits)
    torch.cuda.synchronize()
    assert np.array_equal(np_of(wq), rq)
    assert np.array_equal(np_of(sc), rs) and np.array_equal(np_of(bs), rb)


@pytest.mark.parametrize("mode", MODES)
def test_quantize_fp_modes_bit_exact(mode):
    import quantized_moe_expert_device_gb300 as g

    w = wl.normal_bf16((3, 80, 512), 70, std=0.5, chunk_rows=1)
    w[1] = 0.0                       # an all-zero expert: nvfp4 tensor scale 1, every code 0
    w[0, 0, :32] = torch.tensor([2.5, 5.0, 0.25, 0.75, 1.25, 1.75, -2.5, 7.0, 6.5, 3.5] + [0.0] * 22)  # ties, saturation
    w[2, 3, 64:96] = 2.0 ** -120     # tiny values
    wq, sc, ts = g.gqmm_quantize_fp(w.cuda(), mode)
    rq, rs, rts = oracle.quantize_fp(w, mode)
    torch.cuda.synchronize()
    assert np.array_equal(np_of(wq), rq)
    assert np.array_equal(np_of(sc), rs)
    if mode == "nvfp4":
        assert np.array_equal(ts.cpu().numpy(), rts)
    else:
        assert ts is None


def _run_affine(bits, T, A, E, F, H, idx, sorted_indices=False, seed=0):
    import quantized_moe_expert_device_gb300 as g

    w = wl.normal_bf16((E, F, H), 80 + seed, chunk_rows=1)
    q = oracle.quantize(w, group_size=64, bits=bits)
    x = wl.normal_bf16((T, A, H) if idx is not None else (T, H), 81 + seed)
    ws = g.new_workspace(T * A, F, E)
    y = g.gqmm_gather_qmm(x.cuda(), *_dev_affine(q), None if idx is None else to_dev_idx(idx), group_size=64,
                          bits=bits, sorted_indices=sorted_indices, ws=ws)
    status = g.gqmm_device_status(ws)
    return y, oracle.gather_qmm(x, *q, idx, E, group_size=64, bits=bits), status


def _run_fp(mode, T, A, E, F, H, idx, sorted_indices=False, seed=0, quantize_on_gpu=False):
    import quantized_moe_expert_device_gb300 as g

    w = wl.normal_bf16((E, F, H), 90 + seed, std=0.1, chunk_rows=1)
    wq, sc, ts = oracle.quantize_fp(w, mode)
    if quantize_on_gpu:
        dev = g.gqmm_quantize_fp(w.cuda(), mode)
    else:
        dev = (torch.from_numpy(wq).cuda(), torch.from_numpy(sc).cuda(),
               None if ts is None else torch.from_numpy(ts).cuda())
    x = wl.normal_bf16((T, A, H) if idx is not None else (T, H), 91 + seed)
    ws = g.new_workspace(T * A, F, E)
    y = g.gqmm_gather_qmm_fp(x.cuda(), *dev, None if idx is None else to_dev_idx(idx), mode,
                             sorted_indices=sorted_indices, ws=ws)
    status = g.gqmm_device_status(ws)
    return y, oracle.gather_qmm_fp(x, wq, sc, ts, idx, E, mode), status


# (T, A, E, F, H): 128 rows per expert (wide where the format has it), 16 rows per expert
# (narrow), a decode-sized call that splits K, and F not a multiple of the 128-row tile
SHAPES = [(64, 8, 4, 256, 1024), (32, 4, 8, 384, 512), (2, 4, 4, 256, 2048), (48, 2, 6, 144, 256)]


@pytest.mark.parametrize("bits", BITS)
@pytest.mark.parametrize("T,A,E,F,H", SHAPES)
def test_gather_other_bit_widths_match_oracle(bits, T, A, E, F, H):
    if (H * bits // 8) % 16:
        H *= 2  # a row's codes must fill whole 16-byte units (3- and 5-bit codes: H a multiple of 128)
    idx = np.random.default_rng(T + bits).integers(0, E, size=(T, A)).astype(np.uint32)
    y, ref, status = _run_affine(bits, T, A, E, F, H, idx, seed=bits)
    assert status == 0
    assert_parity(y.reshape(-1, F), ref, f"bits={bits} T={T} A={A} E={E} F={F} H={H}")


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("T,A,E,F,H", SHAPES)
def test_gather_fp_modes_match_oracle(mode, T, A, E, F, H):
    idx = np.random.default_rng(T + 7).integers(0, E, size=(T, A)).astype(np.uint32)
    y, ref, status = _run_fp(mode, T, A, E, F, H, idx, seed=3)
    assert status == 0
    assert_parity(y.reshape(-1, F), ref, f"{mode} T={T} A={A} E={E} F={F} H={H}")


@pytest.mark.parametrize("fmt", ["bits3", "bits8", "mxfp4", "nvfp4", "mxfp8"])
def test_formats_dense_invalid_index_and_sorted(fmt):
    """Dense (E = 1) calls; an invalid index gives a zero row and the status bit; a caller-sorted
    call equals the unsorted one bit for bit."""
    import quantized_moe_expert_device_gb300 as g

    run = (lambda *a, **k: _run_affine(int(fmt[4:]), *a, **k)) if fmt.startswith("bits") else \
        (lambda *a, **k: _run_fp(fmt, *a, **k))
    F, H = 160, 512
    y, ref, status = run(40, 1, 1, F, H, None, seed=5)
    assert status == 0
    assert_parity(y, ref, f"{fmt} dense")
    T, A, E = 24, 4, 6
    idx = np.random.default_rng(11).integers(0, E, size=(T, A)).astype(np.uint32)
    idx[3, 2] = E + 2
    y, ref, status = run(T, A, E, F, H, idx, seed=6)
    assert status & g.STATUS_BAD_INDEX
    assert_parity(y.reshape(-1, F), ref, f"{fmt} invalid index")
    assert torch.count_nonzero(y.reshape(-1, F)[3 * A + 2]).item() == 0
    # the same rows and indices (nondecreasing) through the sorted-route plan and the unsorted
    # route sort: equal bit for bit
    idx_s = np.sort(np.random.default_rng(12).integers(0, E, size=T * A)).astype(np.uint32).reshape(-1, 1)
    y_s, _, st = run(T * A, 1, E, F, H, idx_s, sorted_indices=True, seed=7)
    y_u, _, _ = run(T * A, 1, E, F, H, idx_s, sorted_indices=False, seed=7)
    assert st == 0
    assert torch.equal(y_s, y_u)


@pytest.mark.parametrize("mode", ["mxfp4", "nvfp4"])
def test_fp_modes_on_gpu_quantized_weights(mode):
    """The gather on weights quantized by gqmm_quantize_fp (bit-exact above) at a prefill-like
    shape on the wide variant."""
    T, A, E, F, H = 256, 8, 16, 512, 2048
    idx = wl.idx_uniform(T, A, E, seed=13)
    y, ref, status = _run_fp(mode, T, A, E, F, H, idx, seed=8, quantize_on_gpu=True)
    assert status == 0
    assert_parity(y.reshape(-1, F), ref, f"{mode} prefill-like, GPU-quantized")
