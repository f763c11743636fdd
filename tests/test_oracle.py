"""Pins for the CPU oracle, against facts the pages and the mathematics fix.

None of these re-types the oracle's formulas: each one checks a property, a hand-derived
value, a closed form, a library routine (numpy's stable argsort, bincount, matmul) or a
brute-force loop written independently here.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl


def bf16(values):
    return wl.to_bf16(np.asarray(values, np.float32))


def bits_to_f64(u16: np.ndarray) -> np.ndarray:
    return (u16.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ---------------------------------------------------------------------------------------------
# Quantize
# ---------------------------------------------------------------------------------------------

def test_quantize_packing_order_literal_bytes():
    # A group that is exactly b + s*q with q_k = k mod 16, s = 1, b = 0: codes are k mod 16
    # and the packed bytes, even element in the low nibble, are 0x10, 0x32, ..., 0xfe, repeated.
    q = np.arange(64) % 16
    wq, sc, bs = oracle.quantize(bf16(q[None, :]))
    expected = np.array([0x10, 0x32, 0x54, 0x76, 0x98, 0xBA, 0xDC, 0xFE] * 4, np.uint8)
    assert wq.shape == (1, 32)
    np.testing.assert_array_equal(wq[0], expected)
    assert sc[0, 0] == 0x3F80  # 1.0
    assert bs[0, 0] == 0x0000  # 0.0


def test_quantize_hand_computed_scale_and_bias_bits():
    # min -1, max 2: range 3, 3/15 = 0.2 (float32 0x3E4CCCCD) -> bfloat16 0x3E4D; bias -1 = 0xBF80.
    g = np.zeros(64, np.float32)
    g[0], g[1] = -1.0, 2.0
    wq, sc, bs = oracle.quantize(bf16(g[None, :]))
    assert sc[0, 0] == 0x3E4D
    assert bs[0, 0] == 0xBF80
    # 0 maps to round((0 - (-1)) / 0.2001953125) = round(4.995...) = 5; max maps to 15, min to 0.
    assert wq[0, 0] == (0 | (15 << 4))
    assert (wq[0, 1] & 0xF) == 5


def test_quantize_round_half_to_even():
    # s = 1 (min 0, max 15): (w - b)/s = w exactly; 0.5 -> 0, 1.5 -> 2, 2.5 -> 2, 3.5 -> 4.
    g = np.zeros(64, np.float32)
    g[0], g[1] = 0.0, 15.0
    g[2:6] = [0.5, 1.5, 2.5, 3.5]
    wq, sc, bs = oracle.quantize(bf16(g[None, :]))
    codes = np.stack([wq[0] & 0xF, wq[0] >> 4], axis=1).reshape(-1)
    assert list(codes[2:6]) == [0, 2, 2, 4]


def test_quantize_exactly_representable_groups_round_trip_exactly():
    # w = b + s*q with s a power of two and q hitting 0 and 15 in every group: the stored
    # scale is s, the bias is b, and dequantization gives w back exactly.
    rng = np.random.default_rng(7)
    rows, H = 12, 256
    q = rng.integers(0, 16, size=(rows, H))
    q[:, ::64] = 0
    q[:, 1::64] = 15
    s = 2.0 ** rng.integers(-6, 3, size=(rows, H // 64))
    # b = s*m keeps every b + s*q = s*(m + q) with |m + q| < 256 inside bfloat16's 8 bits
    b = s * rng.integers(-100, 100, size=(rows, H // 64))
    w = b.repeat(64, 1) + s.repeat(64, 1) * q
    wq, sc, bs = oracle.quantize(bf16(w))
    np.testing.assert_array_equal(bits_to_f64(sc), s)
    np.testing.assert_array_equal(bits_to_f64(bs), b)
    np.testing.assert_array_equal(oracle.dequantize(wq, sc, bs), w)
    codes = np.stack([wq & 0xF, wq >> 4], axis=-1).reshape(rows, H)
    np.testing.assert_array_equal(codes, q)


def test_quantize_constant_group():
    g = np.full((2, 64), 0.375, np.float32)
    wq, sc, bs = oracle.quantize(bf16(g))
    assert (sc == 0).all()
    assert (wq == 0).all()
    np.testing.assert_array_equal(oracle.dequantize(wq, sc, bs), g.astype(np.float64))


@pytest.mark.parametrize("std", [1.0, 0.02])
def test_quantize_round_trip_bound_random(std):
    # |w - w_hat| <= s/2 for every element (s the stored scale), codes in [0, 15],
    # each group's minimum maps to code 0 and the bias equals that minimum.
    w = wl.normal_bf16((64, 1024), seed=11, std=std)
    wq, sc, bs = oracle.quantize(w)
    w64 = bits_to_f64(wl.bf16_bits(w))
    what = oracle.dequantize(wq, sc, bs)
    s = bits_to_f64(sc).repeat(64, 1)
    err = np.abs(w64 - what)
    assert (err <= s / 2 * (1 + 1e-6) + 1e-30).all(), float((err - s / 2).max())
    groups = w64.reshape(64, 16, 64)
    np.testing.assert_array_equal(bits_to_f64(bs), groups.min(axis=2))
    codes = np.stack([wq & 0xF, wq >> 4], axis=-1).reshape(64, 16, 64)
    argmin = groups.argmin(axis=2)
    assert (np.take_along_axis(codes, argmin[..., None], 2) == 0).all()
    # the range is 15 steps of the scale, up to the bfloat16 rounding of the scale
    rng_ = groups.max(axis=2) - groups.min(axis=2)
    s_g = bits_to_f64(sc)
    assert (np.abs(15 * s_g - rng_) <= 15 * s_g * 2.0 ** -8 + 1e-30).all()


def test_quantize_rejects_bad_arguments():
    with pytest.raises(ValueError):
        oracle.quantize(bf16(np.zeros((1, 96))))


# ---------------------------------------------------------------------------------------------
# Route sort
# ---------------------------------------------------------------------------------------------

def _check_sort_against_numpy(idx, E):
    perm, offsets, bad = oracle.route_sort(idx, E)
    flat = idx.reshape(-1).astype(np.int64)
    key = np.where(flat < E, flat, E)
    np.testing.assert_array_equal(perm, np.argsort(key, kind="stable"))
    counts = np.bincount(key, minlength=E + 1)
    np.testing.assert_array_equal(offsets, np.concatenate([[0], np.cumsum(counts[:E])]))
    assert bad == counts[E]


@pytest.mark.parametrize("n,E", [(32, 8), (1000, 64), (78, 5), (4096, 256), (17, 1), (0, 4)])
def test_route_sort_matches_stable_argsort(n, E):
    idx = np.random.default_rng(n + E).integers(0, E, size=n, dtype=np.uint32)
    _check_sort_against_numpy(idx, E)


def test_route_sort_edge_cases():
    _check_sort_against_numpy(np.full(100, 3, np.uint32), 8)           # all rows in one expert
    _check_sort_against_numpy(np.arange(64, dtype=np.uint32)[::-1].copy(), 64)  # one row each
    idx = np.array([2, 9, 0, 2, 2**31, 1, 8, 0], np.uint32)            # invalid keys go last
    perm, offsets, bad = oracle.route_sort(idx, 8)
    assert bad == 3  # 9, 2**31 and 8 are all >= E
    assert list(perm) == [2, 7, 5, 0, 3, 1, 4, 6]
    assert list(offsets) == [0, 2, 3, 5, 5, 5, 5, 5, 5]


# ---------------------------------------------------------------------------------------------
# Gather matmul
# ---------------------------------------------------------------------------------------------

def _quantized_tiny(E, F, H, seed):
    w = wl.normal_bf16((E, F, H), seed)
    return oracle.quantize(w)


def _brute_force(x16, wq, sc, bs, idx, E):
    """Direct per-element loops with their own nibble decode (pure Python, tiny inputs)."""
    n, H = x16.shape
    F = wq.shape[1]
    xf = bits_to_f64(x16)
    s = bits_to_f64(sc)
    b = bits_to_f64(bs)
    y = np.zeros((n, F))
    for i in range(n):
        e = int(idx[i])
        if e >= E:
            continue
        for f in range(F):
            acc = 0.0
            for h in range(H):
                byte = int(wq[e, f, h // 2])
                code = (byte >> (4 * (h % 2))) & 15
                acc += xf[i, h] * (s[e, f, h // 64] * code + b[e, f, h // 64])
            y[i, f] = acc
    return y


def test_gather_brute_force_tiny():
    E, F, H, n = 3, 4, 128, 8
    wq, sc, bs = _quantized_tiny(E, F, H, seed=5)
    x = wl.normal_bf16((n, H), seed=6)
    idx = np.array([2, 0, 1, 1, 0, 2, 2, 1], np.uint32)
    y = oracle.gather_qmm(x, wq, sc, bs, idx, E)
    ref = _brute_force(wl.bf16_bits(x), wq, sc, bs, idx, E)
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_gather_matches_numpy_matmul_on_independently_dequantized_weights():
    E, F, H, n = 8, 128, 256, 32
    wq, sc, bs = _quantized_tiny(E, F, H, seed=2)
    x = wl.normal_bf16((n, H), seed=1)
    idx = wl.idx_uniform(16, 2, E)
    # independent vectorized dequantization with numpy bit operations
    codes = np.stack([wq & 0xF, wq >> 4], axis=-1).reshape(E, F, H).astype(np.float64)
    what = codes * bits_to_f64(sc).repeat(64, 2) + bits_to_f64(bs).repeat(64, 2)
    xf = bits_to_f64(wl.bf16_bits(x))
    ref = np.stack([xf[i] @ what[int(e)].T for i, e in enumerate(idx.reshape(-1))])
    y = oracle.gather_qmm(x, wq, sc, bs, idx, E)
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-10)


def test_gather_closed_form_one_hot_rows():
    # w[e, f, h] = (e - 4) + ((f + h) mod 16) / 4 quantizes exactly (each 64-run holds every
    # residue).  A one-hot x at h0 selects w[idx, f, h0]; an all-ones x sums a row:
    # H*(e - 4) + (H/16) * 120 / 4.
    E, F, H = 5, 16, 128
    e_ = np.arange(E)[:, None, None]
    f_ = np.arange(F)[None, :, None]
    h_ = np.arange(H)[None, None, :]
    w = (e_ - 4) + ((f_ + h_) % 16) / 4.0
    wq, sc, bs = oracle.quantize(bf16(w))
    rows = []
    idx = []
    expect = []
    for i, (e, h0) in enumerate([(0, 0), (3, 17), (4, 127), (1, 64), (2, 5)]):
        x = np.zeros(H)
        x[h0] = 1.0
        rows.append(x)
        idx.append(e)
        expect.append([(e - 4) + ((f + h0) % 16) / 4.0 for f in range(F)])
    for e in range(E):
        rows.append(np.ones(H))
        idx.append(e)
        expect.append([H * (e - 4) + (H / 16) * 120 / 4.0] * F)
    y = oracle.gather_qmm(bf16(np.array(rows)), wq, sc, bs, np.array(idx, np.uint32), E)
    np.testing.assert_array_equal(y, np.array(expect))


def test_gather_sorted_equals_unsorted_and_dense_equals_e1():
    E, F, H = 8, 128, 256
    wq, sc, bs = _quantized_tiny(E, F, H, seed=2)
    x = wl.normal_bf16((16, 2, H), seed=1)
    idx = wl.idx_uniform(16, 2, E)
    y = oracle.gather_qmm(x, wq, sc, bs, idx, E)
    xs, idx_s, order = wl.sorted_by_expert(x, idx)
    ys = oracle.gather_qmm(xs, wq, sc, bs, idx_s, E)
    np.testing.assert_array_equal(ys, y[order])
    # E = 1: idx all zero equals the dense call with no index
    y1 = oracle.gather_qmm(x, wq[:1], sc[:1], bs[:1], np.zeros(32, np.uint32), 1)
    yd = oracle.gather_qmm(x, wq[:1], sc[:1], bs[:1], None, 1)
    np.testing.assert_array_equal(y1, yd)


def test_gather_duplicated_expert_gives_identical_rows_and_bad_index_gives_zero():
    E, F, H = 4, 32, 128
    wq, sc, bs = _quantized_tiny(E, F, H, seed=9)
    wq[3], sc[3], bs[3] = wq[1], sc[1], bs[1]
    x = wl.normal_bf16((6, H), seed=3)
    xx = torch.cat([x[:3], x[:3]])
    idx = np.array([1, 1, 1, 3, 3, 3], np.uint32)
    y = oracle.gather_qmm(xx, wq, sc, bs, idx, E)
    np.testing.assert_array_equal(y[:3], y[3:])
    y_bad = oracle.gather_qmm(x, wq, sc, bs, np.array([0, 7, 1, 4, 2, 3], np.uint32), E)
    assert (y_bad[1] == 0).all() and (y_bad[3] == 0).all()
    assert (y_bad[0] != 0).any()


def test_gather_rows_subset_matches_full():
    E, F, H = 8, 64, 256
    wq, sc, bs = _quantized_tiny(E, F, H, seed=4)
    x = wl.normal_bf16((40, H), seed=8)
    idx = np.random.default_rng(1).integers(0, E, 40, dtype=np.uint32)
    y = oracle.gather_qmm(x, wq, sc, bs, idx, E, nthreads=3)
    rows = np.array([39, 0, 17, 17, 5])
    yr = oracle.gather_qmm(x, wq, sc, bs, idx, E, rows=rows)
    np.testing.assert_array_equal(yr, y[rows])


def test_golden_tiny_fixture():
    """Regression pin: the committed fixture written by tests/golden/make_golden.py from the
    oracle for the tiny workload (T=16, A=2, H=256, F=128, E=8, seeds 1/2/3)."""
    import json
    import os

    path = os.path.join(os.path.dirname(__file__), "golden", "tiny_oracle.json")
    with open(path) as fh:
        g = json.load(fh)
    w = wl.workloads()["tiny"]
    inp = wl.make_inputs(w)
    wq, sc, bs = oracle.quantize(inp["w"])
    assert int(wq.astype(np.uint64).sum()) == g["wq_sum"]
    assert [int(v) for v in sc.reshape(-1)[:8]] == g["scales_head"]
    assert [int(v) for v in bs.reshape(-1)[:8]] == g["biases_head"]
    perm, offsets, _ = oracle.route_sort(inp["idx"], w.E)
    assert [int(v) for v in offsets] == g["offsets"]
    y = oracle.gather_qmm(inp["x"], wq, sc, bs, inp["idx"], w.E)
    np.testing.assert_allclose(y[0, :8], g["y_row0_head"], rtol=0, atol=1e-9)
    np.testing.assert_allclose(float(np.abs(y).sum()), g["y_abs_sum"], rtol=1e-12)
