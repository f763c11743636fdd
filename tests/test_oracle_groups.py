"""Pins for the oracle at the other group sizes of the affine 4-bit format (32 and 128 weights
per scale and bias along H; 64 is pinned in test_oracle.py): exact round trips, the
quantization error bound, and the gather matmul against a brute-force loop and against numpy
matmul on weights dequantized here with numpy bit operations.  Nothing here calls the oracle's
own dequantization for the expected values."""
import numpy as np
import pytest

import oracle
import workloads as wl

GROUPS = [32, 128]


def bf16(values):
    return wl.to_bf16(np.asarray(values, np.float32))


def bits_to_f64(u16):
    return (np.asarray(u16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@pytest.mark.parametrize("gs", GROUPS)
def test_quantize_exact_groups_round_trip(gs):
    # w = b + s q with s a power of two and q reaching 0 and 15 in every group
    rng = np.random.default_rng(17)
    rows, H = 6, 256
    q = rng.integers(0, 16, size=(rows, H))
    q[:, ::gs] = 0
    q[:, 1::gs] = 15
    s = 2.0 ** rng.integers(-6, 3, size=(rows, H // gs))
    b = s * rng.integers(-100, 100, size=(rows, H // gs))
    w = b.repeat(gs, 1) + s.repeat(gs, 1) * q
    wq, sc, bs = oracle.quantize(bf16(w), group_size=gs)
    assert sc.shape == (rows, H // gs)
    np.testing.assert_array_equal(bits_to_f64(sc), s)
    np.testing.assert_array_equal(bits_to_f64(bs), b)
    codes = np.stack([wq & 0xF, wq >> 4], axis=-1).reshape(rows, H)
    np.testing.assert_array_equal(codes, q)


@pytest.mark.parametrize("gs", GROUPS)
def test_quantize_error_bound_and_minimum_code(gs):
    w = wl.normal_bf16((32, 512), seed=19)
    wq, sc, bs = oracle.quantize(w, group_size=gs)
    w64 = bits_to_f64(wl.bf16_bits(w))
    codes = np.stack([wq & 0xF, wq >> 4], axis=-1).reshape(32, 512).astype(np.float64)
    s = bits_to_f64(sc).repeat(gs, 1)
    b = bits_to_f64(bs).repeat(gs, 1)
    err = np.abs(w64 - (s * codes + b))
    assert (err <= s / 2 * (1 + 1e-6) + 1e-30).all()
    groups = w64.reshape(32, 512 // gs, gs)
    np.testing.assert_array_equal(bits_to_f64(bs), groups.min(axis=2))
    argmin = groups.argmin(axis=2)
    assert (np.take_along_axis(codes.reshape(32, 512 // gs, gs), argmin[..., None], 2) == 0).all()


def _quantized(E, F, H, gs, seed):
    return oracle.quantize(wl.normal_bf16((E, F, H), seed=seed), group_size=gs)


@pytest.mark.parametrize("gs", GROUPS)
def test_gather_brute_force(gs):
    E, F, H, n = 3, 4, 256, 6
    wq, sc, bs = _quantized(E, F, H, gs, seed=23)
    x = wl.normal_bf16((n, H), seed=24)
    idx = np.array([1, 0, 2, 2, 5, 1], np.uint32)  # 5 >= E: a zero row
    y = oracle.gather_qmm(x, wq, sc, bs, idx, E, group_size=gs)
    xf = bits_to_f64(wl.bf16_bits(x))
    s, b = bits_to_f64(sc), bits_to_f64(bs)
    ref = np.zeros((n, F))
    for i in range(n):
        e = int(idx[i])
        if e >= E:
            continue
        for f in range(F):
            acc = 0.0
            for h in range(H):
                code = (int(wq[e, f, h // 2]) >> (4 * (h % 2))) & 15
                acc += xf[i, h] * (s[e, f, h // gs] * code + b[e, f, h // gs])
            ref[i, f] = acc
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)
    assert not y[4].any()


@pytest.mark.parametrize("gs", GROUPS)
def test_gather_matches_numpy_matmul(gs):
    E, F, H, n = 4, 64, 512, 24
    wq, sc, bs = _quantized(E, F, H, gs, seed=29)
    x = wl.normal_bf16((n, H), seed=30)
    idx = np.random.default_rng(31).integers(0, E, size=n).astype(np.uint32)
    codes = np.stack([wq & 0xF, wq >> 4], axis=-1).reshape(E, F, H).astype(np.float64)
    what = codes * bits_to_f64(sc).repeat(gs, 2) + bits_to_f64(bs).repeat(gs, 2)
    xf = bits_to_f64(wl.bf16_bits(x))
    ref = np.stack([what[int(e)] @ xf[i] for i, e in enumerate(idx)])
    np.testing.assert_allclose(oracle.gather_qmm(x, wq, sc, bs, idx, E, group_size=gs), ref, rtol=1e-12, atol=1e-10)


@pytest.mark.parametrize("gs", GROUPS)
def test_group_size_changes_the_result(gs):
    # the same weights quantized with 64-wide groups and with gs-wide groups differ (a wrong
    # group stride in either would make them agree only by accident)
    w = wl.normal_bf16((2, 16, 256), seed=37)
    q64 = oracle.quantize(w)
    qg = oracle.quantize(w, group_size=gs)
    assert qg[1].shape[-1] == 256 // gs and not np.array_equal(q64[0], qg[0])
