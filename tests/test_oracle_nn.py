"""Pins for the oracle's transpose=False gather (y[i] = x[i] . deq(W[idx[i]]), W[e] = [K, N]
quantized along N): a brute-force loop with its own nibble decode, numpy matmul on weights
dequantized here with numpy bit operations, and a closed form on exactly representable
weights.  None of these calls the oracle's own dequantization for the expected values."""
import numpy as np
import pytest

import oracle
import workloads as wl


def bits_to_f64(u16):
    return (np.asarray(u16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@pytest.mark.parametrize("gs", [32, 64, 128])
def test_nn_brute_force(gs):
    E, K, N, n = 3, 8, 128, 5
    wq, sc, bs = oracle.quantize(wl.normal_bf16((E, K, N), 71), group_size=gs)
    x = wl.normal_bf16((n, K), 72)
    idx = np.array([2, 0, 7, 1, 2], np.uint32)  # 7 >= E: a zero row
    y = oracle.gather_qmm_nn(x, wq, sc, bs, idx, E, group_size=gs)
    xf = bits_to_f64(wl.bf16_bits(x))
    s, b = bits_to_f64(sc), bits_to_f64(bs)
    ref = np.zeros((n, N))
    for i in range(n):
        e = int(idx[i])
        if e >= E:
            continue
        for c in range(N):
            acc = 0.0
            for k in range(K):
                code = (int(wq[e, k, c // 2]) >> (4 * (c % 2))) & 15
                acc += xf[i, k] * (s[e, k, c // gs] * code + b[e, k, c // gs])
            ref[i, c] = acc
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)
    assert not y[2].any()


def test_nn_matches_numpy_matmul():
    E, K, N, n = 4, 256, 192, 40
    wq, sc, bs = oracle.quantize(wl.normal_bf16((E, K, N), 73))
    x = wl.normal_bf16((n, K), 74)
    idx = np.random.default_rng(75).integers(0, E, size=n).astype(np.uint32)
    codes = np.stack([wq & 0xF, wq >> 4], axis=-1).reshape(E, K, N).astype(np.float64)
    what = codes * bits_to_f64(sc).repeat(64, 2) + bits_to_f64(bs).repeat(64, 2)
    xf = bits_to_f64(wl.bf16_bits(x))
    ref = np.stack([xf[i] @ what[int(e)] for i, e in enumerate(idx)])
    np.testing.assert_allclose(oracle.gather_qmm_nn(x, wq, sc, bs, idx, E), ref, rtol=1e-12, atol=1e-10)
    rows = [39, 0, 17]
    np.testing.assert_array_equal(oracle.gather_qmm_nn(x, wq, sc, bs, idx, E, rows=rows),
                                  oracle.gather_qmm_nn(x, wq, sc, bs, idx, E)[rows])


def test_nn_closed_form_one_hot_x():
    # W[e, k, c] = (e - 1) + ((k + c) mod 16) / 8 quantizes exactly (each 64-run of c holds every
    # residue), so a one-hot x at k0 returns row k0 of W[e] exactly, and x = 1 returns its column sums
    E, K, N = 2, 16, 128
    w = (np.arange(E)[:, None, None] - 1) + ((np.arange(K)[None, :, None] + np.arange(N)[None, None, :]) % 16) / 8.0
    wq, sc, bs = oracle.quantize(wl.to_bf16(w.astype(np.float32)))
    x = np.zeros((3, K), np.float32)
    x[0, 5] = 1.0
    x[1, 11] = 1.0
    x[2, :] = 1.0
    idx = np.array([1, 0, 1], np.uint32)
    y = oracle.gather_qmm_nn(wl.to_bf16(x), wq, sc, bs, idx, E)
    np.testing.assert_array_equal(y[0], w[1, 5])
    np.testing.assert_array_equal(y[1], w[0, 11])
    np.testing.assert_allclose(y[2], w[1].sum(axis=0), rtol=0, atol=1e-12)
