"""Pins for the oracle's MoE expert MLP (y = W_dn (SiLU(W_g x) * (W_u x)) per routed row),
against a brute-force loop with its own nibble decode, a closed form on exactly representable
weights, and invariants.  None of these calls the oracle's own dequantization."""
import math

import numpy as np

import oracle
import workloads as wl


def _bits_to_f64(u16):
    return (np.asarray(u16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _decode(wq, sc, bs, e, f, h):
    byte = int(wq[e, f, h // 2])
    code = (byte >> (4 * (h % 2))) & 15
    return _bits_to_f64(sc[e, f, h // 64]) * code + _bits_to_f64(bs[e, f, h // 64])


def test_mlp_brute_force_tiny():
    E, I, H, n = 3, 64, 64, 5  # one quantization group per row in both projections
    q_gu = oracle.quantize(wl.normal_bf16((E, 2 * I, H), 11))
    q_dn = oracle.quantize(wl.normal_bf16((E, H, I), 12))
    x = wl.normal_bf16((n, H), 13)
    idx = np.array([2, 0, 1, 5, 2], np.uint32)  # 5 >= E: a zero row
    y = oracle.moe_mlp(x, q_gu, q_dn, idx, E)
    xf = _bits_to_f64(wl.bf16_bits(x))
    ref = np.zeros((n, H))
    for i in range(n):
        e = int(idx[i])
        if e >= E:
            continue
        g = [sum(xf[i, h] * _decode(*q_gu, e, f, h) for h in range(H)) for f in range(I)]
        u = [sum(xf[i, h] * _decode(*q_gu, e, I + f, h) for h in range(H)) for f in range(I)]
        hh = [g[k] / (1.0 + math.exp(-g[k])) * u[k] for k in range(I)]
        for o in range(H):
            ref[i, o] = sum(hh[k] * _decode(*q_dn, e, o, k) for k in range(I))
    np.testing.assert_allclose(y, ref, rtol=1e-11, atol=1e-11)
    assert not y[3].any()


def test_mlp_closed_form_one_hot_rows():
    # w[e, f, h] = (e - 2) + ((f + h) mod 16) / 4 quantizes exactly (each 64-run holds every
    # residue), so a one-hot x at h0 gives g_f = w_g[e, f, h0], u_f = w_u[e, f, h0] exactly.
    E, I, H = 3, 64, 128
    e_ = np.arange(E)[:, None, None]
    wgu = (e_ - 2) + ((np.arange(2 * I)[None, :, None] + np.arange(H)[None, None, :]) % 16) / 4.0
    wdn = (e_ - 1) / 2 + ((np.arange(H)[None, :, None] * 3 + np.arange(I)[None, None, :]) % 16) / 8.0
    q_gu = oracle.quantize(wl.to_bf16(wgu.astype(np.float32)))
    q_dn = oracle.quantize(wl.to_bf16(wdn.astype(np.float32)))
    cases = [(0, 0), (2, 17), (1, 127), (2, 64)]
    x = np.zeros((len(cases), H), np.float32)
    for i, (_, h0) in enumerate(cases):
        x[i, h0] = 1.0
    idx = np.array([c[0] for c in cases], np.uint32)
    y = oracle.moe_mlp(wl.to_bf16(x), q_gu, q_dn, idx, E)
    for i, (e, h0) in enumerate(cases):
        g = wgu[e, :I, h0]
        u = wgu[e, I:, h0]
        hh = g / (1.0 + np.exp(-g)) * u
        np.testing.assert_allclose(y[i], wdn[e] @ hh, rtol=1e-12, atol=1e-12)


def test_mlp_permutation_invariance_and_rows_subset():
    E, I, H, n = 4, 64, 128, 12
    q_gu = oracle.quantize(wl.normal_bf16((E, 2 * I, H), 21))
    q_dn = oracle.quantize(wl.normal_bf16((E, H, I), 22))
    x = wl.normal_bf16((n, H), 23)
    idx = np.random.default_rng(3).integers(0, E, size=n).astype(np.uint32)
    y = oracle.moe_mlp(x, q_gu, q_dn, idx, E)
    p = np.random.default_rng(4).permutation(n)
    yp = oracle.moe_mlp(x[p], q_gu, q_dn, idx[p], E)
    np.testing.assert_array_equal(yp, y[p])
    rows = [11, 0, 5]
    np.testing.assert_array_equal(oracle.moe_mlp(x, q_gu, q_dn, idx, E, rows=rows), y[rows])
