"""Pins for the oracle's MoE expert MLP (y = W_dn (act(W_g x) * (W_u x)) per routed row, act =
SiLU, GELU or GELU's tanh form), against a brute-force loop with its own nibble decode, a closed
form on exactly representable weights, and invariants; and pins for the three activations
against printed values, identities and PyTorch's float64 implementations.  None of these calls
the oracle's own dequantization."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as wl


def _bits_to_f64(u16):
    return (np.asarray(u16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _decode(wq, sc, bs, e, f, h):
    byte = int(wq[e, f, h // 2])
    code = (byte >> (4 * (h % 2))) & 15
    return _bits_to_f64(sc[e, f, h // 64]) * code + _bits_to_f64(bs[e, f, h // 64])


_ACT = {"silu": lambda v: v / (1.0 + math.exp(-v)),
        "gelu": lambda v: 0.5 * v * (1.0 + math.erf(v / math.sqrt(2.0))),
        "gelu_tanh": lambda v: 0.5 * v * (1.0 + math.tanh(math.sqrt(2.0 / math.pi) * (v + 0.044715 * v ** 3)))}


def test_activation_values_and_identities():
    # Phi(1) = 0.8413447460685429 (standard normal table), so GELU(1) = Phi(1) and GELU(-1) = Phi(1) - 1
    np.testing.assert_allclose(oracle.gelu(np.array([1.0, -1.0, 0.0])), [0.8413447460685429, -0.1586552539314571, 0.0],
                               rtol=0, atol=1e-15)
    # SiLU(1) = 1 / (1 + e^-1); SiLU(-v) = SiLU(v) - v
    assert oracle.silu(np.array([1.0]))[0] == pytest.approx(1.0 / (1.0 + math.exp(-1.0)), abs=1e-16)
    v = np.random.default_rng(5).normal(0, 3, 1000)
    for f in (oracle.silu, oracle.gelu, oracle.gelu_tanh):
        np.testing.assert_allclose(f(v) - f(-v), v, rtol=0, atol=1e-12)  # act(v) = v * (odd-symmetric CDF)
    # the tanh form stays within 5e-4 of the exact GELU on [-6, 6] (its published accuracy)
    grid = np.linspace(-6, 6, 4001)
    assert np.abs(oracle.gelu_tanh(grid) - oracle.gelu(grid)).max() < 5e-4


def test_activations_match_torch_float64():
    v = np.random.default_rng(6).normal(0, 4, 4096)
    t = torch.from_numpy(v)
    np.testing.assert_allclose(oracle.silu(v), torch.nn.functional.silu(t).numpy(), rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(oracle.gelu(v), torch.nn.functional.gelu(t).numpy(), rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(oracle.gelu_tanh(v), torch.nn.functional.gelu(t, approximate="tanh").numpy(),
                               rtol=1e-13, atol=1e-15)


@pytest.mark.parametrize("activation", ["silu", "gelu", "gelu_tanh"])
def test_mlp_brute_force_tiny(activation):
    E, I, H, n = 3, 64, 64, 5  # one quantization group per row in both projections
    q_gu = oracle.quantize(wl.normal_bf16((E, 2 * I, H), 11))
    q_dn = oracle.quantize(wl.normal_bf16((E, H, I), 12))
    x = wl.normal_bf16((n, H), 13)
    idx = np.array([2, 0, 1, 5, 2], np.uint32)  # 5 >= E: a zero row
    y = oracle.moe_mlp(x, q_gu, q_dn, idx, E, activation=activation)
    act = _ACT[activation]
    xf = _bits_to_f64(wl.bf16_bits(x))
    ref = np.zeros((n, H))
    for i in range(n):
        e = int(idx[i])
        if e >= E:
            continue
        g = [sum(xf[i, h] * _decode(*q_gu, e, f, h) for h in range(H)) for f in range(I)]
        u = [sum(xf[i, h] * _decode(*q_gu, e, I + f, h) for h in range(H)) for f in range(I)]
        hh = [act(g[k]) * u[k] for k in range(I)]
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


@pytest.mark.parametrize("gs", [32, 128])
def test_mlp_brute_force_other_group_sizes(gs):
    E, I, H, n = 2, 128, 128, 3
    q_gu = oracle.quantize(wl.normal_bf16((E, 2 * I, H), 31), group_size=gs)
    q_dn = oracle.quantize(wl.normal_bf16((E, H, I), 32), group_size=gs)
    x = wl.normal_bf16((n, H), 33)
    idx = np.array([1, 0, 1], np.uint32)
    y = oracle.moe_mlp(x, q_gu, q_dn, idx, E, group_size=gs)
    xf = _bits_to_f64(wl.bf16_bits(x))

    def deq(q, e, f, h):
        wq, sc, bs = q
        code = (int(wq[e, f, h // 2]) >> (4 * (h % 2))) & 15
        return _bits_to_f64(sc[e, f, h // gs]) * code + _bits_to_f64(bs[e, f, h // gs])

    for i in range(n):
        e = int(idx[i])
        g = [sum(xf[i, h] * deq(q_gu, e, f, h) for h in range(H)) for f in range(I)]
        u = [sum(xf[i, h] * deq(q_gu, e, I + f, h) for h in range(H)) for f in range(I)]
        hh = [_ACT["silu"](g[k]) * u[k] for k in range(I)]
        ref = [sum(hh[k] * deq(q_dn, e, o, k) for k in range(I)) for o in range(H)]
        np.testing.assert_allclose(y[i], ref, rtol=1e-11, atol=1e-11)
