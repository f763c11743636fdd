"""Pins for the oracle's affine format at bit widths 2, 3, 5, 6 and 8 (mlx PR #4023, the author's
follow-up: upstream tests run every bit width).  Each group keeps scale = (max - min) / (2^b - 1)
and bias = min, and a row's codes are one little-endian bit stream (element k in bits
[k*b, (k+1)*b)).  The checks do not reuse the oracle's arithmetic:
  * literal packed bytes, worked out by hand from the bit-stream layout, for groups whose codes
    are known (w = bias + s*q with a power-of-two s, so q comes back exactly);
  * exact round trips of such groups, and the bound |w - w_hat| <= s/2 on random data;
  * the gather against a pure-Python bit-stream decode and numpy float64 matmul.
"""
import numpy as np
import pytest

import oracle
import workloads as wl


def _group_from_codes(q, s=0.125, bias=-1.0):
    """bf16 weights bias + s*q (exact in bfloat16 for the codes used here)."""
    return wl.to_bf16((bias + s * np.asarray(q, np.float64)).astype(np.float32)).reshape(1, -1)


# codes of the 64-element group per bit width, and the packed bytes of its start, by hand
LITERALS = {
    2: ([k % 4 for k in range(64)], [0xE4] * 16),
    3: ([k % 8 for k in range(64)], [0x88, 0xC6, 0xFA] * 8),
    5: ([k % 32 for k in range(64)], [0x20, 0x88, 0x41, 0x8A, 0x39]),
    6: ([k % 64 for k in range(64)], [0x40, 0x20, 0x0C]),
    8: ([min(255, 4 * k) for k in range(63)] + [255], [min(255, 4 * k) for k in range(63)] + [255]),
}


@pytest.mark.parametrize("bits", sorted(LITERALS))
def test_literal_packed_bytes(bits):
    codes, head = LITERALS[bits]
    wq, sc, bs = oracle.quantize(_group_from_codes(codes), group_size=64, bits=bits)
    assert wq.shape == (1, 64 * bits // 8)
    assert list(wq.reshape(-1)[: len(head)]) == head
    assert sc.reshape(-1)[0] == 0x3E00 and bs.reshape(-1)[0] == 0xBF80  # 0.125 and -1.0 in bfloat16


def _unpack(row_bytes, bits, H):
    """Pure-Python decode of one row's bit stream (the layout's definition, bit by bit)."""
    out = []
    for k in range(H):
        v = 0
        for i in range(bits):
            j = k * bits + i
            v |= ((int(row_bytes[j // 8]) >> (j % 8)) & 1) << i
        out.append(v)
    return out


@pytest.mark.parametrize("bits", [2, 3, 5, 6, 8])
@pytest.mark.parametrize("gs", [32, 64, 128])
def test_round_trip_and_codes(bits, gs):
    """Random groups bias + s*q with s = 2^-e and q covering 0 and 2^b - 1: the codes come back
    as q and the dequantized weights equal w exactly."""
    rng = np.random.default_rng(bits * 100 + gs)
    L = (1 << bits) - 1
    rows, H = 3, 256
    q = rng.integers(0, L + 1, size=(rows, H))
    q[:, ::gs] = 0
    q[:, 1::gs] = L
    s = 2.0 ** -rng.integers(2, 5, size=(rows, H // gs))
    # bias a non-positive multiple of s: w = s * (q - k) with |q - k| < 256, exact in bfloat16
    k = np.floor(rng.random((rows, H // gs)) * 8) if bits < 8 else np.zeros((rows, H // gs))
    bias = -k * s
    w = bias.repeat(gs, axis=1) + s.repeat(gs, axis=1) * q
    wb = wl.to_bf16(w.astype(np.float32))
    assert np.array_equal(wb.float().double().numpy(), w)
    wq, sc, bs = oracle.quantize(wb, group_size=gs, bits=bits)
    for r in range(rows):
        assert _unpack(wq[r], bits, H) == list(q[r])
    w_hat = oracle.dequantize(wq, sc, bs, group_size=gs, bits=bits)
    assert np.array_equal(w_hat, w)


@pytest.mark.parametrize("bits", [2, 3, 5, 6, 8])
def test_error_bound_on_random_weights(bits):
    w = wl.normal_bf16((16, 512), 7 + bits)
    wq, sc, bs = oracle.quantize(w, group_size=64, bits=bits)
    w_hat = oracle.dequantize(wq, sc, bs, group_size=64, bits=bits)
    wf = w.float().double().numpy()
    s = (sc.astype(np.uint32) << 16).view(np.float32).astype(np.float64).repeat(64, axis=1)
    b = (bs.astype(np.uint32) << 16).view(np.float32).astype(np.float64).repeat(64, axis=1)
    L = (1 << bits) - 1  # the top code's clamp can add up to L * s * 2^-9 (bf16 rounding of s)
    assert np.all(np.abs(wf - w_hat) <= s / 2 + 1e-12 + L * s * 2.0 ** -9)
    assert np.array_equal(b, wf.reshape(16, 8, 64).min(axis=2).repeat(64, axis=1))  # bias = group min
    codes = np.array([_unpack(wq[r], bits, 512) for r in range(16)])
    assert codes.max() <= (1 << bits) - 1
    assert np.all(codes[wf == b] == 0)  # the minimum maps to code 0


@pytest.mark.parametrize("bits", [2, 3, 5, 6, 8])
def test_gather_against_bit_stream_decode_and_numpy(bits):
    E, F, H, T, A, gs = 3, 8, 128, 5, 2, 32
    w = wl.normal_bf16((E, F, H), 20 + bits)
    x = wl.normal_bf16((T, A, H), 30 + bits)
    idx = wl.idx_uniform(T, A, E, seed=40 + bits)
    wq, sc, bs = oracle.quantize(w, group_size=gs, bits=bits)
    s = (sc.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    b = (bs.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    w_dec = np.zeros((E, F, H))
    for e in range(E):
        for f in range(F):
            q = np.array(_unpack(wq[e, f], bits, H), np.float64)
            w_dec[e, f] = s[e, f].repeat(gs) * q + b[e, f].repeat(gs)
    xf = x.float().double().numpy().reshape(-1, H)
    ref = np.stack([xf[i] @ w_dec[idx.reshape(-1)[i]].T for i in range(T * A)])
    y = oracle.gather_qmm(x, wq, sc, bs, idx, E, group_size=gs, bits=bits)
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-9)
