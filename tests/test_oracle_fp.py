"""Pins for the oracle's block-scaled floating-point modes mxfp4, nvfp4 and mxfp8 (mlx #4339,
"Activity", nastya236: the CUDA back end is to support mxfp8 and nvfp4).  The formats are the
published ones (OCP Microscaling v1.0 for mxfp4 / mxfp8, NVIDIA's NVFP4 for nvfp4); the checks
do not reuse the oracle's arithmetic:
  * literal codes of hand-chosen values (E2M1, E4M3 and E8M0 bit patterns worked out by hand);
  * ties to the even significand and saturation at the largest finite value, by hand;
  * E4M3 rounding against torch's float8_e4m3fn conversion (a library implementation);
  * every element's code is the nearest representable value, by brute force over all codes;
  * the gather against a decode with hand-typed E2M1 values and numpy float64 matmul.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl

# the 8 magnitudes of E2M1 by code (bits: exponent 2, mantissa 1; bias 1; code 1 is subnormal)
E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _e2m1(c):
    return (-1.0 if c & 8 else 1.0) * E2M1[c & 7]


def _e4m3_torch(codes):
    return torch.from_numpy(np.asarray(codes, np.uint8)).view(torch.float8_e4m3fn).float().double().numpy()


def _bf16(v):
    return wl.to_bf16(np.asarray(v, np.float32))


def _nibbles(wq_row):
    out = []
    for b in np.asarray(wq_row, np.uint8):
        out += [int(b) & 15, int(b) >> 4]
    return out


def test_mxfp4_literal_codes_and_scale():
    k = 3  # the block's largest magnitude is 6 * 2^3, so its E8M0 scale is 2^3 (code 130)
    vals = [0, 0.5, 1, 1.5, 2, 3, 4, 6, -0.5, -1, -1.5, -2, -3, -4, -6, 0] * 2
    w = _bf16(np.array(vals) * 2.0 ** k).reshape(1, 32)
    wq, sc, ts = oracle.quantize_fp(w, "mxfp4")
    assert ts is None and sc.reshape(-1).tolist() == [130]
    assert _nibbles(wq[0]) == [0x0, 0x1, 0x2, 0x3, 0x4, 0x5, 0x6, 0x7, 0x9, 0xA, 0xB, 0xC, 0xD, 0xE, 0xF, 0x0] * 2
    assert wq[0, 0] == 0x10 and wq[0, 1] == 0x32  # element 0 in the low nibble
    assert np.array_equal(oracle.dequantize_fp(wq, sc, None, "mxfp4"), w.double().numpy())


def test_mxfp4_ties_to_even_and_saturation():
    # amax 7 gives scale 2^(2 - 2) = 1; 7 and 6.5 saturate to 6
    vals = [2.5, 5.0, 0.25, 0.75, 1.25, 1.75, -2.5, 7.0, 6.5, 3.5] + [0.0] * 22
    wq, sc, _ = oracle.quantize_fp(_bf16(vals).reshape(1, 32), "mxfp4")
    assert sc.reshape(-1).tolist() == [127]
    got = [_e2m1(c) for c in _nibbles(wq[0])[:10]]
    assert got == [2.0, 4.0, 0.0, 1.0, 1.0, 2.0, -2.0, 6.0, 6.0, 4.0]


def test_mxfp8_literal_codes():
    # amax 448 = 1.75 * 2^8: scale 2^(8 - 8) = 1 (code 127)
    vals = [448.0, 1.0, -1.5, 2.0 ** -9, 2.0 ** -6, 0.875 * 2.0 ** -6, 240.0, -448.0] + [0.0] * 24
    wq, sc, _ = oracle.quantize_fp(_bf16(vals).reshape(1, 32), "mxfp8")
    assert sc.reshape(-1).tolist() == [127]
    assert wq[0, :8].tolist() == [0x7E, 0x38, 0xBC, 0x01, 0x08, 0x07, 0x77, 0xFE]
    # scaled block: amax 3 * 2^-20 = 1.5 * 2^-19 gives scale 2^(-19 - 8) (code 100)
    wq2, sc2, _ = oracle.quantize_fp(_bf16([3 * 2.0 ** -20] + [0.0] * 31).reshape(1, 32), "mxfp8")
    assert sc2.reshape(-1).tolist() == [100] and wq2[0, 0] == 0x7C  # 3 * 2^-20 / 2^-27 = 384 = 1.5 * 2^8


def test_mxfp8_rounding_matches_torch_float8():
    """Within range, rounding to E4M3 is the same as torch's float32 -> float8_e4m3fn conversion."""
    w = wl.normal_bf16((64, 256), 5)
    wq, sc, _ = oracle.quantize_fp(w, "mxfp8")
    X = 2.0 ** (sc.astype(np.float64) - 127).repeat(32, axis=1)
    v = (w.double().numpy() / X)  # exact: division by a power of two; |v| < 2^9
    inside = np.abs(v) < 448
    ref = torch.from_numpy(v.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert inside.mean() > 0.9 and np.array_equal(wq[inside], ref[inside])
    # beyond the largest finite value the mx formats saturate: +-448 (0x7E / 0xFE)
    assert np.all(wq[~inside] == np.where(v[~inside] > 0, 0x7E, 0xFE))


def test_nvfp4_literal_codes_and_scales():
    # tensor amax 2688 = 6 * 448: tensor scale 1.0; block 0 amax 6: E4M3 scale 1.0 (0x38);
    # block 1 amax 12: scale 2.0 (0x40), elements halved
    b0 = [6.0, -3.0, 0.5, 1.0] + [0.0] * 12
    b1 = [12.0, 2.0, -1.0, 3.0] + [0.0] * 12
    b2 = [2688.0] + [0.0] * 15  # amax 2688: scale 448 (0x7E), element 6
    w = _bf16(b0 + b1 + b2 + [0.0] * 16).reshape(1, 1, 64)
    wq, sc, ts = oracle.quantize_fp(w, "nvfp4")
    assert ts.tolist() == [1.0]
    assert sc.reshape(-1).tolist() == [0x38, 0x40, 0x7E, 0x00]
    n = _nibbles(wq[0, 0])
    assert n[:4] == [0x7, 0xD, 0x1, 0x2] and n[16:20] == [0x7, 0x2, 0x9, 0x3] and n[32] == 0x7
    assert n[48:] == [0] * 16  # all-zero block: scale 0, codes 0
    assert np.array_equal(oracle.dequantize_fp(wq, sc, ts, "nvfp4"), w.double().numpy())


@pytest.mark.parametrize("mode", ["mxfp4", "nvfp4", "mxfp8"])
def test_codes_are_nearest_by_brute_force(mode):
    """Every element's code is a nearest representable value of the element it encodes (w / X for
    the mx modes; the float32 quotient w / (S * t) for nvfp4), checked against all codes."""
    w = wl.normal_bf16((2, 8, 128), 11)
    wq, sc, ts = oracle.quantize_fp(w, mode)
    wf = w.double().numpy()
    nb = oracle.MODE_BLOCK[mode]
    if mode == "mxfp8":
        table = _e4m3_torch(np.arange(256))
        codes = wq.astype(np.int64)
    else:
        table = np.array([_e2m1(c) for c in range(16)])
        codes = np.array([_nibbles(r) for r in wq.reshape(-1, wq.shape[-1])]).reshape(wf.shape)
    if mode == "nvfp4":
        S = _e4m3_torch(sc.reshape(-1)).reshape(sc.shape).astype(np.float32)
        denom = (S * ts.reshape(-1, 1, 1)).astype(np.float32).repeat(nb, axis=-1)
        target = (wf.astype(np.float32) / denom).astype(np.float64)
        target[denom == 0] = 0.0
    else:
        target = wf / 2.0 ** (sc.astype(np.float64) - 127).repeat(nb, axis=-1)
    finite = np.isfinite(table)
    dist = np.abs(target[..., None] - np.where(finite, table, np.inf))
    best = dist.min(axis=-1)
    chosen = np.take_along_axis(dist, codes[..., None], axis=-1)[..., 0]
    assert np.all(chosen <= best)


@pytest.mark.parametrize("mode", ["mxfp4", "nvfp4", "mxfp8"])
def test_gather_against_decode_and_numpy(mode):
    E, F, H, T, A = 3, 16, 128, 6, 2
    w = wl.normal_bf16((E, F, H), 21, std=0.3)
    x = wl.normal_bf16((T, A, H), 22)
    idx = wl.idx_uniform(T, A, E, seed=23)
    wq, sc, ts = oracle.quantize_fp(w, mode)
    nb = oracle.MODE_BLOCK[mode]
    if mode == "mxfp8":
        vals = _e4m3_torch(wq.reshape(-1)).reshape(E, F, H)
    else:
        vals = np.array([[[_e2m1(c) for c in _nibbles(wq[e, f])] for f in range(F)] for e in range(E)])
    if mode == "nvfp4":
        scale = _e4m3_torch(sc.reshape(-1)).reshape(sc.shape) * ts.astype(np.float64).reshape(-1, 1, 1)
    else:
        scale = 2.0 ** (sc.astype(np.float64) - 127)
    w_dec = vals * scale.repeat(nb, axis=-1)
    assert np.array_equal(oracle.dequantize_fp(wq, sc, ts, mode), w_dec)
    # quantization error stays within the format's resolution (a loose sanity bound)
    assert np.abs(w_dec - w.double().numpy()).max() <= 0.3 * np.abs(w.double().numpy()).max()
    xf = x.double().numpy().reshape(-1, H)
    ref = np.stack([xf[i] @ w_dec[idx.reshape(-1)[i]].T for i in range(T * A)])
    y = oracle.gather_qmm_fp(x, wq, sc, ts, idx, E, mode)
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-9)
    rows = [0, 5, 11]
    assert np.allclose(oracle.gather_qmm_fp(x, wq, sc, ts, idx, E, mode, rows=rows), ref[rows], rtol=1e-12, atol=1e-9)
