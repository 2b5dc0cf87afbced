"""Pins of the oracle's per-block INT8 quantizer (CPU only).

The quantizer reading (128-token blocks, absmax/127 scale, round half to even,
K-smoothing by the FP32 channel mean) follows "SageBwd: A Trainable Low-bit
Attention", Abstract (INT8 attention, K-smoothing).  The golden cases are
hand-derived; the properties below hold for any input.
"""
import os

import numpy as np
import pytest
import torch

HERE = os.path.dirname(os.path.abspath(__file__))


def _expand(tokens):
    out = []
    for t in tokens:
        if "*" in t:
            v, n = t.split("*")
            out += [v] * int(n)
        else:
            out.append(t)
    return out


def load_cases():
    cases, cur = [], None
    with open(os.path.join(HERE, "golden", "quantize_cases.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *rest = line.split()
            if key == "case":
                cur = {"name": rest[0]}
            elif key == "end":
                cases.append(cur)
                cur = None
            else:
                cur[key] = _expand(rest)
    return cases


def _hex_to_f32(h):
    return np.array([int(x, 16) for x in h], np.uint32).view(np.float32)


def _bf16_bits_of(values):
    f = np.array(values, np.float32)
    bits = f.view(np.uint32)
    assert np.all(bits & 0xFFFF == 0), "golden inputs must be exact BF16 values"
    return (bits >> 16).astype(np.uint16)


@pytest.mark.parametrize("case", load_cases(), ids=lambda c: c["name"])
def test_golden_quantize_cases(oracle_mod, case):
    N, d, smooth = int(case["N"][0]), int(case["d"][0]), bool(int(case["smooth"][0]))
    x = _bf16_bits_of([float(v) for v in case["x"]])
    p = oracle_mod.problem(1, 1, 1, N, d, False)
    codes, scales, mean = oracle_mod.quantize(p, x, 1, smooth)
    np.testing.assert_array_equal(codes.reshape(-1), np.array([int(c) for c in case["codes"]], np.int8))
    np.testing.assert_array_equal(scales.reshape(-1).view(np.uint32), _hex_to_f32(case["scales"]).view(np.uint32))
    if "means" in case:
        np.testing.assert_array_equal(mean.reshape(-1).view(np.uint32), _hex_to_f32(case["means"]).view(np.uint32))


def _random_bf16(shape, seed, scale=1.0, offset=0.0):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(*shape, generator=g) * scale + offset
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("N,d,smooth", [(300, 64, False), (300, 64, True), (129, 128, True), (1, 64, False)])
def test_quantize_properties(oracle_mod, N, d, smooth):
    BH = 3
    x = _random_bf16((BH, N, d), seed=N * 7 + d, scale=2.0, offset=1.5)
    p = oracle_mod.problem(1, 1, 1, N, d, False)
    codes, scales, mean = oracle_mod.quantize(p, x, BH, smooth)
    xf = x.float().numpy().astype(np.float64)
    if smooth:
        # channel mean = FP64 mean of the BF16 values, rounded once to FP32 (library special case)
        ref_mean = xf.mean(axis=1).astype(np.float32)
        np.testing.assert_array_equal(mean, ref_mean)
        xf = (x.float().numpy() - mean[:, None, :]).astype(np.float64)  # FP32 subtraction
    nb = (N + 127) // 128
    assert scales.shape == (BH, nb)
    c = codes.astype(np.int64)
    assert c.min() >= -127 and c.max() <= 127
    for bh in range(BH):
        for blk in range(nb):
            sl = slice(blk * 128, min(N, blk * 128 + 128))
            a = np.abs(xf[bh, sl]).max()
            s = float(scales[bh, blk])
            # the element with the largest magnitude maps to +-127 and the scale is a/127 to FP32 precision
            assert np.abs(c[bh, sl]).max() == 127
            assert abs(s * 127 - a) <= 2 * np.spacing(np.float32(a))
            # round-to-nearest: reconstruction error at most half a step (plus FP32 slack)
            err = np.abs(c[bh, sl] * s - xf[bh, sl])
            assert err.max() <= 0.5 * s * (1 + 1e-5) + 1e-30


def test_quantize_zero_and_constant_blocks(oracle_mod):
    N, d = 256, 8
    x = torch.zeros(1, N, d)
    x[0, 128:] = 3.0  # block 1 constant
    x = x.to(torch.bfloat16)
    p = oracle_mod.problem(1, 1, 1, N, d, False)
    codes, scales, _ = oracle_mod.quantize(p, x, 1, False)
    assert scales[0, 0] == 0 and np.all(codes[0, :128] == 0)
    assert np.all(codes[0, 128:] == 127)
    # smoothing a constant-over-tokens tensor leaves an all-zero block with scale 0
    codes, scales, mean = oracle_mod.quantize(p, torch.full((1, N, d), 3.0).to(torch.bfloat16), 1, True)
    assert np.all(mean == 3.0) and np.all(scales == 0) and np.all(codes == 0)


def test_quantize_exact_reconstructs(oracle_mod):
    """Without rounding, code * scale reproduces the (smoothed) input to FP64 precision."""
    N, d = 200, 16
    x = _random_bf16((2, N, d), seed=11, scale=3.0, offset=-2.0)
    p = oracle_mod.problem(1, 1, 1, N, d, False)
    codes, scales, mean = oracle_mod.quantize_exact(p, x, 2, True)
    xf = x.double().numpy()
    ref = xf - xf.mean(axis=1, keepdims=True)
    rec = codes * np.repeat(scales, 128, axis=1)[:, :N, None]
    np.testing.assert_allclose(rec, ref, rtol=0, atol=1e-12 * np.abs(ref).max())
