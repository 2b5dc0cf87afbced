"""Pins of the oracle's FP8 variant quantizer (reading r25) on its edge cases.

* a block whose largest magnitude lies between 2^-120 and 2^-118 keeps INT8 codes (127/max is finite
  in FP32) but gets zero E4M3 values and scale 0 in the FP8 variant (448/max would overflow FP32);
* just above 2^-118 the E4M3 values are finite, the largest one is 448 and the scale is max/448;
* the E4M3 values of an ordinary block equal torch's float8_e4m3fn conversion of x * (448 / max).
"""
import numpy as np
import torch


def _qk(oracle_mod, q_block, fp8):
    """Quantize one 128 x 64 block as Q (K is a copy), without smoothing."""
    q = torch.tensor(q_block, dtype=torch.float32).to(torch.bfloat16).view(1, 1, 128, 64)
    p = oracle_mod.problem(1, 1, 1, 128, 64, False, smooth_k=False, fp8=fp8)
    return oracle_mod.quantize_qk(p, q, q.clone())


def test_fp8_tiny_group_threshold(oracle_mod):
    rng = np.random.default_rng(3)
    base = rng.uniform(-1, 1, (128, 64))
    base[5, 7] = 1.0
    for scale, int8_zero, fp8_zero in ((2.0 ** -119, False, True), (2.0 ** -117, False, False)):
        x = base * scale
        r8 = _qk(oracle_mod, x, False)
        rf = _qk(oracle_mod, x, True)
        assert (not r8["q"].any()) == int8_zero
        assert (not rf["q"].any()) == fp8_zero
        if fp8_zero:
            assert rf["sq"][0, 0] == 0.0
        else:
            assert np.isfinite(rf["q"]).all() and np.abs(rf["q"]).max() == 448.0
            assert rf["sq"][0, 0] == np.float32(np.float32(scale) / np.float32(448.0))


def test_fp8_values_match_torch_e4m3(oracle_mod):
    rng = np.random.default_rng(4)
    x = rng.normal(0, 1, (128, 64))
    xb = torch.tensor(x, dtype=torch.float32).to(torch.bfloat16).float()
    a = xb.abs().max()
    inv = (torch.tensor(448.0) / a).float()
    want = (xb * inv).to(torch.float8_e4m3fn).float().numpy()
    r = _qk(oracle_mod, x, True)
    np.testing.assert_array_equal(r["q"][0], want)
