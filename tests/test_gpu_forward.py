"""GPU parity of the quantize stage and the fused forward against the oracle.

The INT8 codes, block scales and K means the library writes must equal the
oracle's bit for bit; O and LSE must meet the normwise tolerance of
tests/_parity.py.  Small shapes cover several tiles, ragged tails, GQA,
causal masks, N = 1 and both head dims; the five named workloads are checked
at full size on sampled query blocks.
"""
import numpy as np
import pytest
import torch

import bit_trainable_attention_gb300 as sb
from bit_trainable_attention_gb300 import workloads as W
from _parity import (LSE_TOL, assert_parity, block_selection, cos, device_inputs, gpu_forward, oracle_problem,
                     to_np)

pytestmark = pytest.mark.gpu

SMALL = [
    W.WORKLOADS["tiny"],
    W.small("gqa_causal_300_d64", 1, 4, 2, 300, 64, True, 101, qk_norm=True, k_offset_sd=2.0),
    W.small("gqa_noncausal_257_d128", 2, 3, 1, 257, 128, False, 102, k_offset_sd=3.0),
    W.small("outlier_causal_384_d128", 1, 2, 2, 384, 128, True, 103, outlier_frac=0.01),
    W.small("n1_d64", 1, 2, 1, 1, 64, True, 104),
    W.small("n129_d128_noncausal", 1, 2, 2, 129, 128, False, 105, qk_norm=True),
    W.small("n127_d64_causal", 2, 2, 2, 127, 64, True, 106),
]


def check_quantized(oracle_mod, w, x, fwd, smooth_k=True):
    """Q^, K^ (with the default Q/K sub-scales: codes times 2^-k), V^, the block scales and the K mean
    bit for bit against the oracle's quantizers."""
    qk_subexp = bool(fwd["prob"].qk_subexp)
    op = oracle_problem(oracle_mod, w, smooth_k, qk_subexp=qk_subexp)
    views = sb.quantized_views(fwd["prob"], fwd["saved"])
    ref = oracle_mod.quantize_qk(op, x["q"], x["k"])
    for name in ("q", "k"):
        g = views[name].float().cpu().numpy().reshape(ref[name].shape)
        np.testing.assert_array_equal(g, ref[name], err_msg=f"{name} values")
        np.testing.assert_array_equal(views["s" + name].cpu().numpy().view(np.uint32),
                                      ref["s" + name].view(np.uint32), err_msg=f"{name} scales")
    if smooth_k:
        np.testing.assert_array_equal(views["mu"].cpu().numpy().view(np.uint32), ref["mu"].view(np.uint32),
                                      err_msg="k mean")
    codes, scales, _ = oracle_mod.quantize(op, x["v"], w.B * w.Hkv, False)
    gcodes = views["v"].float().cpu().numpy().reshape(codes.shape)
    np.testing.assert_array_equal(gcodes, codes.astype(np.float32), err_msg="v codes")
    np.testing.assert_array_equal(views["sv"].cpu().numpy().view(np.uint32), scales.view(np.uint32),
                                  err_msg="v scales")


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_forward_small(oracle_mod, w):
    x, xd = device_inputs(w)
    fwd = gpu_forward(w, xd)
    assert fwd["status"] == 0
    check_quantized(oracle_mod, w, x, fwd)
    op = oracle_problem(oracle_mod, w)
    o_ref, lse_ref = oracle_mod.fwd(op, x["q"], x["k"], x["v"])
    assert_parity(to_np(fwd["o"]), o_ref, "O")
    np.testing.assert_allclose(to_np(fwd["lse"]), lse_ref, rtol=0, atol=LSE_TOL)
    ex_o, _ = oracle_mod.fwd(op, x["q"], x["k"], x["v"], exact=True)
    if w.outlier_frac == 0:
        assert cos(to_np(fwd["o"]), ex_o) >= 0.995


def test_forward_without_smoothing(oracle_mod):
    w = W.small("nosmooth", 1, 2, 1, 200, 64, True, 111, k_offset_sd=2.0)
    x, xd = device_inputs(w)
    fwd = gpu_forward(w, xd, smooth_k=False)
    check_quantized(oracle_mod, w, x, fwd, smooth_k=False)
    op = oracle_problem(oracle_mod, w, smooth_k=False)
    o_ref, lse_ref = oracle_mod.fwd(op, x["q"], x["k"], x["v"])
    assert_parity(to_np(fwd["o"]), o_ref, "O")
    np.testing.assert_allclose(to_np(fwd["lse"]), lse_ref, rtol=0, atol=LSE_TOL)


@pytest.mark.parametrize("balance", [False, True], ids=["plain", "balanced"])
def test_forward_repeatable(oracle_mod, balance):
    """Two calls on the same inputs give identical bits (no atomics in the forward)."""
    w = W.small("rep", 1, 4, 2, 520, 64, True, 112, qk_norm=True, outlier_frac=0.02 if balance else 0.0)
    _, xd = device_inputs(w)
    a = gpu_forward(w, xd, balance_qk=balance)
    b = gpu_forward(w, xd, balance_qk=balance)
    assert torch.equal(a["o"], b["o"]) and torch.equal(a["lse"], b["lse"])
    va, vb = sb.quantized_views(a["prob"], a["saved"]), sb.quantized_views(b["prob"], b["saved"])
    for key in va:  # the sections of the saved buffer (its alignment padding is never written)
        if key == "e" and not a["prob"].balance_qk:
            continue  # the balancing exponents are written only with balance_qk
        assert torch.equal(va[key], vb[key]), key


@pytest.mark.parametrize("name", ["pretrain", "llama1b", "qwen15b", "videodit"])
def test_forward_full_size_sampled(oracle_mod, name):
    """Full-size workload in the bench's launch configuration; quantized
    operands compared in full, O/LSE on sampled query blocks (first, middle,
    last) of two heads."""
    w = W.WORKLOADS[name]
    x, xd = device_inputs(w)
    fwd = gpu_forward(w, xd)
    assert fwd["status"] == 0
    check_quantized(oracle_mod, w, x, fwd)
    nb = (w.N + 127) // 128
    heads = [0, w.Hq - 1]
    sel = block_selection(w, heads, [0, nb // 2, -1])
    op = oracle_problem(oracle_mod, w)
    o_ref, lse_ref = oracle_mod.fwd(op, x["q"], x["k"], x["v"], qsel=sel)
    o = to_np(fwd["o"])
    lse = to_np(fwd["lse"])
    m = np.isfinite(lse_ref)
    assert m.sum() > 0
    assert_parity(o[m], o_ref[m], "O")
    np.testing.assert_allclose(lse[m], lse_ref[m], rtol=0, atol=LSE_TOL)
    assert np.all(np.isfinite(o))


@pytest.mark.parametrize("balance", [False, True], ids=["kmean", "stats"])
def test_k_mean_over_a_wide_value_range(oracle_mod, balance):
    """K values whose magnitudes span 2^-12 .. 2^13 within a channel: FP32 partial sums
    would round, so the library's exactness check must fall back to FP64; the mean (and the
    codes) still equal the oracle's bit for bit.  Covers both K-mean kernels (the plain one
    and the balancing statistics)."""
    w = W.small("wide", 1, 2, 2, 300, 64, False, 113)
    x = W.make_inputs(w)
    g = torch.Generator().manual_seed(7)
    mag = torch.exp2(torch.randint(-12, 13, x["k"].shape, generator=g).float())  # FP64 sums stay exact
    x["k"] = (x["k"].float().sign() * mag * (1 + torch.rand(x["k"].shape, generator=g))).to(torch.bfloat16)
    xd = {k: v.cuda() for k, v in x.items()}
    fwd = gpu_forward(w, xd, balance_qk=balance)
    assert fwd["status"] == 0
    op = oracle_problem(oracle_mod, w, balance_qk=balance)
    ref = oracle_mod.quantize_qk(op, x["q"], x["k"])
    views = sb.quantized_views(fwd["prob"], fwd["saved"])
    np.testing.assert_array_equal(views["mu"].cpu().numpy().view(np.uint32), ref["mu"].view(np.uint32))
    np.testing.assert_array_equal(views["k"].float().cpu().numpy().reshape(ref["k"].shape),
                                  ref["k"].astype(np.float32))
    if balance:
        np.testing.assert_array_equal(views["e"].cpu().numpy(), ref["e"])
