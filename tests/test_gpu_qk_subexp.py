"""GPU parity of the Q/K granularity against the oracle: the library's default Q/K
sub-scales (qk_subexp), alone and with the other refinements (channel balancing,
dS sub-scales), and the plain one-scale-per-block mode (qk_subexp=False, the
pages' plainest reading), which every other GPU test leaves aside.

The stored Q^ and K^ values (codes times 2^-k per 8-channel group of a block),
the block scales and the K means must equal the oracle's bit for bit; O, LSE,
dQ, dK, dV must meet the normwise tolerance of tests/_parity.py.  On the
long-context outlier workload at full size, with all three refinements, the
library must meet the cosine-similarity criteria against exact attention on
the sampled blocks the oracle computes.
"""
import numpy as np
import pytest
import torch

import bit_trainable_attention_gb300 as sb
from bit_trainable_attention_gb300 import workloads as W
from _parity import (LSE_TOL, assert_parity, block_selection, cos, device_inputs, gpu_backward, gpu_forward,
                     oracle_problem, to_np)

pytestmark = pytest.mark.gpu

ALL = dict(qk_subexp=True, ds_subexp=True, balance_qk=True)
CASES = [
    (W.small("qkx_outlier_gqa_causal_384_d128", 1, 6, 1, 384, 128, True, 601, outlier_frac=0.01), dict(qk_subexp=True)),
    (W.small("qkx_outlier_gqa_nc_257_d64", 2, 4, 2, 257, 64, False, 602, outlier_frac=0.03, k_offset_sd=2.0),
     dict(qk_subexp=True)),
    (W.small("qkx_all_causal_300_d64", 1, 4, 2, 300, 64, True, 603, outlier_frac=0.03, k_offset_sd=2.0), ALL),
    (W.small("qkx_all_n129_d128", 1, 2, 2, 129, 128, False, 604, outlier_frac=0.02), ALL),
    (W.small("qkx_n1_d64", 1, 2, 1, 1, 64, True, 605), dict(qk_subexp=True)),
]


def check_values(oracle_mod, w, x, fwd, kw, smooth_k=True):
    ref = oracle_mod.quantize_qk(oracle_problem(oracle_mod, w, smooth_k, **{k: v for k, v in kw.items()
                                                                            if k != "ds_subexp"}), x["q"], x["k"])
    views = sb.quantized_views(fwd["prob"], fwd["saved"])
    for name in ("q", "k"):
        g = views[name].float().cpu().numpy().reshape(ref[name].shape)
        np.testing.assert_array_equal(g, ref[name], err_msg=f"{name} values")
        np.testing.assert_array_equal(views["s" + name].cpu().numpy().view(np.uint32),
                                      ref["s" + name].view(np.uint32), err_msg=f"{name} scales")
    if smooth_k:
        np.testing.assert_array_equal(views["mu"].cpu().numpy().view(np.uint32), ref["mu"].view(np.uint32))


@pytest.mark.parametrize("w,kw", CASES, ids=lambda c: c.name if hasattr(c, "name") else "-".join(sorted(c)))
def test_qk_subexp_forward_backward_small(oracle_mod, w, kw):
    x, xd = device_inputs(w)
    fwd = gpu_forward(w, xd, **kw)
    bwd = gpu_backward(w, xd, fwd)
    assert fwd["status"] == 0 and bwd["status"] == 0
    check_values(oracle_mod, w, x, fwd, kw)
    ref = oracle_mod.pipeline(oracle_problem(oracle_mod, w, **kw), x["q"], x["k"], x["v"], x["do"])
    assert_parity(to_np(fwd["o"]), ref["o"], "O")
    np.testing.assert_allclose(to_np(fwd["lse"]), ref["lse"], rtol=0, atol=LSE_TOL)
    for key in ("dq", "dk", "dv"):
        assert_parity(to_np(bwd[key]), ref[key], key)


def test_qk_subexp_without_smoothing(oracle_mod):
    w = W.small("qkx_nosmooth", 1, 2, 1, 200, 64, True, 611, outlier_frac=0.03, k_offset_sd=2.0)
    x, xd = device_inputs(w)
    fwd = gpu_forward(w, xd, smooth_k=False, qk_subexp=True)
    check_values(oracle_mod, w, x, fwd, dict(qk_subexp=True), smooth_k=False)


@pytest.mark.parametrize("which", ["q", "k"])
def test_single_operand_quantizer(oracle_mod, which):
    """sagebwd_quantize(Q or K) with qk_subexp stores the same values as the fused forward's quantizer."""
    w = W.small("qkx_single", 1, 4, 2, 300, 128, True, 612, outlier_frac=0.03, k_offset_sd=2.0)
    x, xd = device_inputs(w)
    prob = sb.Problem.make(w.B, w.Hq, w.Hkv, w.N, w.d, w.causal, qk_subexp=True)
    H = w.Hq if which == "q" else w.Hkv
    nb = (w.N + 127) // 128
    xq = torch.empty_like(xd[which])
    sc = torch.empty(w.B * H * nb, dtype=torch.float32, device="cuda")
    mu = torch.empty(w.B * w.Hkv * w.d, dtype=torch.float32, device="cuda")
    ws = sb.empty_bytes(sb.sagebwd_workspace_bytes(prob, 0), "cuda")
    sb.sagebwd_quantize(prob, sb.SAGEBWD_Q if which == "q" else sb.SAGEBWD_K, xd[which], xq, sc, mu, ws)
    torch.cuda.synchronize()
    ref = oracle_mod.quantize_qk(oracle_problem(oracle_mod, w, qk_subexp=True), x["q"], x["k"])
    np.testing.assert_array_equal(xq.float().cpu().numpy().reshape(ref[which].shape), ref[which])
    np.testing.assert_array_equal(sc.cpu().numpy().view(np.uint32), ref["s" + which].reshape(-1).view(np.uint32))


def test_all_refinements_full_size_long_context(oracle_mod):
    """The long-context workload at full size with Q/K sub-scales, channel balancing and dS
    sub-scales: stored values in full; O / LSE on sampled query blocks; the backward stage-wise on
    sampled blocks; and the CosSim criteria against exact attention on one query block of every
    head (the whole-tensor figures come from the bench)."""
    w = W.WORKLOADS["qwen15b"]
    x, xd = device_inputs(w)
    fwd = gpu_forward(w, xd, **ALL)
    bwd = gpu_backward(w, xd, fwd)
    assert fwd["status"] == 0 and bwd["status"] == 0
    check_values(oracle_mod, w, x, fwd, ALL)
    nb = (w.N + 127) // 128
    op = oracle_problem(oracle_mod, w, **ALL)
    fsel = block_selection(w, [0, 2, w.Hq - 1], [0, nb // 2, -1])
    o_ref, lse_ref = oracle_mod.fwd(op, x["q"], x["k"], x["v"], qsel=fsel)
    o, lse = to_np(fwd["o"]), to_np(fwd["lse"])
    m = np.isfinite(lse_ref)
    assert_parity(o[m], o_ref[m], "O")
    np.testing.assert_allclose(lse[m], lse_ref[m], rtol=0, atol=LSE_TOL)
    qsel = block_selection(w, [2, w.Hq - 1], [nb // 2, -1])
    ksel = block_selection(w, [0, 1], [1, nb // 2], kv=True)
    ref = dict(zip(("dq", "dk", "dv"), oracle_mod.bwd(op, x["q"], x["k"], x["v"], o, x["do"],
                                                        lse.astype(np.float64), qsel=qsel, ksel=ksel)))
    for key in ("dq", "dk", "dv"):
        g = to_np(bwd[key])
        mk = np.isfinite(ref[key])
        assert_parity(g[mk], ref[key][mk], key)
    # the criteria against exact attention on one query block of every head (O rows and dQ)
    csel = block_selection(w, list(range(w.Hq)), [nb // 2])
    ex = oracle_mod.pipeline(oracle_problem(oracle_mod, w), x["q"], x["k"], x["v"], x["do"], qsel=csel, exact=True)
    mq = np.isfinite(ex["dq"])
    rows = np.isfinite(ex["o"]) & mq
    assert cos(o[rows], ex["o"][rows]) >= 0.995
    assert cos(to_np(bwd["dq"])[mq], ex["dq"][mq]) >= 0.99


PLAIN = [
    W.small("plain_gqa_causal_300_d64", 1, 4, 2, 300, 64, True, 621, qk_norm=True, k_offset_sd=2.0),
    W.small("plain_outlier_gqa_nc_257_d128", 2, 3, 1, 257, 128, False, 622, outlier_frac=0.02),
    W.small("plain_outlier_causal_384_d128", 1, 6, 1, 384, 128, True, 623, outlier_frac=0.01),
    W.small("plain_n1_d64", 1, 2, 1, 1, 64, True, 624),
]


@pytest.mark.parametrize("w", PLAIN, ids=lambda w: w.name)
def test_plain_block_scales_forward_backward(oracle_mod, w):
    """qk_subexp=False: one FP32 scale per 128-token block of Q and K, all the way through."""
    x, xd = device_inputs(w)
    fwd = gpu_forward(w, xd, qk_subexp=False)
    bwd = gpu_backward(w, xd, fwd)
    assert fwd["status"] == 0 and bwd["status"] == 0
    check_values(oracle_mod, w, x, fwd, dict(qk_subexp=False))
    views = sb.quantized_views(fwd["prob"], fwd["saved"])
    for name in ("q", "k"):  # integer codes: no sub-scale anywhere
        a = views[name].float().cpu().numpy()
        assert np.all(a == np.round(a)), name
    ref = oracle_mod.pipeline(oracle_problem(oracle_mod, w, qk_subexp=False), x["q"], x["k"], x["v"], x["do"])
    assert_parity(to_np(fwd["o"]), ref["o"], "O")
    np.testing.assert_allclose(to_np(fwd["lse"]), ref["lse"], rtol=0, atol=LSE_TOL)
    for key in ("dq", "dk", "dv"):
        assert_parity(to_np(bwd[key]), ref[key], key)
