"""GPU parity of the optional Q/K channel balancing (balance_qk) against the oracle.

The balancing exponents, the K means and the balanced Q/K codes and block
scales must equal the oracle's bit for bit; O, LSE, dQ, dK, dV must meet the
normwise tolerance of tests/_parity.py, like the unbalanced path.  On the
long-context channel-outlier recipe the balanced library must reach the
cosine-similarity criteria against exact attention (O >= 0.995, gradients
>= 0.99), and the full-size workload is checked on sampled blocks.
"""
import numpy as np
import pytest
import torch

import bit_trainable_attention_gb300 as sb
from bit_trainable_attention_gb300 import workloads as W
from _parity import (LSE_TOL, assert_parity, block_selection, cos, device_inputs, gpu_backward, gpu_forward,
                     oracle_problem, to_np)

pytestmark = pytest.mark.gpu

SMALL = [
    W.small("bal_outlier_gqa_causal_384_d128", 1, 6, 1, 384, 128, True, 401, outlier_frac=0.01),
    W.small("bal_outlier_gqa_nc_257_d64", 2, 4, 2, 257, 64, False, 402, outlier_frac=0.03, k_offset_sd=2.0),
    W.small("bal_qknorm_causal_300_d64", 1, 4, 2, 300, 64, True, 403, qk_norm=True, k_offset_sd=2.0),
    W.small("bal_n1_d128", 1, 2, 1, 1, 128, True, 404, outlier_frac=0.02),
    W.small("bal_n129_d128_nc", 1, 2, 2, 129, 128, False, 405, outlier_frac=0.02),
]


def check_balanced_quantization(oracle_mod, w, x, fwd, smooth_k=True):
    op = oracle_problem(oracle_mod, w, smooth_k, balance_qk=True)
    ref = oracle_mod.quantize_qk(op, x["q"], x["k"])
    views = sb.quantized_views(fwd["prob"], fwd["saved"])
    np.testing.assert_array_equal(views["e"].cpu().numpy(), ref["e"], err_msg="balancing exponents")
    if smooth_k:
        np.testing.assert_array_equal(views["mu"].cpu().numpy().view(np.uint32), ref["mu"].view(np.uint32),
                                      err_msg="k mean")
    for name in ("q", "k"):
        g = views[name].float().cpu().numpy().reshape(ref[name].shape)
        np.testing.assert_array_equal(g, ref[name].astype(np.float32), err_msg=f"{name} codes")
        gs = views["s" + name].cpu().numpy()
        np.testing.assert_array_equal(gs.view(np.uint32), ref["s" + name].view(np.uint32), err_msg=f"{name} scales")
    return ref


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_balanced_forward_backward_small(oracle_mod, w):
    x, xd = device_inputs(w)
    fwd = gpu_forward(w, xd, balance_qk=True)
    assert fwd["status"] == 0
    check_balanced_quantization(oracle_mod, w, x, fwd)
    bwd = gpu_backward(w, xd, fwd)
    assert bwd["status"] == 0
    op = oracle_problem(oracle_mod, w, balance_qk=True)
    ref = oracle_mod.pipeline(op, x["q"], x["k"], x["v"], x["do"])
    assert_parity(to_np(fwd["o"]), ref["o"], "O")
    np.testing.assert_allclose(to_np(fwd["lse"]), ref["lse"], rtol=0, atol=LSE_TOL)
    for key in ("dq", "dk", "dv"):
        assert_parity(to_np(bwd[key]), ref[key], key)


def test_balanced_without_smoothing(oracle_mod):
    w = W.small("bal_nosmooth", 1, 2, 1, 200, 64, True, 411, outlier_frac=0.03, k_offset_sd=2.0)
    x, xd = device_inputs(w)
    fwd = gpu_forward(w, xd, smooth_k=False, balance_qk=True)
    check_balanced_quantization(oracle_mod, w, x, fwd, smooth_k=False)
    bwd = gpu_backward(w, xd, fwd)
    op = oracle_problem(oracle_mod, w, smooth_k=False, balance_qk=True)
    ref = oracle_mod.pipeline(op, x["q"], x["k"], x["v"], x["do"])
    assert_parity(to_np(fwd["o"]), ref["o"], "O")
    for key in ("dq", "dk", "dv"):
        assert_parity(to_np(bwd[key]), ref[key], key)


def test_balancing_meets_the_cossim_criteria_on_channel_outliers(oracle_mod):
    """The long-context workload's recipe (GQA 6:1, d = 128, 1% of channels x20) at 1024 tokens, with
    one scale per Q/K block (the plain mode; the default sub-scales meet the criteria by themselves):
    unbalanced it misses the criteria, balanced it meets them, on the GPU as in the oracle."""
    w = W.WORKLOADS["qwen15b"].with_(N=1024)
    x, xd = device_inputs(w)
    op = oracle_problem(oracle_mod, w)
    ex = oracle_mod.pipeline(op, x["q"], x["k"], x["v"], x["do"], exact=True)
    got = {}
    for bal in (False, True):
        fwd = gpu_forward(w, xd, balance_qk=bal, qk_subexp=False)
        bwd = gpu_backward(w, xd, fwd)
        assert fwd["status"] == 0 and bwd["status"] == 0
        got[bal] = {"o": cos(to_np(fwd["o"]), ex["o"]), **{k: cos(to_np(bwd[k]), ex[k]) for k in ("dq", "dk", "dv")}}
    assert got[False]["o"] < 0.995, got
    assert got[True]["o"] >= 0.995, got
    for key in ("dq", "dk", "dv"):
        assert got[True][key] >= 0.99, (key, got)


def test_balanced_autograd_function(oracle_mod):
    w = W.small("bal_autograd", 1, 4, 2, 200, 128, True, 412, outlier_frac=0.02)
    x, xd = device_inputs(w)
    q, k, v = (xd[n].clone().requires_grad_(True) for n in ("q", "k", "v"))
    o = sb.attention(q, k, v, causal=True, balance_qk=True)
    o.backward(xd["do"])
    op = oracle_problem(oracle_mod, w, balance_qk=True)
    ref = oracle_mod.pipeline(op, x["q"], x["k"], x["v"], x["do"])
    assert_parity(to_np(o), ref["o"], "O")
    for name, t in (("dq", q), ("dk", k), ("dv", v)):
        assert_parity(to_np(t.grad), ref[name], name)


def test_balanced_full_size_qwen15b_sampled(oracle_mod):
    """The long-context workload at full size in the bench's launch configuration: exponents, means,
    codes and scales in full; O and LSE on sampled query blocks; the backward stage-wise, i.e. the
    oracle's backward fed the library's own O and LSE, on sampled dQ and dK / dV blocks.

    Stage-wise because at this size the first key block, which all 16384 queries of six heads
    see, sums about 10^5 rows of dS: forward differences that are within the O / LSE tolerance
    move its dK by up to ~4e-3 (relative L2) when each side runs its own forward, while the
    backward itself agrees to ~1e-5 on identical inputs."""
    w = W.WORKLOADS["qwen15b"]
    x, xd = device_inputs(w)
    fwd = gpu_forward(w, xd, balance_qk=True)
    bwd = gpu_backward(w, xd, fwd)
    assert fwd["status"] == 0 and bwd["status"] == 0
    check_balanced_quantization(oracle_mod, w, x, fwd)
    nb = (w.N + 127) // 128
    op = oracle_problem(oracle_mod, w, balance_qk=True)
    fsel = block_selection(w, [0, w.Hq - 1], [0, nb // 2, -1])
    o_ref, lse_ref = oracle_mod.fwd(op, x["q"], x["k"], x["v"], qsel=fsel)
    o, lse = to_np(fwd["o"]), to_np(fwd["lse"])
    m = np.isfinite(lse_ref)
    assert_parity(o[m], o_ref[m], "O")
    np.testing.assert_allclose(lse[m], lse_ref[m], rtol=0, atol=LSE_TOL)
    qsel = block_selection(w, [w.Hq - 1], [nb // 2, -1])
    ksel = block_selection(w, [1], [0, 1, -1], kv=True)
    ref = dict(zip(("dq", "dk", "dv"), oracle_mod.bwd(op, x["q"], x["k"], x["v"], o, x["do"],
                                                        lse.astype(np.float64), qsel=qsel, ksel=ksel)))
    for key in ("dq", "dk", "dv"):
        g = to_np(bwd[key])
        mk = np.isfinite(ref[key])
        assert mk.sum() > 0, key
        assert_parity(g[mk], ref[key][mk], key)
        assert np.all(np.isfinite(g)), key
