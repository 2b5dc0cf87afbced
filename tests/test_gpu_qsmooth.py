"""GPU parity of the optional Q-smoothing (smooth_q) against the oracle.

"SageBwd: A Trainable Low-bit Attention" (Abstract, finding (iv)) names
Q-smoothing as optional, with limited benefit in pre-training.  The library's
reading: each 128-token block of a query head subtracts its channel means
before quantizing; the logits gain mean_Q(block) . K'_k in FP32 and dK gains
scale * s_dS * (column sum of the dS codes) * mean_Q per tile.

* the Q codes, block scales and block means equal the oracle's bit for bit
  (the means are exact sums rounded once);
* the logit terms agree with the oracle's FP64 dot products to FP32 rounding
  (the kernel sums d FP32 products);
* O, LSE, dQ, dK, dV meet the normwise tolerance of tests/_parity.py, causal
  and not, GQA, ragged, d = 64 and 128, with the dS sub-scales and the Q/K
  sub-scales as well;
* on queries with a per-channel offset the library's gradients get closer to
  exact attention with Q-smoothing than without (the direction the oracle pins).
"""
import numpy as np
import pytest

import bit_trainable_attention_gb300 as sb
from bit_trainable_attention_gb300 import workloads as W
from _parity import (LSE_TOL, assert_parity, block_selection, cos, device_inputs, gpu_backward, gpu_forward,
                     oracle_problem, to_np)

pytestmark = pytest.mark.gpu

QS = dict(smooth_q=True)
CASES = [
    (W.small("qs_gqa_causal_300_d64", 1, 4, 2, 300, 64, True, 701, k_offset_sd=2.0, q_offset_sd=3.0), QS),
    (W.small("qs_gqa_causal_384_d128", 1, 6, 1, 384, 128, True, 702, q_offset_sd=2.0), QS),
    (W.small("qs_mha_nc_257_d64", 2, 2, 2, 257, 64, False, 703, k_offset_sd=3.0, q_offset_sd=3.0), QS),
    (W.small("qs_nc_129_d128", 1, 2, 2, 129, 128, False, 704, qk_norm=True, q_offset_sd=1.0), QS),
    (W.small("qs_subexp_causal_300_d64", 1, 4, 2, 300, 64, True, 705, outlier_frac=0.03, q_offset_sd=3.0),
     dict(smooth_q=True, ds_subexp=True, qk_subexp=True)),
    (W.small("qs_subexp_nc_200_d128", 1, 4, 4, 200, 128, False, 706, q_offset_sd=3.0),
     dict(smooth_q=True, ds_subexp=True)),
    (W.small("qs_n1_d64", 1, 2, 1, 1, 64, True, 707, q_offset_sd=3.0), QS),
]


def check_quantized(oracle_mod, w, x, fwd, kw):
    op = oracle_problem(oracle_mod, w, **{k: v for k, v in kw.items() if k != "ds_subexp"})
    ref = oracle_mod.quantize_qk(op, x["q"], x["k"])
    terms = oracle_mod.qsmooth_terms(op, x["q"], x["k"])
    views = sb.quantized_views(fwd["prob"], fwd["saved"])
    for name in ("q", "k"):
        g = views[name].float().cpu().numpy().reshape(ref[name].shape)
        np.testing.assert_array_equal(g, ref[name], err_msg=f"{name} codes")
        np.testing.assert_array_equal(views["s" + name].cpu().numpy().view(np.uint32),
                                      ref["s" + name].view(np.uint32), err_msg=f"{name} scales")
    np.testing.assert_array_equal(views["qm"].cpu().numpy().view(np.uint32), terms["qm"].view(np.uint32),
                                  err_msg="block means of Q")
    # the logit terms the kernels read, for every (query block, key) they read
    nb = (w.N + 127) // 128
    qb = views["qb"].cpu().numpy()[:, :, :w.N]
    ib = np.arange(nb)[:, None]
    seen = (np.arange(w.N)[None, :] // 128 <= ib) if w.causal else np.ones((nb, w.N), bool)
    ref_b = terms["bias"]
    tol = 1e-5 * max(1.0, float(np.abs(ref_b).max()))
    err = np.abs(qb - ref_b)[:, seen]
    assert err.max() <= tol, f"logit terms differ by {err.max():.3e}"


@pytest.mark.parametrize("w,kw", CASES, ids=lambda c: c.name if hasattr(c, "name") else "-".join(sorted(c)))
def test_q_smoothing_forward_backward_small(oracle_mod, w, kw):
    x, xd = device_inputs(w)
    fwd = gpu_forward(w, xd, **kw)
    bwd = gpu_backward(w, xd, fwd)
    assert fwd["status"] == 0 and bwd["status"] == 0
    check_quantized(oracle_mod, w, x, fwd, kw)
    ref = oracle_mod.pipeline(oracle_problem(oracle_mod, w, **kw), x["q"], x["k"], x["v"], x["do"])
    assert_parity(to_np(fwd["o"]), ref["o"], "O")
    np.testing.assert_allclose(to_np(fwd["lse"]), ref["lse"], rtol=0, atol=LSE_TOL)
    for key in ("dq", "dk", "dv"):
        assert_parity(to_np(bwd[key]), ref[key], key)


def test_q_smoothing_without_k_smoothing(oracle_mod):
    w = W.small("qs_nosmoothk", 1, 2, 1, 200, 64, True, 711, k_offset_sd=1.0, q_offset_sd=3.0)
    x, xd = device_inputs(w)
    fwd = gpu_forward(w, xd, smooth_k=False, smooth_q=True)
    bwd = gpu_backward(w, xd, fwd)
    assert fwd["status"] == 0 and bwd["status"] == 0
    ref = oracle_mod.pipeline(oracle_problem(oracle_mod, w, smooth_k=False, smooth_q=True), x["q"], x["k"], x["v"],
                              x["do"])
    assert_parity(to_np(fwd["o"]), ref["o"], "O")
    for key in ("dq", "dk", "dv"):
        assert_parity(to_np(bwd[key]), ref[key], key)


def test_q_smoothing_helps_with_query_offsets(oracle_mod):
    """Per (head, channel) query offsets of sd 3 on a d = 128 GQA workload: against exact attention
    the library's O and dK get closer with Q-smoothing than without."""
    w = W.small("qs_helps", 1, 4, 2, 512, 128, True, 712, k_offset_sd=3.0, q_offset_sd=3.0)
    x, xd = device_inputs(w)
    ex = oracle_mod.pipeline(oracle_problem(oracle_mod, w), x["q"], x["k"], x["v"], x["do"], exact=True)
    res = {}
    for name, kw in (("plain", {}), ("smooth_q", QS)):
        fwd = gpu_forward(w, xd, **kw)
        bwd = gpu_backward(w, xd, fwd)
        assert fwd["status"] == 0 and bwd["status"] == 0
        res[name] = {"o": 1 - cos(to_np(fwd["o"]), ex["o"]), "dk": 1 - cos(to_np(bwd["dk"]), ex["dk"])}
    for key in ("o", "dk"):
        assert res["smooth_q"][key] < res["plain"][key], res


def test_q_smoothing_full_size_video(oracle_mod):
    """The video workload (non-causal, 17776 tokens, ragged last block) at full size with
    Q-smoothing: block means and codes in full; O / LSE on sampled query blocks; the backward on
    sampled blocks."""
    w = W.WORKLOADS["videodit"].with_(q_offset_sd=2.0)
    x, xd = device_inputs(w)
    fwd = gpu_forward(w, xd, **QS)
    bwd = gpu_backward(w, xd, fwd)
    assert fwd["status"] == 0 and bwd["status"] == 0
    op = oracle_problem(oracle_mod, w, **QS)
    ref_q = oracle_mod.quantize_qk(op, x["q"], x["k"])
    views = sb.quantized_views(fwd["prob"], fwd["saved"])
    np.testing.assert_array_equal(views["q"].float().cpu().numpy().reshape(ref_q["q"].shape), ref_q["q"])
    nb = (w.N + 127) // 128
    fsel = block_selection(w, [0, w.Hq - 1], [0, nb // 2, -1])
    o_ref, lse_ref = oracle_mod.fwd(op, x["q"], x["k"], x["v"], qsel=fsel)
    o, lse = to_np(fwd["o"]), to_np(fwd["lse"])
    m = np.isfinite(lse_ref)
    assert_parity(o[m], o_ref[m], "O")
    np.testing.assert_allclose(lse[m], lse_ref[m], rtol=0, atol=LSE_TOL)
    qsel = block_selection(w, [1], [nb // 2, -1])
    ksel = block_selection(w, [1], [0, -1], kv=True)
    ref = dict(zip(("dq", "dk", "dv"), oracle_mod.bwd(op, x["q"], x["k"], x["v"], o, x["do"],
                                                        lse.astype(np.float64), qsel=qsel, ksel=ksel)))
    for key in ("dq", "dk", "dv"):
        g = to_np(bwd[key])
        mk = np.isfinite(ref[key])
        assert_parity(g[mk], ref[key][mk], key)
