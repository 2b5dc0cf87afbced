"""Pins of the oracle's optional Q/K channel balancing (CPU only).

Channel balancing is this library's addition to SageBwd (after SmoothQuant,
listed under "Builds on" of the SageBwd page): per (batch, kv head, channel)
an exponent e = floor((E(aQ) - E(aK)) / 2), E the binary exponent of the
channel's largest |Q| (over the kv head's query heads) and largest |K - mean|,
moves magnitude from the larger side to the smaller one -- Q times 2^-e,
K times 2^e -- before the per-block quantizers.  Q K^T is unchanged exactly;
dQ is multiplied by 2^-e and dK by 2^e at the end.

* the exponents against hand-computed channel maxima (closed form);
* the balanced codes against the plain block quantizer applied to inputs
  pre-scaled by the same powers of two (exact in BF16);
* with every quantizer unrounded, the balanced pipeline is exact attention
  (pins the direction of the dQ / dK factors);
* on the channel-outlier recipe, balancing lifts the cosine similarity to
  exact attention over the criteria (O >= 0.995, gradients >= 0.99), and it
  leaves the outlier-free recipes at that level too.
"""
import numpy as np
import pytest
import torch

from bit_trainable_attention_gb300 import workloads as W


def cos(a, b):
    a = np.nan_to_num(np.asarray(a, np.float64)).ravel()
    b = np.nan_to_num(np.asarray(b, np.float64)).ravel()
    return float(a @ b / np.linalg.norm(a) / np.linalg.norm(b))


def bf16(a):
    return torch.tensor(np.asarray(a, np.float32)).to(torch.bfloat16)


def test_exponents_closed_form(oracle_mod):
    """Two query heads share one kv head; N = 3 tokens, d = 16 channels."""
    d, N = 16, 3
    q = np.zeros((1, 2, N, d), np.float32)
    k = np.zeros((1, 1, N, d), np.float32)
    # channel: (Q values head 0, Q values head 1, K values) -> expected e
    cases = [
        ([-8.0, 1.0, 0.5], [2.0, 0.0, 0.0], [0.5, -0.25, 0.0], 2),  # E(8)=3, E(.5)=-1: diff 4
        ([1.0, 0.0, 0.0], [0.5, 0.0, 0.0], [1.0, 0.0, 0.0], 0),  # equal exponents
        ([0.25, 0.0, 0.0], [0.0, 0.0, 0.0], [-2.0, 1.0, 0.0], -2),  # diff -3 -> floor(-1.5)
        ([0.0, 0.0, 0.0], [0.0, 0.0, 0.0], [5.0, 0.0, 0.0], 0),  # Q channel all zero
        ([7.0, 0.0, 0.0], [0.0, 0.0, 0.0], [0.0, 0.0, 0.0], 0),  # K channel all zero
        ([3.0, 0.0, 0.0], [0.0, 0.0, 0.0], [1.0, 0.0, 0.0], 0),  # E(3)=1, E(1)=0: floor(0.5)
        ([1.0, 0.0, 0.0], [0.0, -40.0, 0.0], [1.0, 0.0, 0.0], 2),  # max over heads: E(40)=5
        ([1.0, 0.0, 0.0], [0.0, 0.0, 0.0], [2.0 ** -10, 0.0, 0.0], 5),  # diff 10
        ([2.0 ** 127 * 1.5, 0.0, 0.0], [0.0, 0.0, 0.0], [2.0 ** -133, 0.0, 0.0], 126),  # 130, clamped
        ([2.0 ** -133, 0.0, 0.0], [0.0, 0.0, 0.0], [2.0 ** 127, 0.0, 0.0], -126),  # -130, clamped
        ([2.0 ** -130 * 3, 0.0, 0.0], [0.0, 0.0, 0.0], [1.0, 0.0, 0.0], -65),  # subnormal: E = -129
        ([1.0, -1.0, 0.0], [0.0, 0.0, 0.0], [-(2.0 ** 20) * 1.75, 0.0, 0.0], -10),  # K's max is negative
    ]
    for ch, (q0, q1, kk, _) in enumerate(cases):
        q[0, 0, :, ch], q[0, 1, :, ch], k[0, 0, :, ch] = q0, q1, kk
    p = oracle_mod.problem(1, 2, 1, N, d, False, smooth_k=False, balance_qk=True)
    r = oracle_mod.quantize_qk(p, bf16(q), bf16(k))
    expect = [c[3] for c in cases] + [0] * (d - len(cases))  # unused channels are all zero
    np.testing.assert_array_equal(r["e"][0], expect)
    p0 = oracle_mod.problem(1, 2, 1, N, d, False, smooth_k=False, balance_qk=False)
    assert not oracle_mod.quantize_qk(p0, bf16(q), bf16(k))["e"].any()


def test_exponents_use_the_smoothed_k(oracle_mod):
    """With K-smoothing the K side of the rule is max |K - mean|: K = (10, 10, 14)
    has mean 34/3 and max |K - mean| = 8/3 (exponent 1); raw max 14 has exponent 3."""
    d, N = 8, 3
    q = np.zeros((1, 1, N, d), np.float32)
    k = np.zeros((1, 1, N, d), np.float32)
    q[0, 0, 0, :] = 64.0  # E = 6 on every channel
    k[0, 0, :, :] = np.array([10.0, 10.0, 14.0])[:, None]
    for smooth, e in ((True, 2), (False, 1)):  # floor((6 - 1) / 2) = 2, floor((6 - 3) / 2) = 1
        p = oracle_mod.problem(1, 1, 1, N, d, False, smooth_k=smooth, balance_qk=True)
        np.testing.assert_array_equal(oracle_mod.quantize_qk(p, bf16(q), bf16(k))["e"], e)


OUTLIER = W.small("outlier_gqa", 1, 4, 2, 300, 64, True, 41, outlier_frac=0.03)


@pytest.mark.parametrize("smooth", [True, False])
def test_balanced_codes_equal_prescaled_inputs(oracle_mod, smooth):
    w = OUTLIER.with_(k_offset_sd=2.0)
    x = W.make_inputs(w)
    pb = oracle_mod.problem(w.B, w.Hq, w.Hkv, w.N, w.d, w.causal, smooth_k=smooth, balance_qk=True)
    r = oracle_mod.quantize_qk(pb, x["q"], x["k"])
    e = r["e"].reshape(w.B, w.Hkv, 1, w.d).astype(np.float64)
    assert (e != 0).sum() >= 2  # the outlier channels are balanced
    fq = torch.tensor(np.exp2(-e)).repeat_interleave(w.G, dim=1)
    fk = torch.tensor(np.exp2(e))
    qs = (x["q"].double() * fq).to(torch.bfloat16)
    ks = (x["k"].double() * fk).to(torch.bfloat16)
    assert torch.equal(qs.double() / fq, x["q"].double()) and torch.equal(ks.double() / fk, x["k"].double())
    p = oracle_mod.problem(w.B, w.Hq, w.Hkv, w.N, w.d, w.causal, smooth_k=smooth)
    qc, qsc, _ = oracle_mod.quantize(p, qs, w.B * w.Hq, False)
    kc, ksc, mu = oracle_mod.quantize(p, ks, w.B * w.Hkv, smooth)
    np.testing.assert_array_equal(r["q"], qc)
    np.testing.assert_array_equal(r["sq"].view(np.uint32), qsc.view(np.uint32))
    np.testing.assert_array_equal(r["k"], kc)
    np.testing.assert_array_equal(r["sk"].view(np.uint32), ksc.view(np.uint32))
    if smooth:  # the mean is the unscaled K's; scaling by a power of two commutes with it
        np.testing.assert_array_equal((r["mu"] * np.exp2(r["e"])).astype(np.float32), mu)


@pytest.mark.parametrize("w", [OUTLIER, W.small("outlier_mha_nc", 2, 2, 2, 200, 32, False, 42, outlier_frac=0.05,
                                                k_offset_sd=3.0)], ids=lambda w: w.name)
def test_unrounded_balanced_pipeline_is_exact_attention(oracle_mod, w):
    x = W.make_inputs(w)
    pe = oracle_mod.problem(w.B, w.Hq, w.Hkv, w.N, w.d, w.causal, exact_codes=True, balance_qk=True)
    assert oracle_mod.quantize_qk(pe, x["q"], x["k"])["e"].any()
    r = oracle_mod.pipeline(pe, x["q"], x["k"], x["v"], x["do"])
    p_plain = oracle_mod.problem(w.B, w.Hq, w.Hkv, w.N, w.d, w.causal, exact_codes=True)
    ref = oracle_mod.pipeline(p_plain, x["q"], x["k"], x["v"], x["do"], exact=True)
    for key in ("o", "dq", "dk", "dv"):
        np.testing.assert_allclose(r[key], ref[key], rtol=0, atol=1e-10 * np.abs(ref[key]).max(), err_msg=key)


def _cossims(oracle_mod, w, x, balance):
    p = oracle_mod.problem(w.B, w.Hq, w.Hkv, w.N, w.d, w.causal, balance_qk=balance)
    r = oracle_mod.pipeline(p, x["q"], x["k"], x["v"], x["do"])
    ex = oracle_mod.pipeline(p, x["q"], x["k"], x["v"], x["do"], exact=True)
    return {key: cos(r[key], ex[key]) for key in ("o", "dq", "dk", "dv")}


def test_balancing_restores_accuracy_on_channel_outliers(oracle_mod):
    """The long-context workload (12 query heads, 2 kv heads, d = 128, causal, 1%
    of the Q and K channels x20, no QK-norm) at 1024 tokens instead of 16384."""
    w = W.WORKLOADS["qwen15b"].with_(N=1024)
    x = W.make_inputs(w)
    plain = _cossims(oracle_mod, w, x, False)
    bal = _cossims(oracle_mod, w, x, True)
    assert plain["o"] < 0.995 and min(plain["dq"], plain["dk"]) < 0.99, plain  # the recipe defeats block scales
    assert bal["o"] >= 0.995, bal
    for key in ("dq", "dk", "dv"):
        assert bal[key] >= 0.99, (key, bal)
    for key in bal:
        assert bal[key] > plain[key], (key, plain, bal)


@pytest.mark.parametrize("w", [W.small("qknorm_gqa", 1, 4, 1, 384, 64, True, 44, qk_norm=True, k_offset_sd=2.0),
                               W.small("offset_nc", 1, 2, 2, 256, 64, False, 45, k_offset_sd=3.0)],
                         ids=lambda w: w.name)
def test_balancing_keeps_outlier_free_recipes_accurate(oracle_mod, w):
    x = W.make_inputs(w)
    bal = _cossims(oracle_mod, w, x, True)
    assert bal["o"] >= 0.995, bal
    for key in ("dq", "dk", "dv"):
        assert bal[key] >= 0.99, (key, bal)
