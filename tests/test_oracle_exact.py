"""Pins of the oracle's exact FP64 attention (the full-precision reference).

Checked against a library special case (torch's FP64 scaled-dot-product
attention and its autograd) and against identities that hold for softmax
attention whatever its implementation: the derivative of the loss with
respect to the softmax scale (central finite differences), and the
linearity of the loss in V.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

from bit_trainable_attention_gb300 import workloads as W


def _torch_ref(x, w, sc):
    q = x["q"].double().requires_grad_(True)
    k = x["k"].double().requires_grad_(True)
    v = x["v"].double().requires_grad_(True)
    kk = k.repeat_interleave(w.G, dim=1)
    vv = v.repeat_interleave(w.G, dim=1)
    o = F.scaled_dot_product_attention(q, kk, vv, is_causal=w.causal, scale=sc)
    s = (q @ kk.transpose(-1, -2)) * sc
    if w.causal:
        s = s.masked_fill(torch.ones(w.N, w.N, dtype=torch.bool).triu(1), float("-inf"))
    lse = torch.logsumexp(s, dim=-1)
    o.backward(x["do"].double())
    return o.detach().numpy(), lse.detach().numpy(), q.grad.numpy(), k.grad.numpy(), v.grad.numpy()


CASES = [
    W.small("mha", 1, 2, 2, 37, 16, False, 1),
    W.small("gqa_causal", 2, 4, 2, 37, 16, True, 2, k_offset_sd=2.0),
    W.small("gqa3", 1, 6, 2, 130, 8, True, 3, qk_norm=True),
    W.small("one_token", 1, 2, 1, 1, 8, True, 4),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_exact_matches_torch_sdpa(oracle_mod, w):
    x = W.make_inputs(w)
    p = oracle_mod.problem(w.B, w.Hq, w.Hkv, w.N, w.d, w.causal)
    r = oracle_mod.pipeline(p, x["q"], x["k"], x["v"], x["do"], exact=True)
    o, lse, dq, dk, dv = _torch_ref(x, w, 1.0 / np.sqrt(w.d))
    for name, got, ref in [("o", r["o"], o), ("lse", r["lse"], lse), ("dq", r["dq"], dq), ("dk", r["dk"], dk),
                           ("dv", r["dv"], dv)]:
        np.testing.assert_allclose(got, ref, rtol=0, atol=1e-11 * max(1.0, np.abs(ref).max()), err_msg=name)


@pytest.mark.parametrize("w", CASES[:3], ids=lambda w: w.name)
def test_exact_gradient_identities(oracle_mod, w):
    """L(sc) = sum(O(sc) * dO).  dL/dsc = <dQ, Q>/sc = <dK, K>/sc (central
    differences), and L = <dV, V> because O is linear in V."""
    x = W.make_inputs(w)
    sc = 0.3
    qd, kd, vd = (x[n].double().numpy() for n in ("q", "k", "v"))
    dod = x["do"].double().numpy()

    def loss(scale):
        p = oracle_mod.problem(w.B, w.Hq, w.Hkv, w.N, w.d, w.causal, softmax_scale=scale)
        o, _ = oracle_mod.fwd(p, x["q"], x["k"], x["v"], exact=True)
        return float((o * dod).sum())

    p = oracle_mod.problem(w.B, w.Hq, w.Hkv, w.N, w.d, w.causal, softmax_scale=sc)
    r = oracle_mod.pipeline(p, x["q"], x["k"], x["v"], x["do"], exact=True)
    h = 1e-5
    fd = (loss(sc + h) - loss(sc - h)) / (2 * h)
    via_q = float((r["dq"] * qd).sum()) / sc
    via_k = float((r["dk"] * kd).sum()) / sc
    assert abs(fd - via_q) <= 1e-6 * max(1.0, abs(fd))
    assert abs(fd - via_k) <= 1e-6 * max(1.0, abs(fd))
    assert abs(loss(sc) - float((r["dv"] * vd).sum())) <= 1e-9 * max(1.0, abs(loss(sc)))


def test_exact_block_selection_matches_full(oracle_mod):
    """Selecting query / key blocks computes exactly the same rows as the full call."""
    w = W.small("sel", 1, 4, 2, 300, 16, True, 5)
    x = W.make_inputs(w)
    p = oracle_mod.problem(w.B, w.Hq, w.Hkv, w.N, w.d, w.causal)
    full = oracle_mod.pipeline(p, x["q"], x["k"], x["v"], x["do"], exact=True)
    nb = oracle_mod.nblocks(w.N)
    qsel = np.zeros(w.B * w.Hq * nb, np.uint8)
    qsel[3 * nb + 2] = 1  # head 3, last (ragged) query block
    ksel = np.zeros(w.B * w.Hkv * nb, np.uint8)
    ksel[0 * nb + 1] = 1  # kv head 0, middle key block
    part = oracle_mod.pipeline(p, x["q"], x["k"], x["v"], x["do"], qsel=qsel, ksel=ksel, exact=True)
    np.testing.assert_array_equal(part["dq"][0, 3, 256:], full["dq"][0, 3, 256:])
    np.testing.assert_array_equal(part["dk"][0, 0, 128:256], full["dk"][0, 0, 128:256])
    np.testing.assert_array_equal(part["dv"][0, 0, 128:256], full["dv"][0, 0, 128:256])
    assert np.isnan(part["dq"][0, 0]).all()
