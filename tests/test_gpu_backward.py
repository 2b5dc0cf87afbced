"""GPU parity of the fused backward (and the whole forward + backward
pipeline) against the oracle.

The library and the oracle each run their own forward and then their own
backward from the same seeded inputs (the library's backward consumes the
library's O and LSE, the oracle's the oracle's), so every stage is compared
as it is used.  dQ, dK, dV must meet the normwise tolerance of
tests/_parity.py; the quantized dO codes and scales and D = rowsum(dO * O)
are checked too.  Full-size workloads are checked on sampled query blocks
(dQ) and key blocks (dK, dV).
"""
import numpy as np
import pytest
import torch

import bit_trainable_attention_gb300 as sb
from bit_trainable_attention_gb300 import workloads as W
from _parity import (assert_parity, cos, device_inputs, gpu_backward, gpu_forward, oracle_problem,
                     to_np)

pytestmark = pytest.mark.gpu

SMALL = [
    W.WORKLOADS["tiny"],
    W.small("gqa_causal_300_d64", 1, 4, 2, 300, 64, True, 201, qk_norm=True, k_offset_sd=2.0),
    W.small("gqa_noncausal_257_d128", 2, 3, 1, 257, 128, False, 202, k_offset_sd=3.0),
    W.small("mha_causal_384_d128", 1, 2, 2, 384, 128, True, 203, qk_norm=True),
    W.small("n1_d64", 1, 2, 1, 1, 64, True, 204),
    W.small("n129_d128_noncausal", 1, 2, 2, 129, 128, False, 205, qk_norm=True),
    W.small("n127_d64_causal_b2", 2, 2, 2, 127, 64, True, 206),
    W.small("gqa6_causal_520_d128", 1, 6, 1, 520, 128, True, 207, outlier_frac=0.01),
    W.small("gqa8_causal_260_d64", 1, 8, 1, 260, 64, True, 208, qk_norm=True, k_offset_sd=2.0),
    W.small("gqa12_noncausal_384_d64_b2", 2, 12, 1, 384, 64, False, 209, k_offset_sd=3.0),
]


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_backward_small(oracle_mod, w):
    x, xd = device_inputs(w)
    fwd = gpu_forward(w, xd)
    bwd = gpu_backward(w, xd, fwd)
    assert fwd["status"] == 0 and bwd["status"] == 0
    op = oracle_problem(oracle_mod, w)
    ref = oracle_mod.pipeline(op, x["q"], x["k"], x["v"], x["do"])
    errs = {}
    for key in ("dq", "dk", "dv"):
        errs[key] = assert_parity(to_np(bwd[key]), ref[key], key)
    if w.outlier_frac == 0 and w.N > 1:
        ex = oracle_mod.pipeline(op, x["q"], x["k"], x["v"], x["do"], exact=True)
        for key in ("dq", "dk", "dv"):
            assert cos(to_np(bwd[key]), ex[key]) >= 0.99, key


def test_backward_preprocess(oracle_mod):
    """D = rowsum(dO * O) in FP32 and the dO block quantization (bit-exact codes and scales)."""
    w = W.small("prep", 1, 3, 1, 300, 128, True, 211)
    x, xd = device_inputs(w)
    fwd = gpu_forward(w, xd)
    prob = fwd["prob"]
    ws = sb.empty_bytes(sb.sagebwd_workspace_bytes(prob, 1), "cuda")
    sb.sagebwd_bwd_prepare(prob, fwd["o"], xd["do"], ws)
    torch.cuda.synchronize()
    al = lambda n: (n + 255) // 256 * 256  # noqa: E731
    nb = 3
    off_d = 256
    off_doq = off_d + al(w.B * w.Hq * w.N * 4)
    off_sdo = off_doq + al(w.B * w.Hq * w.N * w.d * 2)
    Dg = ws[off_d:off_d + w.B * w.Hq * w.N * 4].view(torch.float32).cpu().numpy()
    doq = ws[off_doq:off_doq + w.B * w.Hq * w.N * w.d * 2].view(torch.bfloat16).float().cpu().numpy()
    sdo = ws[off_sdo:off_sdo + w.B * w.Hq * nb * 4].view(torch.float32).cpu().numpy()
    op = oracle_problem(oracle_mod, w)
    codes, scales, _ = oracle_mod.quantize(op, x["do"], w.B * w.Hq, False)
    np.testing.assert_array_equal(doq.reshape(codes.shape), codes.astype(np.float32))
    np.testing.assert_array_equal(sdo.view(np.uint32), scales.reshape(-1).view(np.uint32))
    Dref = (x["do"].double() * fwd["o"].double().cpu()).sum(-1).numpy().reshape(-1)
    np.testing.assert_allclose(Dg, Dref, rtol=1e-5, atol=1e-5 * np.abs(Dref).max())


def test_backward_stages_equal_single_call(oracle_mod):
    """prepare + attention + finish on one stream is the same computation as sagebwd_bwd."""
    w = W.small("stages", 1, 4, 2, 260, 64, True, 212, qk_norm=True)
    _, xd = device_inputs(w)
    fwd = gpu_forward(w, xd)
    a = gpu_backward(w, xd, fwd)
    prob = fwd["prob"]
    ws = sb.empty_bytes(sb.sagebwd_workspace_bytes(prob, 1), "cuda")
    dq, dk, dv = torch.empty_like(xd["q"]), torch.empty_like(xd["k"]), torch.empty_like(xd["v"])
    sb.sagebwd_bwd_prepare(prob, fwd["o"], xd["do"], ws)
    sb.sagebwd_bwd_attention(prob, xd["v"], xd["do"], fwd["lse"], fwd["saved"], dk, dv, ws)
    sb.sagebwd_bwd_finish(prob, fwd["saved"], dq, dk, dv, ws)
    torch.cuda.synchronize()
    assert torch.equal(dk, a["dk"]) and torch.equal(dv, a["dv"])
    # dQ is summed with FP32 atomics: equal up to the summation order
    np.testing.assert_allclose(to_np(dq), to_np(a["dq"]), rtol=0, atol=2e-3 * float(a["dq"].abs().max()))


def test_autograd_function(oracle_mod):
    w = W.small("autograd", 1, 4, 2, 200, 64, True, 213, qk_norm=True, k_offset_sd=2.0)
    x, xd = device_inputs(w)
    q, k, v = (xd[n].clone().requires_grad_(True) for n in ("q", "k", "v"))
    o = sb.attention(q, k, v, causal=True)
    o.backward(xd["do"])
    op = oracle_problem(oracle_mod, w)
    ref = oracle_mod.pipeline(op, x["q"], x["k"], x["v"], x["do"])
    assert_parity(to_np(o), ref["o"], "O")
    assert_parity(to_np(q.grad), ref["dq"], "dq")
    assert_parity(to_np(k.grad), ref["dk"], "dk")
    assert_parity(to_np(v.grad), ref["dv"], "dv")


@pytest.mark.parametrize("name", ["pretrain", "llama1b", "qwen15b", "videodit"])
def test_backward_full_size_sampled(oracle_mod, name):
    w = W.WORKLOADS[name]
    x, xd = device_inputs(w)
    fwd = gpu_forward(w, xd)
    bwd = gpu_backward(w, xd, fwd)
    assert fwd["status"] == 0 and bwd["status"] == 0
    nb = (w.N + 127) // 128
    # bounded oracle work: in batch 0, two query blocks of the last query head and two key blocks of
    # kv head 0; in the last batch, one query block of the last query head and one key block of the
    # last kv head (a batch- or head-stride error shows there)
    qsel = np.zeros((w.B, w.Hq, nb), np.uint8)
    ksel = np.zeros((w.B, w.Hkv, nb), np.uint8)
    qsel[0, w.Hq - 1, [nb - 1, nb // 2]] = 1
    ksel[0, 0, [0, nb - 1]] = 1
    qsel[w.B - 1, w.Hq - 1, nb // 3] = 1
    ksel[w.B - 1, w.Hkv - 1, (2 * nb) // 3] = 1
    qsel, ksel = qsel.reshape(-1), ksel.reshape(-1)
    op = oracle_problem(oracle_mod, w)
    ref = oracle_mod.pipeline(op, x["q"], x["k"], x["v"], x["do"], qsel=qsel, ksel=ksel)
    for key in ("dq", "dk", "dv"):
        g = to_np(bwd[key])
        m = np.isfinite(ref[key])
        assert m.sum() > 0, key
        assert_parity(g[m], ref[key][m], key)
        assert np.all(np.isfinite(g)), key
