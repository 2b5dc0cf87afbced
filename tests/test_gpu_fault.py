"""Failure detection on the GPU without a GPU fault.

The problem flag SAGEBWD_FLAG_DROP_ONE_LOAD makes the forward kernel's producer
skip the TMA load of one K tile (and the backward kernel's that of one dO^ tile).  Nothing then completes that tile's mbarrier:
the waits behind it run out after the problem's short wait_timeout_ms, record
SAGEBWD_ERR_TIMEOUT with the site of the first wait that gave up, raise the
CTA's abort flag so every other role leaves its loop, drain the copies and MMAs
already issued and free TMEM.  The call must come back with that status, the
CUDA context must stay usable, and the next ordinary call must be correct.
"""
import time

import numpy as np
import pytest
import torch

import bit_trainable_attention_gb300 as sb
from bit_trainable_attention_gb300 import workloads as W
from _parity import LSE_TOL, assert_parity, device_inputs, gpu_backward, gpu_forward, oracle_problem, to_np

pytestmark = pytest.mark.gpu

SAGEBWD_ERR_TIMEOUT = 5
SAGEBWD_FLAG_DROP_ONE_LOAD = 0x1
FWD_SITES = range(1, 10)  # the forward kernel's wait sites (Q .. O empty)


@pytest.mark.parametrize("causal", [False, True], ids=["noncausal", "causal"])
def test_dropped_load_times_out_and_the_context_survives(oracle_mod, causal):
    # 512 tokens: 4 key tiles, so every CTA with a second key tile waits for the dropped one
    w = W.small(f"fault_{int(causal)}", 1, 2, 2, 512, 64, causal, 301)
    x, xd = device_inputs(w)
    t0 = time.time()
    bad = gpu_forward(w, xd, flags=SAGEBWD_FLAG_DROP_ONE_LOAD, timeout_ms=100)
    elapsed = time.time() - t0
    assert bad["status"] == SAGEBWD_ERR_TIMEOUT, sb.sagebwd_status_string(bad["status"])
    assert bad["word"] & 0xFF == SAGEBWD_ERR_TIMEOUT
    assert (bad["word"] >> 8) in FWD_SITES, hex(bad["word"])
    assert elapsed < 30.0  # bounded: the waits gave up instead of hanging
    assert sb.sagebwd_status_string(bad["status"]).strip()

    # the context is still usable: an ordinary forward and backward on the same inputs
    torch.cuda.synchronize()
    good = gpu_forward(w, xd)
    assert good["status"] == 0
    op = oracle_problem(oracle_mod, w)
    o_ref, lse_ref = oracle_mod.fwd(op, x["q"], x["k"], x["v"])
    assert_parity(to_np(good["o"]), o_ref, "O")
    np.testing.assert_allclose(to_np(good["lse"]), lse_ref, rtol=0, atol=LSE_TOL)
    bwd = gpu_backward(w, xd, good)
    assert bwd["status"] == 0


BWD_SITES = range(16, 39)  # the backward kernel's wait sites (K/V .. dP^T)


@pytest.mark.parametrize("d", [64, 128])
def test_backward_dropped_load_times_out_and_the_context_survives(oracle_mod, d):
    """The same flag makes the backward kernel skip the dO^ load of each CTA's second tile: the MMA
    issuer's wait for it runs out, every other role leaves on the abort flag, the copies and MMAs in
    flight are drained and TMEM is freed.  The call reports a backward wait site, and an ordinary
    backward afterwards is correct."""
    # 384 tokens, two query heads per kv head: every CTA has at least two tiles
    w = W.small(f"fault_bwd_{d}", 1, 4, 2, 384, d, False, 303)
    x, xd = device_inputs(w)
    fwd = gpu_forward(w, xd)
    assert fwd["status"] == 0
    prob = fwd["prob"]
    prob.flags = SAGEBWD_FLAG_DROP_ONE_LOAD
    prob.wait_timeout_ms = 100
    t0 = time.time()
    bad = gpu_backward(w, xd, fwd)
    elapsed = time.time() - t0
    assert bad["status"] == SAGEBWD_ERR_TIMEOUT, sb.sagebwd_status_string(bad["status"])
    assert (bad["word"] >> 8) in BWD_SITES, hex(bad["word"])
    assert elapsed < 30.0
    # the context is still usable: the ordinary backward of the same forward matches the oracle
    torch.cuda.synchronize()
    prob.flags = 0
    prob.wait_timeout_ms = 0
    good = gpu_backward(w, xd, fwd)
    assert good["status"] == 0
    op = oracle_problem(oracle_mod, w)
    ref = oracle_mod.pipeline(op, x["q"], x["k"], x["v"], x["do"])
    for key in ("dq", "dk", "dv"):
        assert_parity(to_np(good[key]), ref[key], key)


def test_autograd_path_reports_a_device_timeout():
    """The autograd path does not synchronize after each call; the status word of every call is read
    back behind its kernels and a non-OK word raises at the next call (here the backward of the same
    forward) or at check_errors()."""
    w = W.small("fault_autograd", 1, 2, 2, 512, 64, False, 302)
    _, xd = device_inputs(w)
    q, k, v = (xd[n].clone().requires_grad_(True) for n in ("q", "k", "v"))
    o = sb.attention(q, k, v, flags=SAGEBWD_FLAG_DROP_ONE_LOAD, wait_timeout_ms=100)
    torch.cuda.synchronize()
    with pytest.raises(RuntimeError, match="TIMEOUT"):
        o.backward(xd["do"])
    sb.check_errors()  # reported once
    o = sb.attention(q, k, v, flags=SAGEBWD_FLAG_DROP_ONE_LOAD, wait_timeout_ms=100)
    with pytest.raises(sb.SageBwdError) as err:
        sb.check_errors()
    assert err.value.code == SAGEBWD_ERR_TIMEOUT
    # ordinary calls afterwards raise nothing
    q.grad = k.grad = v.grad = None
    sb.attention(q, k, v).backward(xd["do"])
    sb.check_errors()
    assert q.grad is not None and torch.isfinite(q.grad.float()).all()
