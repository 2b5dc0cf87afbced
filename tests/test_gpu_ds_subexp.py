"""GPU parity of the optional dS sub-scales (ds_subexp) against the oracle.

With ds_subexp the backward kernel refines each key's dS codes within a group
of 32 queries of a tile by a power of two (see the oracle's ds_subexp_of);
dQ, dK, dV must meet the normwise tolerance of tests/_parity.py against the
oracle with the same option, on small shapes that cover both head dims,
causal and not, GQA, ragged tails and N = 1, and on sampled blocks of a
full-size workload.  Against exact attention the option must bring dQ and dK
closer than the per-tile scale does.
"""
import numpy as np
import pytest

import bit_trainable_attention_gb300 as sb
from bit_trainable_attention_gb300 import workloads as W
from _parity import (assert_parity, block_selection, cos, device_inputs, gpu_backward, gpu_forward, oracle_problem,
                     to_np)

pytestmark = pytest.mark.gpu

SMALL = [
    W.small("dsx_gqa_causal_300_d64", 1, 4, 2, 300, 64, True, 501, qk_norm=True, k_offset_sd=2.0),
    W.small("dsx_gqa_noncausal_257_d128", 2, 3, 1, 257, 128, False, 502, k_offset_sd=3.0),
    W.small("dsx_mha_causal_384_d128", 1, 2, 2, 384, 128, True, 503, qk_norm=True),
    W.small("dsx_n1_d64", 1, 2, 1, 1, 64, True, 504),
    W.small("dsx_n129_d64_noncausal", 1, 2, 2, 129, 64, False, 505, qk_norm=True),
]


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_ds_subexp_backward_small(oracle_mod, w):
    x, xd = device_inputs(w)
    fwd = gpu_forward(w, xd, ds_subexp=True)
    bwd = gpu_backward(w, xd, fwd)
    assert fwd["status"] == 0 and bwd["status"] == 0
    op = oracle_problem(oracle_mod, w, ds_subexp=True)
    ref = oracle_mod.pipeline(op, x["q"], x["k"], x["v"], x["do"])
    for key in ("dq", "dk", "dv"):
        assert_parity(to_np(bwd[key]), ref[key], key)


def test_ds_subexp_is_closer_to_exact(oracle_mod):
    w = W.WORKLOADS["llama1b"].with_(Hq=8, Hkv=2, N=1024)
    x, xd = device_inputs(w)
    ex = oracle_mod.pipeline(oracle_problem(oracle_mod, w), x["q"], x["k"], x["v"], x["do"], exact=True)
    err = {}
    for on in (False, True):
        fwd = gpu_forward(w, xd, ds_subexp=on)
        bwd = gpu_backward(w, xd, fwd)
        err[on] = {k: 1 - cos(to_np(bwd[k]), ex[k]) for k in ("dq", "dk")}
    for key in ("dq", "dk"):
        assert err[True][key] * 2.5 < err[False][key], err


def test_ds_subexp_full_size_sampled(oracle_mod):
    """The 8K-token GQA workload in the bench's launch configuration, dQ and dK / dV on
    sampled blocks, stage-wise (the oracle's backward reads the library's O and LSE)."""
    w = W.WORKLOADS["llama1b"]
    x, xd = device_inputs(w)
    fwd = gpu_forward(w, xd, ds_subexp=True)
    bwd = gpu_backward(w, xd, fwd)
    assert fwd["status"] == 0 and bwd["status"] == 0
    nb = (w.N + 127) // 128
    qsel = block_selection(w, [w.Hq - 1], [nb // 2, -1])
    ksel = block_selection(w, [0], [0, -1], kv=True)
    op = oracle_problem(oracle_mod, w, ds_subexp=True)
    o, lse = to_np(fwd["o"]), to_np(fwd["lse"]).astype(np.float64)
    ref = dict(zip(("dq", "dk", "dv"), oracle_mod.bwd(op, x["q"], x["k"], x["v"], o, x["do"], lse, qsel=qsel,
                                                        ksel=ksel)))
    for key in ("dq", "dk", "dv"):
        g = to_np(bwd[key])
        m = np.isfinite(ref[key])
        assert m.sum() > 0, key
        assert_parity(g[m], ref[key][m], key)
