"""Long sequences: 1024 key blocks per head, beyond the named workloads.

The index arithmetic of the kernels (tile counts, per-tile offsets, the
backward's longest-first CTA order, the forward's query-tile pairs) at
N = 131067 (causal, d = 64, a ragged last block) and N = 65613 (non-causal,
d = 128, GQA 2:1), against the oracle on sampled blocks: O, LSE on the first,
a middle and the last query block; dQ on two query blocks; dK, dV on the first
and the last key block (whose causal column spans every query block).
"""
import numpy as np
import pytest

from bit_trainable_attention_gb300 import workloads as W
from _parity import (LSE_TOL, assert_parity, block_selection, device_inputs, gpu_backward, gpu_forward,
                     oracle_problem, to_np)

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("w", [W.small("long_causal_131067_d64", 1, 1, 1, 131067, 64, True, 901, qk_norm=True,
                                       k_offset_sd=2.0),
                               W.small("long_nc_65613_d128", 1, 2, 1, 65613, 128, False, 902, qk_norm=True)],
                         ids=lambda w: w.name)
def test_long_sequence_sampled(oracle_mod, w):
    x, xd = device_inputs(w)
    fwd = gpu_forward(w, xd)
    bwd = gpu_backward(w, xd, fwd)
    assert fwd["status"] == 0 and bwd["status"] == 0
    nb = (w.N + 127) // 128
    op = oracle_problem(oracle_mod, w)
    fsel = block_selection(w, [0], [0, nb // 2, -1])
    o_ref, lse_ref = oracle_mod.fwd(op, x["q"], x["k"], x["v"], qsel=fsel)
    o, lse = to_np(fwd["o"]), to_np(fwd["lse"])
    m = np.isfinite(lse_ref)
    assert m.sum() > 0
    assert_parity(o[m], o_ref[m], "O")
    np.testing.assert_allclose(lse[m], lse_ref[m], rtol=0, atol=LSE_TOL)
    qsel = block_selection(w, [w.Hq - 1], [nb // 3, -1])
    ksel = block_selection(w, [0], [0, -1], kv=True)
    ref = dict(zip(("dq", "dk", "dv"), oracle_mod.bwd(op, x["q"], x["k"], x["v"], o, x["do"], lse.astype(np.float64),
                                                        qsel=qsel, ksel=ksel)))
    for key in ("dq", "dk", "dv"):
        g = to_np(bwd[key])
        mk = np.isfinite(ref[key])
        assert mk.sum() > 0, key
        assert_parity(g[mk], ref[key][mk], key)
        assert np.all(np.isfinite(g)), key
