"""Error attribution on the GPU path (SAGEBWD_FLAG_BF16_*), against the oracle's bf16_mask.

Each flag makes one quantizer keep its scale but store the BF16 rounding of its scaled values
instead of INT8 codes.  Checked here:
* parity: for every flag the library's O, LSE, dQ, dK, dV meet the normwise tolerance of
  tests/_parity.py against the oracle run with the same quantizer in BF16, and the stored Q^, K^,
  V^ values equal the oracle's bit for bit when their flag is set;
* at full size (the 8K-token GQA workload), keeping dS in BF16 brings dQ and dK closer to FP32
  attention than keeping any other single quantizer in BF16 ("SageBwd: A Trainable Low-bit
  Attention", Abstract, finding (ii): the error comes mainly from dS).
"""
import numpy as np
import pytest
import torch

import bit_trainable_attention_gb300 as sb
from bit_trainable_attention_gb300 import workloads as W
from _parity import (LSE_TOL, assert_parity, cos, device_inputs, gpu_backward, gpu_forward, oracle_problem,
                     to_np)

pytestmark = pytest.mark.gpu

ORDER = ["q", "k", "v", "do", "p_fwd", "p_bwd", "ds"]  # the oracle's quantizer bits 0..6
CASES = [W.small("attr_gqa_causal_300_d64", 1, 4, 2, 300, 64, True, 1001, qk_norm=True, k_offset_sd=2.0),
         W.small("attr_outlier_nc_257_d128", 1, 3, 1, 257, 128, False, 1002, outlier_frac=0.02)]


@pytest.mark.parametrize("which", ORDER)
@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_bf16_quantizer_parity(oracle_mod, w, which):
    x, xd = device_inputs(w)
    fwd = gpu_forward(w, xd, flags=sb.FLAG_BF16[which])
    bwd = gpu_backward(w, xd, fwd)
    assert fwd["status"] == 0 and bwd["status"] == 0
    op = oracle_problem(oracle_mod, w)
    op.bf16_mask = 1 << ORDER.index(which)
    if which in ("q", "k"):
        ref = oracle_mod.quantize_qk(op, x["q"], x["k"])
        g = sb.quantized_views(fwd["prob"], fwd["saved"])[which].float().cpu().numpy()
        np.testing.assert_array_equal(g.reshape(ref[which].shape), ref[which])
    ref = oracle_mod.pipeline(op, x["q"], x["k"], x["v"], x["do"])
    assert_parity(to_np(fwd["o"]), ref["o"], "O")
    np.testing.assert_allclose(to_np(fwd["lse"]), ref["lse"], rtol=0, atol=LSE_TOL)
    for key in ("dq", "dk", "dv"):
        assert_parity(to_np(bwd[key]), ref[key], key)


def test_ds_carries_most_of_the_gradient_error_at_full_size():
    w = W.WORKLOADS["llama1b"]
    x, xd = device_inputs(w)
    q, k, v = (xd[n].float().requires_grad_(True) for n in ("q", "k", "v"))
    o = torch.nn.functional.scaled_dot_product_attention(q, k.repeat_interleave(w.G, 1),
                                                         v.repeat_interleave(w.G, 1), is_causal=w.causal)
    o.backward(xd["do"].float())
    ref = {"dq": q.grad.double().cpu().numpy(), "dk": k.grad.double().cpu().numpy()}
    del q, k, v, o
    torch.cuda.empty_cache()
    err = {}
    for which in ORDER:
        fwd = gpu_forward(w, xd, flags=sb.FLAG_BF16[which])
        bwd = gpu_backward(w, xd, fwd)
        assert fwd["status"] == 0 and bwd["status"] == 0
        err[which] = {key: 1.0 - cos(to_np(bwd[key]), ref[key]) for key in ("dq", "dk")}
    for key in ("dq", "dk"):
        best = min(err, key=lambda wh: err[wh][key])
        assert best == "ds", (key, err)
