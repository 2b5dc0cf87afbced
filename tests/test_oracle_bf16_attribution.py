"""Pins of the oracle's per-quantizer BF16 mode (bf16_mask), the error-attribution switch.

With a quantizer's bit set, that quantizer keeps its scale but stores the BF16 rounding of the
scaled value instead of its INT8 code.  Pinned here against what does not come from the oracle:
* the stored Q and K values equal torch's own FP32 -> bfloat16 conversion of x * (127 / max) (the
  scale computed in FP32 as the quantizer reading fixes it);
* with every quantizer in BF16 the pipeline is exact attention up to BF16 rounding of the operands
  (relative L2 error well below the INT8 pipeline's, against torch FP64 attention);
* error attribution: keeping dS in BF16 removes more of the dQ/dK error than keeping any other
  single quantizer in BF16 ("SageBwd: A Trainable Low-bit Attention", Abstract, finding (ii): the
  error comes mainly from dS).
"""
import numpy as np
import torch

from bit_trainable_attention_gb300 import workloads as W

W_SMALL = W.small("bf16attr", 1, 4, 2, 384, 64, True, 901, qk_norm=True, k_offset_sd=2.0)


def exact_attention(x, w):
    q, k, v, do = (x[n].double().requires_grad_(n != "do") for n in ("q", "k", "v", "do"))
    kk, vv = k.repeat_interleave(w.G, 1), v.repeat_interleave(w.G, 1)
    o = torch.nn.functional.scaled_dot_product_attention(q, kk, vv, is_causal=w.causal)
    o.backward(do)
    return {"o": o.detach().numpy(), "dq": q.grad.numpy(), "dk": k.grad.numpy(), "dv": v.grad.numpy()}


def rel(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def test_bf16_values_are_torch_bfloat16_of_the_scaled_inputs(oracle_mod):
    w = W.small("bf16q", 1, 2, 2, 200, 64, False, 902)
    x = W.make_inputs(w)
    p = oracle_mod.problem(w.B, w.Hq, w.Hkv, w.N, w.d, w.causal, smooth_k=False,
                           bf16_mask=(1 << oracle_mod.QZ_Q) | (1 << oracle_mod.QZ_K))
    r = oracle_mod.quantize_qk(p, x["q"], x["k"])
    for name, H in (("q", w.Hq), ("k", w.Hkv)):
        t = x[name].float().reshape(w.B * H, w.N, w.d)
        for blk in range((w.N + 127) // 128):
            xb = t[:, blk * 128:(blk + 1) * 128]
            a = xb.abs().amax(dim=(1, 2))  # FP32 block maxima
            inv = (torch.tensor(127.0) / a).float()  # IEEE FP32 division
            want = (xb * inv[:, None, None]).to(torch.bfloat16).float().numpy()
            np.testing.assert_array_equal(r[name][:, blk * 128:(blk + 1) * 128], want)
            np.testing.assert_array_equal(r["s" + name][:, blk], (a / 127.0).numpy())


def test_all_bf16_is_exact_attention_up_to_bf16(oracle_mod):
    w = W_SMALL
    x = W.make_inputs(w)
    ex = exact_attention(x, w)
    p8 = oracle_mod.problem(w.B, w.Hq, w.Hkv, w.N, w.d, w.causal)
    p16 = oracle_mod.problem(w.B, w.Hq, w.Hkv, w.N, w.d, w.causal, bf16_mask=0x7F)
    q8 = oracle_mod.pipeline(p8, x["q"], x["k"], x["v"], x["do"])
    q16 = oracle_mod.pipeline(p16, x["q"], x["k"], x["v"], x["do"])
    for key in ("o", "dq", "dk", "dv"):
        e16, e8 = rel(q16[key], ex[key]), rel(q8[key], ex[key])
        assert e16 < 1e-2, (key, e16)
        assert e16 < 0.25 * e8, (key, e16, e8)


def test_ds_dominates_in_bf16_attribution(oracle_mod):
    w = W_SMALL
    x = W.make_inputs(w)
    ex = exact_attention(x, w)
    err = {}
    for bit in range(7):
        p = oracle_mod.problem(w.B, w.Hq, w.Hkv, w.N, w.d, w.causal, bf16_mask=1 << bit)
        r = oracle_mod.pipeline(p, x["q"], x["k"], x["v"], x["do"])
        err[bit] = {key: rel(r[key], ex[key]) for key in ("dq", "dk")}
    for key in ("dq", "dk"):
        best = min(err, key=lambda b: err[b][key])
        assert best == oracle_mod.QZ_DS, (key, err)
