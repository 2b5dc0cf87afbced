"""The oracle's Q-smoothing quantities, checked against their definitions (CPU only).

"SageBwd: A Trainable Low-bit Attention" (Abstract, finding (iv)) names
Q-smoothing; the library's reading subtracts each 128-token block's channel
means from Q and adds mean_Q(block) . K'_k back to the logits.  Here the
oracle's block means must be the plain mean of the block's valid rows
(FP64, rounded once to FP32), and its logit terms c0 * (mean_Q . K') with
K' = K - mean_K (each rounded to FP32), recomputed with numpy.
"""
import numpy as np

from bit_trainable_attention_gb300 import workloads as W


def test_block_means_and_logit_terms(oracle_mod):
    w = W.small("qs_terms", 1, 4, 2, 300, 64, True, 81, k_offset_sd=2.0, q_offset_sd=3.0)
    x = W.make_inputs(w)
    p = oracle_mod.problem(w.B, w.Hq, w.Hkv, w.N, w.d, w.causal, smooth_q=True)
    t = oracle_mod.qsmooth_terms(p, x["q"], x["k"])
    q = x["q"].float().double().numpy().reshape(w.B * w.Hq, w.N, w.d)
    k = x["k"].float().double().numpy().reshape(w.B * w.Hkv, w.N, w.d)
    nb = (w.N + 127) // 128
    qm = np.stack([np.stack([q[bh, b * 128:min(w.N, (b + 1) * 128)].mean(axis=0) for b in range(nb)])
                   for bh in range(w.B * w.Hq)]).astype(np.float32)
    np.testing.assert_array_equal(t["qm"], qm)
    mu = k.mean(axis=1).astype(np.float32).astype(np.float64)
    kp = (k - mu[:, None, :]).astype(np.float32).astype(np.float64)  # K', one FP32 rounding
    c0 = np.float32(1.0 / np.sqrt(w.d) * np.log2(np.e))
    G = w.Hq // w.Hkv
    for bhq in range(w.B * w.Hq):
        ref = np.einsum("bc,nc->bn", t["qm"][bhq].astype(np.float64), kp[bhq // G]) * np.float64(c0)
        np.testing.assert_allclose(t["bias"][bhq], ref, rtol=1e-6, atol=1e-6 * np.abs(ref).max())
