"""Helpers shared by the GPU parity tests: run the library through its C ABI
(the ctypes binding) and compare against the oracle.

Tolerances (derived in tests/test_tolerance_calibration.py):
* quantized operands (codes, scales, K mean, dO codes): bit-exact;
* O, dQ, dK, dV (BF16): against the oracle's result rounded to BF16,
  relative Frobenius error ||gpu - ref|| / ||ref|| <= 2e-3, and every element
  within 1e-2 * max|ref| plus one BF16 ulp.  A code computed in FP32 by two
  different operation orders can differ by one at a rounding tie; one flipped
  dS code moves a whole dQ/dK row by one dS quantum (the dS scale is shared by
  a 128 x 128 tile), so a single element can move by several 1e-3 of the
  tensor's maximum while the tensor as a whole stays within 1e-3;
* LSE: absolute 1e-4 (FP32 statistics of unquantized probabilities).
"""
import numpy as np
import torch

import bit_trainable_attention_gb300 as sb
from bit_trainable_attention_gb300 import workloads as W

REL_L2_TOL = 2e-3
ELEM_TOL = 1e-2
LSE_TOL = 1e-4


def bf16_ulp(x):
    a = np.abs(np.asarray(x, np.float64))
    e = np.floor(np.log2(np.maximum(a, 1e-30)))
    return np.exp2(e - 7)


def normwise_error(gpu, ref):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    m = np.isfinite(ref)
    return float(np.max(np.abs(gpu[m] - ref[m])) / np.max(np.abs(ref[m])))


def bf16_round(x):
    f = np.asarray(x, np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return r.astype(np.uint32).view(np.float32).astype(np.float64)


# Every assert_parity call records (test, tensor, relative L2, max element error / max|ref|) here;
# tests/conftest.py prints the table at the end of the run, so the distance of each config from
# the 2e-3 target is visible in the log.
REPORT = []


def _current_test():
    import os
    return os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]


def assert_parity(gpu, ref, name, rel_l2_tol=REL_L2_TOL, elem_tol=ELEM_TOL):
    """gpu: the library's BF16 output; ref: the oracle's FP64 result (NaN = not computed).

    Returns {"rel_l2": ||gpu - ref|| / ||ref||, "max_elem": max|gpu - ref| / max|ref|} (ref rounded
    to BF16), after checking both bounds."""
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    m = np.isfinite(ref)
    assert m.any(), name
    g, r = gpu[m], bf16_round(ref[m])
    assert np.all(np.isfinite(g)), f"{name}: non-finite GPU values"
    if not np.any(r):
        # e.g. one token: P = 1 and dS = dP - D = 0 exactly, so dQ = dK = 0; the
        # library's FP32 dP - D leaves at most rounding-level residue
        assert np.abs(g).max() <= 1e-4, f"{name}: reference is zero, GPU max {np.abs(g).max():.3e}"
        out = {"rel_l2": 0.0, "max_elem": 0.0}
        REPORT.append((_current_test(), name, out["rel_l2"], out["max_elem"]))
        return out
    rel_l2 = float(np.linalg.norm(g - r) / np.linalg.norm(r))
    scale = np.max(np.abs(r))
    err = np.abs(g - r)
    out = {"rel_l2": rel_l2, "max_elem": float(err.max() / scale)}
    REPORT.append((_current_test(), name, out["rel_l2"], out["max_elem"]))
    assert rel_l2 <= rel_l2_tol, f"{name}: relative L2 error {rel_l2:.3e} > {rel_l2_tol}"
    bad = err > elem_tol * scale + bf16_ulp(r)
    assert not bad.any(), (f"{name}: {int(bad.sum())} of {bad.size} elements beyond {elem_tol} of the max; "
                           f"worst at ref={r[bad][0]:.6g} gpu={g[bad][0]:.6g}")
    return out


def cos(a, b):
    a = np.nan_to_num(np.asarray(a, np.float64)).ravel()
    b = np.nan_to_num(np.asarray(b, np.float64)).ravel()
    return float(a @ b / np.linalg.norm(a) / np.linalg.norm(b))


def to_np(t):
    return t.detach().float().cpu().double().numpy() if t.dtype == torch.bfloat16 else t.detach().cpu().numpy()


def device_inputs(w, dev="cuda"):
    x = W.make_inputs(w)
    return x, {k: v.to(dev) for k, v in x.items()}


def gpu_forward(w, xd, smooth_k=True, flags=0, timeout_ms=0, balance_qk=False, ds_subexp=False, qk_subexp=None,
                smooth_q=False, fp8=False):
    prob = sb.Problem.make(w.B, w.Hq, w.Hkv, w.N, w.d, w.causal, smooth_k=smooth_k, flags=flags,
                           wait_timeout_ms=timeout_ms, balance_qk=balance_qk, ds_subexp=ds_subexp,
                           qk_subexp=qk_subexp, smooth_q=smooth_q, fp8=fp8)
    dev = xd["q"].device
    o = torch.empty_like(xd["q"])
    lse = torch.empty(w.B, w.Hq, w.N, dtype=torch.float32, device=dev)
    saved = sb.empty_bytes(sb.sagebwd_saved_bytes(prob), dev)
    ws = sb.empty_bytes(sb.sagebwd_workspace_bytes(prob, 0), dev)
    sb.sagebwd_fwd(prob, xd["q"], xd["k"], xd["v"], o, lse, saved, ws)
    code, word = sb.sagebwd_check_status(ws)
    return {"prob": prob, "o": o, "lse": lse, "saved": saved, "ws": ws, "status": code, "word": word}


def gpu_backward(w, xd, fwd):
    prob = fwd["prob"]
    dev = xd["q"].device
    dq = torch.empty_like(xd["q"])
    dk = torch.empty_like(xd["k"])
    dv = torch.empty_like(xd["v"])
    ws = sb.empty_bytes(sb.sagebwd_workspace_bytes(prob, 1), dev)
    sb.sagebwd_bwd(prob, xd["q"], xd["k"], xd["v"], fwd["o"], xd["do"], fwd["lse"], fwd["saved"], dq, dk, dv, ws)
    code, word = sb.sagebwd_check_status(ws)
    return {"dq": dq, "dk": dk, "dv": dv, "ws": ws, "status": code, "word": word}


def oracle_problem(oracle_mod, w, smooth_k=True, balance_qk=False, ds_subexp=False, qk_subexp=None, smooth_q=False,
                   fp8=False):
    """The oracle problem matching gpu_forward's defaults (the library's: K-smoothing and, for INT8,
    the Q/K sub-scales on)."""
    if qk_subexp is None:
        qk_subexp = not fp8
    return oracle_mod.problem(w.B, w.Hq, w.Hkv, w.N, w.d, w.causal, smooth_k=smooth_k, balance_qk=balance_qk,
                              ds_subexp=ds_subexp, qk_subexp=qk_subexp, smooth_q=smooth_q, fp8=fp8)


def block_selection(w, heads, blocks, kv=False):
    """Flags [B*H*nb] selecting (b, h, block) triples; heads/blocks index lists (negative blocks from the end)."""
    nb = (w.N + 127) // 128
    H = w.Hkv if kv else w.Hq
    sel = np.zeros((w.B, H, nb), np.uint8)
    for b in range(w.B):
        for h in heads:
            for blk in blocks:
                sel[b, h % H, blk % nb] = 1
    return sel.reshape(-1)
