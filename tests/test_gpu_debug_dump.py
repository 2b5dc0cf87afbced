"""Tile-level parity through the debug dump (SAGEBWD_FLAG_DEBUG_DUMP).

With the flag the attention kernels also write, per 128 x 128 tile, the
INT8-semantics operands they produced and the raw FP32 tensor-core products
("SageBwd: A Trainable Low-bit Attention", Abstract: INT8 S = Q K^T, P V,
dV = P^T dO, dK = dS^T Q, dQ = dS K).  Checked here:

* every raw product equals the exact integer product of its operands, the
  dumped codes and the stored Q^, K^, V^, dO^ codes, computed in int64 by
  brute force: the integer-valued BF16 operands with FP32 accumulation are
  exact on the tensor cores (|sum| <= 128 * 127^2 < 2^24).  This holds in the
  plain Q/K mode everywhere and, in the library's default mode (Q/K
  sub-scales), on every tile whose Q^ and K^ values are integers (all of them
  on inputs without channel outliers).  Where a sub-scale k > 0 makes a value
  code * 2^-k, the products that read Q^ or K^ (S, dK, dQ) are compared with
  the exact rational sum (int64 at 2^-16 or 2^-8 resolution) within the
  worst-case FP32 summation bound, 128 * 2^-23 * sum |a_k b_k|;
* the P~, P^T and dS codes equal the oracle's codes of the same tile except at
  rounding ties, where the GPU's ex2.approx and FP32 operation order may move a
  code by one (at most 0.3 % of a tile's codes, never by more than one);
* the flag leaves O, LSE and the gradients unchanged.
"""
import numpy as np
import pytest
import torch

import bit_trainable_attention_gb300 as sb
from bit_trainable_attention_gb300 import workloads as W
from _parity import device_inputs, gpu_forward, oracle_problem, to_np

pytestmark = pytest.mark.gpu

CASES = [W.small("dump_gqa_causal_300_d64", 1, 4, 2, 300, 64, True, 801, k_offset_sd=2.0, qk_norm=True),
         W.small("dump_nc_257_d128", 1, 2, 1, 257, 128, False, 802, outlier_frac=0.02),
         W.small("dump_mha_causal_200_d128", 2, 2, 2, 200, 128, True, 803, k_offset_sd=2.0)]
MODES = {"default": True, "plain": False}  # qk_subexp
TIE_FRAC = 3e-3
SUB = 256  # 2^8: the largest Q/K sub-scale exponent, so 2^8 * value is an integer


def padded_blocks(x, nb):
    """[BH, N, d] integer codes -> [BH, nb, 128, d] int64 with zero rows past N."""
    BH, N, d = x.shape
    out = np.zeros((BH, nb * 128, d), np.int64)
    out[:, :N] = x
    return out.reshape(BH, nb, 128, d)


def codes(t):
    a = t.float().cpu().numpy()
    assert np.all(a == np.round(a)), "operand values are not integers"
    return a.astype(np.int64)


def scaled(t):
    """Q^ / K^ values (codes, or codes * 2^-k with the sub-scales) times 2^8, as exact int64."""
    a = t.float().cpu().numpy().astype(np.float64) * SUB
    assert np.all(a == np.round(a)), "operand values are not multiples of 2^-8"
    return a.astype(np.int64)


def check_product(gpu, a, b, what):
    """gpu: the dumped FP32 tile product A B, with a = 2^8 A and b = 2^8 B given as exact int64.
    When every operand value is an integer, A B is an integer sum below 2^24, which the tensor
    core's FP32 accumulation holds exactly: compared bit for bit.  Otherwise (a sub-scaled value,
    code * 2^-k) within the worst-case FP32 summation bound.  Returns 1 when compared bit for bit."""
    exact = a @ b  # 2^16 A B, exact
    g = np.asarray(gpu, np.float64) * (SUB * SUB)
    if np.all(a % SUB == 0) and np.all(b % SUB == 0):
        np.testing.assert_array_equal(g, exact.astype(np.float64), err_msg=what)
        return 1
    bound = a.shape[1] * 2.0 ** -23 * (np.abs(a) @ np.abs(b)).astype(np.float64)
    err = np.abs(g - exact)
    assert np.all(err <= bound), f"{what}: error {float(err.max()):.3g} beyond the FP32 summation bound"
    return 0


def check_codes_against_oracle(gpu, ref, what):
    diff = np.abs(gpu.astype(np.int64) - ref.astype(np.int64))
    assert diff.max() <= 1, f"{what}: a code differs by {diff.max()}"
    frac = float((diff > 0).mean())
    assert frac <= TIE_FRAC, f"{what}: {frac:.2e} of the codes differ (ties allowed up to {TIE_FRAC})"


def run(w, xd, flags, qk_subexp=True):
    fwd = gpu_forward(w, xd, flags=flags, qk_subexp=qk_subexp)
    prob = fwd["prob"]
    dq, dk, dv = torch.empty_like(xd["q"]), torch.empty_like(xd["k"]), torch.empty_like(xd["v"])
    ws1 = sb.empty_bytes(sb.sagebwd_workspace_bytes(prob, 1), "cuda")
    sb.sagebwd_bwd(prob, xd["q"], xd["k"], xd["v"], fwd["o"], xd["do"], fwd["lse"], fwd["saved"], dq, dk, dv, ws1)
    code, _ = sb.sagebwd_check_status(ws1)
    assert fwd["status"] == 0 and code == 0
    return fwd, {"dq": dq, "dk": dk, "dv": dv, "ws": ws1}


@pytest.mark.parametrize("mode", sorted(MODES))
@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_tile_products_are_exact_and_codes_match(oracle_mod, w, mode):
    x, xd = device_inputs(w)
    fwd, bwd = run(w, xd, sb.FLAG_DEBUG_DUMP, qk_subexp=MODES[mode])
    prob = fwd["prob"]
    nb, G, d = (w.N + 127) // 128, w.Hq // w.Hkv, w.d
    views = sb.quantized_views(prob, fwd["saved"])
    qc = padded_blocks(scaled(views["q"]).reshape(w.B * w.Hq, w.N, d), nb)  # 2^8 * Q^
    kc = padded_blocks(scaled(views["k"]).reshape(w.B * w.Hkv, w.N, d), nb)  # 2^8 * K^
    vc = padded_blocks(codes(views["v"]).reshape(w.B * w.Hkv, w.N, d), nb)
    # dO^ codes: the single-operand quantizer (the backward's own quantizer of dO, bit-exact
    # against the oracle in the quantizer tests)
    doq = torch.empty_like(xd["do"])
    sdo = torch.empty(w.B * w.Hq * nb, dtype=torch.float32, device="cuda")
    ws0 = sb.empty_bytes(sb.sagebwd_workspace_bytes(prob, 0), "cuda")
    sb.sagebwd_quantize(prob, sb.SAGEBWD_DO, xd["do"], doq, sdo, None, ws0)
    torch.cuda.synchronize()
    dc = padded_blocks(codes(doq).reshape(w.B * w.Hq, w.N, d), nb)
    fd = {k: v.cpu() for k, v in sb.debug_dump_views(prob, fwd["ws"], 0).items()}
    bd = {k: v.cpu() for k, v in sb.debug_dump_views(prob, bwd["ws"], 1).items()}
    op = oracle_problem(oracle_mod, w, qk_subexp=MODES[mode])
    o_in, lse_in = to_np(fwd["o"]), to_np(fwd["lse"]).astype(np.float64)
    checked = exact_tiles = 0
    for bhq in range(w.B * w.Hq):
        b, h = divmod(bhq, w.Hq)
        bhk = b * w.Hkv + h // G
        for ib in range(nb):
            for jb in range(nb):
                if w.causal and jb > ib:
                    continue
                # forward: S = Q^ K^T (exact, or within the FP32 bound), [P^ V^] = P~ codes V^ exactly
                exact_tiles += check_product(fd["s"][bhq, ib, jb].double().numpy(), qc[bhq, ib], kc[bhk, jb].T,
                                             f"S tile {bhq},{ib},{jb}")
                pc = codes(fd["p"][bhq, ib, jb])
                np.testing.assert_array_equal(fd["pv"][bhq, ib, jb].double().numpy(),
                                              (pc @ vc[bhk, jb]).astype(np.float64))
                rows = min(128, w.N - ib * 128)
                ref_p, _ = oracle_mod.fwd_tile(op, x["q"], x["k"], b, h, ib, jb)
                check_codes_against_oracle(pc[:rows], ref_p[:rows], f"P~ codes tile {bhq},{ib},{jb}")
                # backward: [P^T dO^], [dS^T Q^], [dS K^] exactly from the dumped codes
                pt, ds = codes(bd["pt"][bhq, ib, jb]), codes(bd["ds"][bhq, ib, jb])  # [key][query]
                np.testing.assert_array_equal(bd["dv"][bhq, ib, jb].double().numpy(),
                                              (pt @ dc[bhq, ib]).astype(np.float64))
                check_product(bd["dk"][bhq, ib, jb].double().numpy(), SUB * ds, qc[bhq, ib], f"dK tile {bhq},{ib},{jb}")
                check_product(bd["dq"][bhq, ib, jb].double().numpy(), SUB * ds.T, kc[bhk, jb],
                              f"dQ tile {bhq},{ib},{jb}")
                keys = min(128, w.N - jb * 128)
                ref_pt, _, ref_ds, _ = oracle_mod.bwd_tile(op, x["q"], x["k"], x["v"], o_in, x["do"], lse_in, b, h,
                                                           ib, jb)
                check_codes_against_oracle(pt[:keys, :rows], ref_pt[:keys, :rows], f"P^T codes {bhq},{ib},{jb}")
                check_codes_against_oracle(ds[:keys, :rows], ref_ds.T[:keys, :rows], f"dS codes {bhq},{ib},{jb}")
                checked += 1
    assert checked >= 6
    if mode == "plain" or w.outlier_frac == 0:
        assert exact_tiles == checked  # integer operands: every S tile bit-exact


def test_dump_leaves_outputs_unchanged():
    w = CASES[0]
    _, xd = device_inputs(w)
    f0, b0 = run(w, xd, 0)
    f1, b1 = run(w, xd, sb.FLAG_DEBUG_DUMP)
    for key in ("o", "lse"):
        assert torch.equal(f0[key], f1[key]), key
    for key in ("dq", "dk", "dv"):
        # the FP32 reductions into dQ (and dK, dV across CTAs) add in run-dependent order
        a, c = b0[key].float(), b1[key].float()
        assert float((a - c).abs().max()) <= 1e-2 * float(a.abs().max()), key
