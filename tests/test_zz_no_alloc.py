"""sagebwd_quantize_k_noalloc: K quantization for callers that cannot allocate
device memory (its K-mean scratch is a fixed array inside the library).

Checked through the C ABI against sagebwd_quantize(SAGEBWD_K, ...), which
keeps the same scratch in a caller-provided workspace: two calls in a row
must both give exactly the codes, scales and channel means of the workspace
version (the quantized operands are compared bit-exactly everywhere in these
tests).  Kept in a file of its own that is collected last.
"""
import ctypes

import pytest
import torch

import bit_trainable_attention_gb300 as sb
from bit_trainable_attention_gb300 import workloads as W

pytestmark = pytest.mark.gpu

CASES = [
    W.small("k_d64_ragged", 2, 6, 3, 300, 64, True, 301, k_offset_sd=2.0),
    W.small("k_d128", 1, 4, 2, 1024, 128, True, 302, outlier_frac=0.01),
    W.WORKLOADS["videodit"],
]


def _workspace_version(prob, k):
    BH = prob.B * prob.Hkv
    nb = (prob.N + 127) // 128
    kq = torch.empty_like(k)
    sc = torch.empty(BH, nb, dtype=torch.float32, device=k.device)
    mu = torch.empty(BH, prob.d, dtype=torch.float32, device=k.device)
    ws = sb.empty_bytes(sb.sagebwd_workspace_bytes(prob, 0), k.device)
    sb.sagebwd_quantize(prob, sb.SAGEBWD_K, k, kq, sc, mu, ws)
    return kq, sc, mu


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_noalloc_matches_workspace_version_twice(w):
    k = W.make_inputs(w)["k"].cuda()
    prob = sb.Problem.make(w.B, w.Hq, w.Hkv, w.N, w.d, w.causal)
    ref = _workspace_version(prob, k)
    for _ in range(2):
        kq = torch.full_like(k, 99.0)
        sc = torch.full_like(ref[1], -1.0)
        mu = torch.full_like(ref[2], -1.0)
        sb.sagebwd_quantize_k_noalloc(prob, k, kq, sc, mu)
        torch.cuda.synchronize()
        assert torch.equal(kq, ref[0])
        assert torch.equal(sc.view(torch.int32), ref[1].view(torch.int32))
        assert torch.equal(mu.view(torch.int32), ref[2].view(torch.int32))


def test_noalloc_rejects_problems_beyond_its_scratch():
    lib = sb.load_library()
    # B * Hkv * ceil(N/128) * d = 4 * 32 * 64 * 128 = 2^20 * 1.0 fits; one more block does not
    fits = sb.Problem.make(4, 32, 32, 64 * 128, 128, True)
    over = sb.Problem.make(4, 32, 32, 64 * 128 + 1, 128, True)
    dummy = ctypes.c_void_p(1 << 20)  # never dereferenced: the size check fails first
    assert lib.sagebwd_quantize_k_noalloc(ctypes.byref(over), dummy, dummy, dummy, dummy, None) == 6
    assert sb.STATUS_NAMES[6] == "SCRATCH_LIMIT"
    k = torch.zeros(fits.B, fits.Hkv, fits.N, fits.d, dtype=torch.bfloat16, device="cuda")
    kq = torch.empty_like(k)
    sc = torch.empty(fits.B * fits.Hkv, 64, dtype=torch.float32, device="cuda")
    mu = torch.empty(fits.B * fits.Hkv, fits.d, dtype=torch.float32, device="cuda")
    sb.sagebwd_quantize_k_noalloc(fits, k, kq, sc, mu)
    torch.cuda.synchronize()
    assert not kq.any() and not sc.any() and not mu.any()
