"""SageBwd CPU oracle -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never calls it and shares no code with it.

This module builds ``sagebwd_oracle.cpp`` with g++ (OpenMP, no FP contraction)
on first use and wraps its C functions with numpy arrays.  See the header of
the C++ file for what is computed and which passages it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sagebwd_oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

BLK = 128


class OracleProblem(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int32), ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32),
        ("N", ctypes.c_int32), ("d", ctypes.c_int32), ("causal", ctypes.c_int32),
        ("smooth_k", ctypes.c_int32), ("balance_qk", ctypes.c_int32), ("exact_codes", ctypes.c_int32),
        ("threads", ctypes.c_int32), ("exact_mask", ctypes.c_uint32), ("int8_dp", ctypes.c_int32),
        ("ds_subexp", ctypes.c_int32), ("qk_subexp", ctypes.c_int32), ("fp8", ctypes.c_int32),
        ("smooth_q", ctypes.c_int32), ("l_from_codes", ctypes.c_int32), ("bf16_mask", ctypes.c_uint32),
        ("softmax_scale", ctypes.c_double),
    ]


def build(force: bool = False) -> str:
    """Compile the oracle shared library next to its source (idempotent)."""
    with _lock:
        if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
            tmp = _LIB + f".tmp{os.getpid()}"
            cmd = ["g++", "-O2", "-std=c++17", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
                   "-fPIC", "-shared", _SRC, "-o", tmp]
            subprocess.run(cmd, check=True)
            os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.POINTER(OracleProblem)
        vp = ctypes.c_void_p
        lib.oracle_quantize.argtypes = [P, vp, ctypes.c_int, ctypes.c_int, vp, vp, vp]
        lib.oracle_quantize_exact.argtypes = [P, vp, ctypes.c_int, ctypes.c_int, vp, vp, vp]
        for name in ("oracle_fwd", "oracle_exact_fwd"):
            getattr(lib, name).argtypes = [P, vp, vp, vp, vp, vp, vp]
        for name in ("oracle_bwd", "oracle_exact_bwd"):
            getattr(lib, name).argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        lib.oracle_quantize_qk.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp]
        lib.oracle_fwd_tile.argtypes = [P, vp, vp] + [ctypes.c_int] * 4 + [vp, vp]
        lib.oracle_bwd_tile.argtypes = [P, vp, vp, vp, vp, vp, vp] + [ctypes.c_int] * 4 + [vp, vp, vp, vp]
        lib.oracle_max_threads.restype = ctypes.c_int
        lib.oracle_round_e4m3.argtypes = [vp, vp, ctypes.c_int64]
        lib.oracle_qsmooth_terms.argtypes = [P, vp, vp, vp, vp]
        _lib = lib
    return _lib


def round_e4m3(x) -> np.ndarray:
    """FP8 E4M3 rounding (nearest, ties to even, saturating at 448) of FP64 values."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty_like(x)
    assert _load().oracle_round_e4m3(_ptr(x), _ptr(y), x.size) == 0
    return y


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _bf16_bits(x) -> np.ndarray:
    """Accept a uint16 array of BF16 bit patterns, or a torch bfloat16 tensor."""
    if isinstance(x, np.ndarray):
        assert x.dtype == np.uint16
        return np.ascontiguousarray(x)
    import torch  # only for converting test tensors
    assert x.dtype == torch.bfloat16
    return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


# Quantizer bits of exact_mask and bf16_mask.
QZ_Q, QZ_K, QZ_V, QZ_DO, QZ_PF, QZ_PB, QZ_DS = range(7)


def problem(B, Hq, Hkv, N, d, causal, smooth_k=True, exact_codes=False, softmax_scale=0.0, threads=0, exact_mask=0,
            balance_qk=False, int8_dp=False, ds_subexp=False, qk_subexp=False, fp8=False, smooth_q=False,
            l_from_codes=False, bf16_mask=0):
    """l_from_codes plants a misreading (softmax denominator from the dequantized P~ codes); only the
    tests that show a pin catches it set it.  exact_mask / bf16_mask (bits QZ_*): those quantizers keep
    their scales but skip the rounding (FP64) / round to BF16 instead of to an INT8 code."""
    return OracleProblem(B, Hq, Hkv, N, d, int(causal), int(smooth_k), int(balance_qk), int(exact_codes),
                         int(threads), int(exact_mask), int(int8_dp), int(ds_subexp), int(qk_subexp), int(fp8),
                         int(smooth_q), int(l_from_codes), int(bf16_mask), float(softmax_scale))


def nblocks(N: int) -> int:
    return (N + BLK - 1) // BLK


def quantize(p: OracleProblem, x, BH: int, smooth: bool):
    """Per-128-token-block absmax INT8 codes, FP32 scales and (smooth) FP32 channel means."""
    x = _bf16_bits(x)
    assert x.size == BH * p.N * p.d
    codes = np.zeros(x.size, np.int8)
    scales = np.zeros(BH * nblocks(p.N), np.float32)
    mean = np.zeros(BH * p.d, np.float32) if smooth else None
    rc = _load().oracle_quantize(ctypes.byref(p), _ptr(x), BH, int(smooth), _ptr(codes), _ptr(scales), _ptr(mean))
    assert rc == 0
    return codes.reshape(BH, p.N, p.d), scales.reshape(BH, -1), (mean.reshape(BH, p.d) if smooth else None)


def quantize_exact(p: OracleProblem, x, BH: int, smooth: bool):
    """The same quantizer without rounding (codes = x / s in FP64)."""
    x = _bf16_bits(x)
    codes = np.zeros(x.size, np.float64)
    scales = np.zeros(BH * nblocks(p.N), np.float64)
    mean = np.zeros(BH * p.d, np.float64) if smooth else None
    rc = _load().oracle_quantize_exact(ctypes.byref(p), _ptr(x), BH, int(smooth), _ptr(codes), _ptr(scales),
                                       _ptr(mean))
    assert rc == 0
    return codes.reshape(BH, p.N, p.d), scales.reshape(BH, -1), (mean.reshape(BH, p.d) if smooth else None)


def quantize_qk(p: OracleProblem, q, k):
    """Q and K as the forward quantizes them (K-smoothing and channel balancing as p selects).

    Returns dict: q / k operand values as float32 [B*H, N, d] (integer codes; code * 2^-k with qk_subexp), sq / sk FP32 block scales [B*H, nb], mu FP32 K channel
    means [B*Hkv, d] (zeros without smoothing), e int32 balancing exponents [B*Hkv, d] (zeros unless
    balance_qk)."""
    q, k = _bf16_bits(q), _bf16_bits(k)
    BHq, BHk, nb = p.B * p.Hq, p.B * p.Hkv, nblocks(p.N)
    out = {"q": np.zeros((BHq, p.N, p.d), np.float32), "sq": np.zeros((BHq, nb), np.float32),
           "k": np.zeros((BHk, p.N, p.d), np.float32), "sk": np.zeros((BHk, nb), np.float32),
           "mu": np.zeros((BHk, p.d), np.float32), "e": np.zeros((BHk, p.d), np.int32)}
    rc = _load().oracle_quantize_qk(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(out["q"]), _ptr(out["sq"]),
                                    _ptr(out["k"]), _ptr(out["sk"]), _ptr(out["mu"]), _ptr(out["e"]))
    assert rc == 0
    return out


def qsmooth_terms(p: OracleProblem, q, k):
    """Q-smoothing's FP32 block means of Q [B*Hq, nb, d] and base-2 logit terms
    c0 * (mean_Q(block) . K'_key) [B*Hq, nb, N] (p.smooth_q must be set)."""
    q, k = _bf16_bits(q), _bf16_bits(k)
    BHq, nb = p.B * p.Hq, nblocks(p.N)
    qm = np.zeros((BHq, nb, p.d), np.float32)
    bias = np.zeros((BHq, nb, p.N), np.float32)
    assert _load().oracle_qsmooth_terms(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(qm), _ptr(bias)) == 0
    return {"qm": qm, "bias": bias}


def _sel(sel, n):
    if sel is None:
        return None
    s = np.ascontiguousarray(np.asarray(sel, dtype=np.uint8).reshape(-1))
    assert s.size == n
    return s


def fwd(p: OracleProblem, q, k, v, qsel=None, exact=False):
    """Quantized forward (exact=False) or exact FP64 attention (exact=True).

    Returns O (FP64, [B,Hq,N,d]) and LSE (FP64, [B,Hq,N], natural log).
    Rows of unselected query blocks are NaN."""
    q, k, v = _bf16_bits(q), _bf16_bits(k), _bf16_bits(v)
    o = np.full((p.B, p.Hq, p.N, p.d), np.nan)
    lse = np.full((p.B, p.Hq, p.N), np.nan)
    s = _sel(qsel, p.B * p.Hq * nblocks(p.N))
    fn = _load().oracle_exact_fwd if exact else _load().oracle_fwd
    rc = fn(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(s))
    assert rc == 0
    return o, lse


def bwd(p: OracleProblem, q, k, v, o, dO, lse, qsel=None, ksel=None, exact=False):
    """Quantized (exact=False) or exact FP64 backward.

    o, lse: the forward's outputs as FP64 arrays.  Returns dQ, dK, dV (FP64);
    unselected blocks are NaN."""
    q, k, v, dO = _bf16_bits(q), _bf16_bits(k), _bf16_bits(v), _bf16_bits(dO)
    o = np.ascontiguousarray(o, dtype=np.float64)
    lse = np.ascontiguousarray(lse, dtype=np.float64)
    dq = np.full((p.B, p.Hq, p.N, p.d), np.nan)
    dk = np.full((p.B, p.Hkv, p.N, p.d), np.nan)
    dv = np.full((p.B, p.Hkv, p.N, p.d), np.nan)
    nb = nblocks(p.N)
    qs, ks = _sel(qsel, p.B * p.Hq * nb), _sel(ksel, p.B * p.Hkv * nb)
    fn = _load().oracle_exact_bwd if exact else _load().oracle_bwd
    rc = fn(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO), _ptr(lse), _ptr(dq), _ptr(dk),
            _ptr(dv), _ptr(qs), _ptr(ks))
    assert rc == 0
    return dq, dk, dv


def rows_needed_for_bwd(p: OracleProblem, qsel=None, ksel=None) -> np.ndarray:
    """Query-block flags [B*Hq*nb] whose forward O/LSE the backward of the selection reads."""
    nb = nblocks(p.N)
    G = p.Hq // p.Hkv
    need = np.zeros((p.B, p.Hq, nb), np.uint8)
    if qsel is None and ksel is None:
        need[:] = 1
        return need.reshape(-1)
    if qsel is not None:
        need |= np.asarray(qsel, np.uint8).reshape(p.B, p.Hq, nb)
    if ksel is not None:
        ks = np.asarray(ksel, np.uint8).reshape(p.B, p.Hkv, nb)
        for b in range(p.B):
            for hk in range(p.Hkv):
                for jb in np.nonzero(ks[b, hk])[0]:
                    lo = jb if p.causal else 0
                    need[b, hk * G:(hk + 1) * G, lo:] = 1
    return need.reshape(-1)


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round FP64 values to BF16 (round to nearest even) and return them as FP64."""
    f = np.asarray(x, np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16) << 16
    nan = np.isnan(f)
    out = r.astype(np.uint32).view(np.float32).astype(np.float64)
    out[nan] = np.nan
    return out


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """FP64 -> BF16 bit patterns (uint16), round to nearest even."""
    return (bf16_round(x).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def pipeline(p: OracleProblem, q, k, v, dO, qsel=None, ksel=None, exact=False):
    """Forward then backward the way the library is called: the backward gets
    the forward's O rounded to BF16 (as the library's BF16 output) and its LSE.

    Returns dict with o, lse, dq, dk, dv (FP64)."""
    need = rows_needed_for_bwd(p, qsel, ksel)
    fsel = need if (qsel is not None or ksel is not None) else None
    o, lse = fwd(p, q, k, v, qsel=fsel, exact=exact)
    o_in = o if (exact or p.exact_codes) else bf16_round(o)
    o_in = np.nan_to_num(o_in, nan=0.0)
    lse_in = np.nan_to_num(lse, nan=0.0)
    dq, dk, dv = bwd(p, q, k, v, o_in, dO, lse_in, qsel=qsel, ksel=ksel, exact=exact)
    return {"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv}


def fwd_tile(p: OracleProblem, q, k, b: int, h: int, ib: int, jb: int):
    """Codes of P~ for one forward tile ([128,128], query x key) and the row maxima (base-2 logits)."""
    q, k = _bf16_bits(q), _bf16_bits(k)
    codes = np.zeros((BLK, BLK), np.int32)
    tmax = np.zeros(BLK, np.float64)
    rc = _load().oracle_fwd_tile(ctypes.byref(p), _ptr(q), _ptr(k), b, h, ib, jb, _ptr(codes), _ptr(tmax))
    assert rc == 0
    return codes, tmax


def bwd_tile(p: OracleProblem, q, k, v, o, dO, lse, b: int, h: int, ib: int, jb: int):
    """P^T codes [key, query], their per-key scales, dS codes [query, key] and the dS scale of one tile."""
    q, k, v, dO = _bf16_bits(q), _bf16_bits(k), _bf16_bits(v), _bf16_bits(dO)
    o = np.ascontiguousarray(o, dtype=np.float64)
    lse = np.ascontiguousarray(lse, dtype=np.float64)
    pt = np.zeros((BLK, BLK), np.int32)
    spc = np.zeros(BLK, np.float64)
    ds = np.zeros((BLK, BLK), np.float64)  # integer codes; with ds_subexp code * 2^-k
    sds = np.zeros(1, np.float64)
    rc = _load().oracle_bwd_tile(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO), _ptr(lse), b, h, ib,
                                 jb, _ptr(pt), _ptr(spc), _ptr(ds), _ptr(sds))
    assert rc == 0
    return pt, spc, ds, float(sds[0])
