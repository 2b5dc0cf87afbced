"""SageBwd trainable INT8 attention for GB300 (sm_103a).

Python binding of the C ABI declared in ``include/sagebwd.h``: every function
named ``sagebwd_*`` here marshals torch tensors (device memory and the current
stream) into the C call of the same name; all computation happens in the
library's CUDA kernels.  ``SageBwdAttention`` / ``attention`` wrap the forward
and backward calls as a ``torch.autograd.Function``.

There is no fallback: if ``libsagebwd.so`` cannot be built or loaded, every
call raises.
"""
from __future__ import annotations

import ctypes
import threading

import torch

from . import _build

__all__ = [
    "Problem", "SageBwdError", "load_library", "sagebwd_saved_bytes", "sagebwd_workspace_bytes",
    "sagebwd_quantize", "sagebwd_fwd", "sagebwd_bwd", "sagebwd_fwd_quantize", "sagebwd_fwd_attention",
    "sagebwd_bwd_prepare", "sagebwd_bwd_attention", "sagebwd_bwd_finish", "sagebwd_check_status",
    "sagebwd_status_string", "sagebwd_version", "sagebwd_quantize_k_noalloc", "attention", "SageBwdAttention",
    "SAGEBWD_Q", "SAGEBWD_K", "SAGEBWD_V", "SAGEBWD_DO", "FLAG_DROP_ONE_LOAD", "FLAG_DEBUG_DUMP", "FLAG_BF16",
    "sagebwd_debug_dump_offset", "debug_dump_views", "check_errors",
]

SAGEBWD_Q, SAGEBWD_K, SAGEBWD_V, SAGEBWD_DO = 0, 1, 2, 3
FLAG_DROP_ONE_LOAD = 0x1
FLAG_DEBUG_DUMP = 0x2
# error attribution: one quantizer stores BF16 of its scaled values instead of INT8 codes
FLAG_BF16 = {"q": 0x10, "k": 0x20, "v": 0x40, "do": 0x80, "p_fwd": 0x100, "p_bwd": 0x200, "ds": 0x400}
STATUS_NAMES = {0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED", 3: "MISALIGNED", 4: "CUDA", 5: "TIMEOUT",
                6: "SCRATCH_LIMIT"}

EXPORTED_SYMBOLS = (
    "sagebwd_saved_bytes", "sagebwd_workspace_bytes", "sagebwd_quantize", "sagebwd_fwd", "sagebwd_bwd",
    "sagebwd_fwd_quantize", "sagebwd_fwd_attention", "sagebwd_bwd_prepare", "sagebwd_bwd_attention",
    "sagebwd_bwd_finish", "sagebwd_check_status", "sagebwd_status_string", "sagebwd_version",
    "sagebwd_quantize_k_noalloc", "sagebwd_debug_dump_offset",
)


class SageBwdError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS_NAMES.get(code, code)} ({_status_text(code)})")


class Problem(ctypes.Structure):
    """Mirror of ``sagebwd_problem``."""
    _fields_ = [
        ("B", ctypes.c_int32), ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32), ("N", ctypes.c_int32),
        ("d", ctypes.c_int32), ("causal", ctypes.c_int32), ("smooth_k", ctypes.c_int32),
        ("balance_qk", ctypes.c_int32), ("ds_subexp", ctypes.c_int32),
        ("qk_subexp", ctypes.c_int32), ("smooth_q", ctypes.c_int32), ("flags", ctypes.c_uint32),
        ("softmax_scale", ctypes.c_float), ("wait_timeout_ms", ctypes.c_uint32), ("fp8", ctypes.c_int32),
    ]

    @classmethod
    def make(cls, B, Hq, Hkv, N, d, causal, smooth_k=True, flags=0, softmax_scale=0.0, wait_timeout_ms=0,
             balance_qk=False, ds_subexp=False, qk_subexp=None, smooth_q=False, fp8=False):
        """The library's defaults: K-smoothing on and, for INT8, the Q/K 8-channel sub-scales on
        (qk_subexp=False selects the plain one-scale-per-block mode for Q and K).  fp8=True selects
        the FP8 E4M3 variant, which has no sub-scales."""
        if qk_subexp is None:
            qk_subexp = not fp8
        return cls(B, Hq, Hkv, N, d, int(bool(causal)), int(bool(smooth_k)), int(bool(balance_qk)),
                   int(bool(ds_subexp)), int(bool(qk_subexp)), int(bool(smooth_q)), flags, softmax_scale,
                   wait_timeout_ms, int(bool(fp8)))

    @classmethod
    def from_tensors(cls, q, k, causal, **kw):
        B, Hq, N, d = q.shape
        return cls.make(B, Hq, k.shape[1], N, d, causal, **kw)


_lock = threading.Lock()
_lib = None


def load_library():
    """Build (if needed) and load libsagebwd.so; raises if that is impossible."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            path = _build.build()
            lib = ctypes.CDLL(path)
            P = ctypes.POINTER(Problem)
            vp, st = ctypes.c_void_p, ctypes.c_int
            lib.sagebwd_saved_bytes.argtypes = [P]
            lib.sagebwd_saved_bytes.restype = ctypes.c_size_t
            lib.sagebwd_workspace_bytes.argtypes = [P, ctypes.c_int]
            lib.sagebwd_workspace_bytes.restype = ctypes.c_size_t
            lib.sagebwd_quantize.argtypes = [P, ctypes.c_int, vp, vp, vp, vp, vp, vp]
            lib.sagebwd_fwd.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp]
            lib.sagebwd_bwd.argtypes = [P] + [vp] * 12
            lib.sagebwd_fwd_quantize.argtypes = [P, vp, vp, vp, vp, vp, vp]
            lib.sagebwd_fwd_attention.argtypes = [P, vp, vp, vp, vp, vp]
            lib.sagebwd_bwd_prepare.argtypes = [P, vp, vp, vp, vp]
            lib.sagebwd_bwd_attention.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp]
            lib.sagebwd_bwd_finish.argtypes = [P, vp, vp, vp, vp, vp, vp]
            lib.sagebwd_check_status.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_int32)]
            lib.sagebwd_quantize_k_noalloc.argtypes = [P, vp, vp, vp, vp, vp]
            lib.sagebwd_status_string.argtypes = [ctypes.c_int]
            lib.sagebwd_status_string.restype = ctypes.c_char_p
            lib.sagebwd_version.restype = ctypes.c_int32
            lib.sagebwd_debug_dump_offset.argtypes = [P, ctypes.c_int]
            lib.sagebwd_debug_dump_offset.restype = ctypes.c_size_t
            for name in ("sagebwd_quantize", "sagebwd_fwd", "sagebwd_bwd", "sagebwd_fwd_quantize",
                         "sagebwd_fwd_attention", "sagebwd_bwd_prepare", "sagebwd_bwd_attention",
                         "sagebwd_bwd_finish", "sagebwd_check_status", "sagebwd_quantize_k_noalloc"):
                getattr(lib, name).restype = st
            _lib = lib
    return _lib


def _status_text(code: int) -> str:
    try:
        return load_library().sagebwd_status_string(code).decode()
    except Exception:  # noqa: BLE001 - only used to decorate an error message
        return "?"


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return ctypes.c_void_p(t)
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _check(code: int, where: str):
    if code != 0:
        raise SageBwdError(code, where)


def sagebwd_saved_bytes(prob: Problem) -> int:
    return int(load_library().sagebwd_saved_bytes(ctypes.byref(prob)))


def sagebwd_workspace_bytes(prob: Problem, pass_: int) -> int:
    return int(load_library().sagebwd_workspace_bytes(ctypes.byref(prob), pass_))


def sagebwd_quantize(prob, which, x, x_q, scales, k_mean, ws, stream=None):
    _check(load_library().sagebwd_quantize(ctypes.byref(prob), which, _ptr(x), _ptr(x_q), _ptr(scales),
                                           _ptr(k_mean), _ptr(ws), _stream(stream)), "sagebwd_quantize")


def sagebwd_fwd(prob, q, k, v, o, lse, saved, ws, stream=None):
    _check(load_library().sagebwd_fwd(ctypes.byref(prob), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                      _ptr(saved), _ptr(ws), _stream(stream)), "sagebwd_fwd")


def sagebwd_bwd(prob, q, k, v, o, dO, lse, saved, dq, dk, dv, ws, stream=None):
    _check(load_library().sagebwd_bwd(ctypes.byref(prob), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO), _ptr(lse),
                                      _ptr(saved), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws), _stream(stream)),
           "sagebwd_bwd")


def sagebwd_fwd_quantize(prob, q, k, v, saved, ws, stream=None):
    _check(load_library().sagebwd_fwd_quantize(ctypes.byref(prob), _ptr(q), _ptr(k), _ptr(v), _ptr(saved), _ptr(ws),
                                               _stream(stream)), "sagebwd_fwd_quantize")


def sagebwd_fwd_attention(prob, saved, o, lse, ws, stream=None):
    _check(load_library().sagebwd_fwd_attention(ctypes.byref(prob), _ptr(saved), _ptr(o), _ptr(lse), _ptr(ws),
                                                _stream(stream)), "sagebwd_fwd_attention")


def sagebwd_bwd_prepare(prob, o, dO, ws, stream=None):
    _check(load_library().sagebwd_bwd_prepare(ctypes.byref(prob), _ptr(o), _ptr(dO), _ptr(ws), _stream(stream)),
           "sagebwd_bwd_prepare")


def sagebwd_bwd_attention(prob, v, dO, lse, saved, dk, dv, ws, stream=None):
    _check(load_library().sagebwd_bwd_attention(ctypes.byref(prob), _ptr(v), _ptr(dO), _ptr(lse), _ptr(saved),
                                                _ptr(dk), _ptr(dv), _ptr(ws), _stream(stream)),
           "sagebwd_bwd_attention")


def sagebwd_bwd_finish(prob, saved, dq, dk, dv, ws, stream=None):
    _check(load_library().sagebwd_bwd_finish(ctypes.byref(prob), _ptr(saved), _ptr(dq), _ptr(dk), _ptr(dv),
                                             _ptr(ws), _stream(stream)),
           "sagebwd_bwd_finish")


def sagebwd_quantize_k_noalloc(prob, k, k_q, scales, k_mean, stream=None):
    """K quantization without a workspace, for callers that cannot allocate device memory: the
    K-mean scratch is a fixed 8 MiB array inside the library (limit B*Hkv*ceil(N/128)*d <= 2^20).
    Calls that overlap on the GPU share that array and race; the first call on a device should
    come before any stream capture."""
    _check(load_library().sagebwd_quantize_k_noalloc(ctypes.byref(prob), _ptr(k), _ptr(k_q), _ptr(scales),
                                                     _ptr(k_mean), _stream(stream)), "sagebwd_quantize_k_noalloc")


def sagebwd_check_status(ws, stream=None):
    """Synchronize the stream; return (status code, raw status word)."""
    word = ctypes.c_int32(0)
    code = load_library().sagebwd_check_status(_ptr(ws), _stream(stream), ctypes.byref(word))
    return int(code), int(word.value)


def sagebwd_status_string(code: int) -> str:
    return load_library().sagebwd_status_string(code).decode()


def sagebwd_version() -> int:
    return int(load_library().sagebwd_version())


def sagebwd_debug_dump_offset(prob, pass_: int) -> int:
    return int(load_library().sagebwd_debug_dump_offset(ctypes.byref(prob), pass_))


def debug_dump_views(prob: Problem, ws: torch.Tensor, pass_: int) -> dict:
    """Views of the debug dump (SAGEBWD_FLAG_DEBUG_DUMP) inside a workspace, one record per
    tile [B*Hq, nb (query block), nb (key block)].  Forward (pass 0): s [.., 128 q, 128 k] FP32,
    p [.., 128 q, 128 k] BF16 codes, pv [.., 128 q, d] FP32.  Backward (pass 1): pt and ds
    [.., 128 keys, 128 queries] BF16 codes, dv and dk [.., 128 keys, d], dq [.., 128 queries, d] FP32."""
    off = sagebwd_debug_dump_offset(prob, pass_)
    if off == 0:
        raise ValueError("the problem has no debug dump (SAGEBWD_FLAG_DEBUG_DUMP not set)")
    nb = (prob.N + 127) // 128
    d = prob.d
    n = prob.B * prob.Hq * nb * nb
    if pass_ == 0:
        parts = [("s", 128 * 128 * 4, torch.float32, (128, 128)), ("p", 128 * 128 * 2, torch.bfloat16, (128, 128)),
                 ("pv", 128 * d * 4, torch.float32, (128, d))]
    else:
        parts = [("pt", 128 * 128 * 2, torch.bfloat16, (128, 128)), ("ds", 128 * 128 * 2, torch.bfloat16, (128, 128)),
                 ("dv", 128 * d * 4, torch.float32, (128, d)), ("dk", 128 * d * 4, torch.float32, (128, d)),
                 ("dq", 128 * d * 4, torch.float32, (128, d))]
    rec = sum(nbytes for _, nbytes, _, _ in parts)
    raw = ws[off:off + n * rec].view(n, rec)
    out, o = {}, 0
    for name, nbytes, dt, shape in parts:
        out[name] = raw[:, o:o + nbytes].contiguous().view(dt).view(prob.B * prob.Hq, nb, nb, *shape)
        o += nbytes
    return out


# ---------------------------------------------------------------------------- buffers and autograd


def empty_bytes(nbytes: int, device) -> torch.Tensor:
    """A device byte buffer (torch allocations are 256-byte aligned)."""
    return torch.empty(max(int(nbytes), 16), dtype=torch.uint8, device=device)


def quantized_views(prob: Problem, saved: torch.Tensor) -> dict:
    """Views of the `saved` buffer of sagebwd_fwd (layout of the library: 256-byte aligned sections
    q^, k^, v^ (BF16), sQ, sK, sV (FP32 block scales), mean of K (FP32), channel balancing exponents (int32))."""
    def al(x):
        return (x + 255) // 256 * 256
    B, Hq, Hkv, N, d = prob.B, prob.Hq, prob.Hkv, prob.N, prob.d
    nb = (N + 127) // 128
    sizes = [("q", B * Hq * N * d * 2), ("k", B * Hkv * N * d * 2), ("v", B * Hkv * N * d * 2),
             ("sq", B * Hq * nb * 4), ("sk", B * Hkv * nb * 4), ("sv", B * Hkv * nb * 4), ("mu", B * Hkv * d * 4),
             ("e", B * Hkv * d * 4)]
    if prob.smooth_q:
        sizes += [("qm", B * Hq * nb * d * 4), ("qb", B * Hq * nb * nb * 128 * 4)]
    if prob.fp8:
        sizes += [("q8", B * Hq * N * d), ("k8", B * Hkv * N * d), ("v8t", B * Hkv * d * nb * 128)]
    out, off = {}, 0
    for name, n in sizes:
        out[name] = saved[off:off + n]
        off += al(n)
    out["q"] = out["q"].view(torch.bfloat16).view(B, Hq, N, d)
    out["k"] = out["k"].view(torch.bfloat16).view(B, Hkv, N, d)
    out["v"] = out["v"].view(torch.bfloat16).view(B, Hkv, N, d)
    out["sq"] = out["sq"].view(torch.float32).view(B * Hq, nb)
    out["sk"] = out["sk"].view(torch.float32).view(B * Hkv, nb)
    out["sv"] = out["sv"].view(torch.float32).view(B * Hkv, nb)
    out["mu"] = out["mu"].view(torch.float32).view(B * Hkv, d)
    out["e"] = out["e"].view(torch.int32).view(B * Hkv, d)
    if prob.smooth_q:
        out["qm"] = out["qm"].view(torch.float32).view(B * Hq, nb, d)
        out["qb"] = out["qb"].view(torch.float32).view(B * Hq, nb, nb * 128)
    if prob.fp8:  # E4M3 bytes
        out["q8"] = out["q8"].view(B * Hq, N, d)
        out["k8"] = out["k8"].view(B * Hkv, N, d)
        out["v8t"] = out["v8t"].view(B * Hkv, d, nb * 128)
    return out


def _check_inputs(q, k, v):
    for t in (q, k, v):
        if not (t.is_cuda and t.dtype == torch.bfloat16 and t.is_contiguous() and t.dim() == 4):
            raise ValueError("q, k, v must be contiguous 4-D bfloat16 CUDA tensors [B, H, N, d]")


# ---------------------------------------------------------------------------- device status of autograd calls
# Every kernel bounds its waits; a wait that runs out writes SAGEBWD_ERR_TIMEOUT into the status word
# of the call's workspace and the call's outputs are then incomplete.  The autograd path does not
# synchronize after each call: it copies the status word to pinned host memory behind the call's
# kernels and records an event; the word is read once the event has completed -- at the start of
# any later forward or backward call, or by check_errors(), which waits -- and a non-OK word raises
# SageBwdError there, naming the call it came from.
_status_lock = threading.Lock()
_status_pending = []  # (event, pinned int32 host tensor, call name)


def _queue_status(ws: torch.Tensor, where: str):
    host = torch.empty(1, dtype=torch.int32, pin_memory=True)
    host.copy_(ws[:4].view(torch.int32), non_blocking=True)
    ev = torch.cuda.Event()
    ev.record()
    with _status_lock:
        _status_pending.append((ev, host, where))


def _poll_status(block: bool = False):
    with _status_lock:
        pending = list(_status_pending)
        _status_pending.clear()
    keep, err = [], None
    for ev, host, where in pending:
        if block:
            ev.synchronize()
        if err is None and (block or ev.query()):
            code = int(host.item()) & 0xFF
            if code != 0:
                err = SageBwdError(code, f"{where} (device status)")
        elif err is None:
            keep.append((ev, host, where))
    with _status_lock:
        _status_pending[:0] = keep
    if err is not None:
        raise err


def check_errors():
    """Wait for every attention() call issued so far and raise SageBwdError if any of them reported a
    device-side error (a bounded wait that ran out).  Later calls also raise the errors of earlier
    calls whose kernels have finished by then."""
    _poll_status(block=True)


class SageBwdAttention(torch.autograd.Function):
    """softmax(scale Q K^T) V with SageBwd's INT8 forward and backward."""

    @staticmethod
    def forward(ctx, q, k, v, causal=False, softmax_scale=0.0, smooth_k=True, balance_qk=False, ds_subexp=False,
                qk_subexp=None, smooth_q=False, flags=0, wait_timeout_ms=0, fp8=False):
        _poll_status()
        _check_inputs(q, k, v)
        prob = Problem.from_tensors(q, k, causal, smooth_k=smooth_k, softmax_scale=softmax_scale,
                                    balance_qk=balance_qk, ds_subexp=ds_subexp, qk_subexp=qk_subexp,
                                    smooth_q=smooth_q, flags=flags, wait_timeout_ms=wait_timeout_ms, fp8=fp8)
        o = torch.empty_like(q)
        lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
        saved = empty_bytes(sagebwd_saved_bytes(prob), q.device)
        ws = empty_bytes(sagebwd_workspace_bytes(prob, 0), q.device)
        sagebwd_fwd(prob, q, k, v, o, lse, saved, ws)
        _queue_status(ws, "sagebwd_fwd")
        ctx.prob = prob
        ctx.save_for_backward(q, k, v, o, lse, saved)
        return o

    @staticmethod
    def backward(ctx, do):
        _poll_status()
        q, k, v, o, lse, saved = ctx.saved_tensors
        prob = ctx.prob
        do = do.contiguous()
        dq = torch.empty_like(q)
        dk = torch.empty_like(k)
        dv = torch.empty_like(v)
        ws = empty_bytes(sagebwd_workspace_bytes(prob, 1), q.device)
        sagebwd_bwd(prob, q, k, v, o, do, lse, saved, dq, dk, dv, ws)
        _queue_status(ws, "sagebwd_bwd")
        return dq, dk, dv, None, None, None, None, None, None, None, None, None, None


def attention(q, k, v, causal=False, softmax_scale=0.0, smooth_k=True, balance_qk=False, ds_subexp=False,
              qk_subexp=None, smooth_q=False, flags=0, wait_timeout_ms=0, fp8=False):
    """SageBwd attention on BF16 [B, H, N, d] CUDA tensors (GQA when k/v have fewer heads).

    balance_qk turns on the library's power-of-two Q/K channel balancing before quantization
    (for inputs with channel outliers; Q K^T is unchanged exactly); ds_subexp refines the dS codes
    with power-of-two sub-scales per key and 32-query group (dQ, dK several times closer to exact);
    qk_subexp (on by default, the library's Q/K granularity) refines Q and K with power-of-two
    sub-scales per 8-channel group of each block; qk_subexp=False keeps one scale per block;
    smooth_q subtracts each 128-token block's channel means from Q before quantizing and adds their
    logit term back in FP32 (for queries with a large common offset; not with balance_qk).
    flags (SAGEBWD_FLAG_*) and wait_timeout_ms pass through to the library (0: defaults).
    fp8=True runs the FP8 E4M3 variant of the method (every quantizer stores E4M3 values scaled to
    448 instead of INT8 codes; not with the optional refinements).

    Device-side errors of a call (a bounded wait that ran out) raise SageBwdError at the next
    forward or backward call once the failing kernels have finished, or at check_errors()."""
    return SageBwdAttention.apply(q, k, v, causal, softmax_scale, smooth_k, balance_qk, ds_subexp, qk_subexp,
                                  smooth_q, flags, wait_timeout_ms, fp8)
