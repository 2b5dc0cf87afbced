"""Benchmark of the SageBwd hot path: INT8 attention forward + backward.

One step = the whole path on one batch of synthetic input already resident
in HBM: K mean + Q/K/V quantization, the fused forward, the backward
preprocess (D, dO quantization), the fused backward and the dQ conversion.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Prints ONE JSON line.  Throughput is TOPS with the FlashAttention FLOP
convention (forward 4 B Hq N^2 d, backward 2.5x forward, causal halves both).
Under torchrun (N > 1) every rank runs its own batch (independent problems,
weak scaling, no collective on the data path); rank 0 prints the line with
the maximum time over ranks.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import bit_trainable_attention_gb300 as sb  # noqa: E402
from bit_trainable_attention_gb300 import workloads as W  # noqa: E402

METRIC = "SageBwd fwd+bwd TOPS at seq 8K/16K (1 GB300); % of INT8 tensor peak; cos-sim"
L2_FLUSH_BYTES = 256 << 20
# tcgen05 kind::f16 is the instruction the six INT8-semantics products run on (integer-valued BF16
# operands); legacy mma.sync s8 and torch._int_mm measured on this GPU for the "% of INT8 peak" line.
INT8_MMA_SYNC_TOPS = 150.5
INT8_TORCH_INT_MM_TOPS = 78.3


# DRAM bytes (read + write) of one bwd_kernel launch on the qwen15b workload, from a
# one-pass ncu capture (dram__bytes_read.sum + dram__bytes_write.sum of the timed step's
# launch).  The figure belongs to the kernel sources it was taken from: once any of them
# changes the line reports null until the capture is repeated.
BWD_TRAFFIC = {"workload": "qwen15b", "bytes": 771040512 + 281135360,
               "sources_sha256": "31e4ead463e229feda528d0fbcabbb57133c3fc75b1c80dcefae01fa31ccb2a8"}
BWD_SOURCES = ["bit_trainable_attention_gb300/csrc/bwd.cu", "bit_trainable_attention_gb300/csrc/kernel_common.cuh",
               "bit_trainable_attention_gb300/csrc/ptx.cuh", "bit_trainable_attention_gb300/csrc/sagebwd_internal.h",
               "include/sagebwd.h"]


def bwd_traffic(w):
    import hashlib
    h = hashlib.sha256()
    for f in BWD_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    ok = h.hexdigest() == BWD_TRAFFIC["sources_sha256"] and w.name == BWD_TRAFFIC["workload"]
    return BWD_TRAFFIC["bytes"] if ok else None


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"bf16_burst": float(d["bf16_tflops"]), "bf16_sustained": float(d["bf16_tflops_sustained"]),
                "hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"bf16_burst": 1900.0, "bf16_sustained": 1700.0, "hbm_gbs": 6800.0, "source": "fallback"}


# ---------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every 25 ms, read by a background thread; wait()
    returns once the first sample has arrived, so the timed region that follows is covered."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        import threading
        self.proc, self.lines, self.first = None, [], threading.Event()
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "25",
                 "-i", str(device_index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.reader = threading.Thread(target=self._read, daemon=True)
        self.reader.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line)
            self.first.set()

    def wait(self, timeout: float = 10.0):
        if self.proc is not None:
            self.first.wait(timeout)

    def mark(self):
        """Index of the next sample: samples before it are not part of the timed region."""
        return len(self.lines)

    def stop(self, start: int = 0, end: int = None):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.reader.join(timeout=5)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        lines = self.lines[start:end] or self.lines[-1:]  # a very short region: the sample that follows it
        for line in lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------- the library arm
class Step:
    """Buffers and the stage-by-stage calls of one forward + backward step."""

    def __init__(self, w: W.Workload, dev, balance_qk=False, ds_subexp=False, qk_subexp=None, inputs=None,
                 smooth_q=False, flags=0, fp8=False):
        self.w = w
        x = W.make_inputs(w) if inputs is None else inputs
        self.host = x
        self.x = {k: v.to(dev) for k, v in x.items()}
        self.prob = sb.Problem.make(w.B, w.Hq, w.Hkv, w.N, w.d, w.causal, balance_qk=balance_qk,
                                    ds_subexp=ds_subexp, qk_subexp=qk_subexp, smooth_q=smooth_q, flags=flags,
                                    fp8=fp8)
        p = self.prob
        self.o = torch.empty_like(self.x["q"])
        self.lse = torch.empty(w.B, w.Hq, w.N, dtype=torch.float32, device=dev)
        self.saved = sb.empty_bytes(sb.sagebwd_saved_bytes(p), dev)
        self.ws0 = sb.empty_bytes(sb.sagebwd_workspace_bytes(p, 0), dev)
        self.ws1 = sb.empty_bytes(sb.sagebwd_workspace_bytes(p, 1), dev)
        self.dq = torch.empty_like(self.x["q"])
        self.dk = torch.empty_like(self.x["k"])
        self.dv = torch.empty_like(self.x["v"])

    def run(self, ev=None):
        """The five stages; ev (optional) = 6 events recorded between them."""
        p, x = self.prob, self.x
        s = torch.cuda.current_stream()
        rec = (lambda i: ev[i].record(s)) if ev is not None else (lambda i: None)
        rec(0)
        sb.sagebwd_fwd_quantize(p, x["q"], x["k"], x["v"], self.saved, self.ws0, s)
        rec(1)
        sb.sagebwd_fwd_attention(p, self.saved, self.o, self.lse, self.ws0, s)
        rec(2)
        sb.sagebwd_bwd_prepare(p, self.o, x["do"], self.ws1, s)
        rec(3)
        sb.sagebwd_bwd_attention(p, x["v"], x["do"], self.lse, self.saved, self.dk, self.dv, self.ws1, s)
        rec(4)
        sb.sagebwd_bwd_finish(p, self.saved, self.dq, self.dk, self.dv, self.ws1, s)
        rec(5)

    # kernels of ours per step: [K mean or Q/K statistics: partial + final] + quantize + fwd + prep + bwd
    # + gradient convert
    def launches(self):
        return (2 if (self.prob.smooth_k or self.prob.balance_qk) else 0) + 5 + (1 if self.prob.smooth_q else 0)


def time_torch_sdpa(step: Step, steps: int, warmup: int, flush: torch.Tensor):
    """PyTorch's BF16 scaled_dot_product_attention forward + backward on the same inputs (the
    backend torch picks on this GPU), timed like the library's step: context for the INT8 path,
    which here runs on the BF16 tensor-core instructions (no INT8 tcgen05 form on sm_103a)."""
    w, x = step.w, step.x
    q = x["q"].detach().clone().requires_grad_(True)
    k = x["k"].detach().clone().requires_grad_(True)
    v = x["v"].detach().clone().requires_grad_(True)
    do = x["do"]
    gqa = w.Hq != w.Hkv

    def one():
        o = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=w.causal, enable_gqa=gqa)
        o.backward(do)
        q.grad = k.grad = v.grad = None

    for _ in range(warmup):
        flush.zero_()
        one()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    for i in range(steps):
        flush.zero_()
        ev[i][0].record()
        one()
        ev[i][1].record()
    torch.cuda.synchronize()
    ms = statistics.median(e[0].elapsed_time(e[1]) for e in ev)
    return {"ms_per_step": round(ms, 4), "tflops": round((w.flops_fwd() + w.flops_bwd()) / (ms * 1e-3) / 1e12, 2),
            "dtype": "bf16", "note": "torch.nn.functional.scaled_dot_product_attention fwd+bwd, same shapes"}


_REF_CACHE = {}


def torch_reference(step: Step):
    """O, dQ, dK, dV of PyTorch FP32 attention on the step's inputs (computed once per input set)."""
    key = (step.w, id(step.host))
    if key not in _REF_CACHE:
        _REF_CACHE.clear()
        w, x = step.w, step.x
        q = x["q"].float().requires_grad_(True)
        k = x["k"].float().requires_grad_(True)
        v = x["v"].float().requires_grad_(True)
        kk = k.repeat_interleave(w.G, dim=1)
        vv = v.repeat_interleave(w.G, dim=1)
        o = torch.nn.functional.scaled_dot_product_attention(q, kk, vv, is_causal=w.causal)
        o.backward(x["do"].float())
        _REF_CACHE[key] = {"o": o.detach(), "dq": q.grad, "dk": k.grad, "dv": v.grad}
    return _REF_CACHE[key]


def cossim_vs_torch(step: Step):
    """Cosine similarity of O, dQ, dK, dV against PyTorch FP32 attention (not timed)."""
    ref = torch_reference(step)
    got = {"o": step.o, "dq": step.dq, "dk": step.dk, "dv": step.dv}
    out = {}
    for name in ("o", "dq", "dk", "dv"):
        a, b = got[name].float().reshape(-1), ref[name].reshape(-1)
        out[name] = round(float(torch.nn.functional.cosine_similarity(a, b, dim=0)), 6)
    return out


def fp8_variant(step: Step, args, dev, flush):
    """The FP8 E4M3 variant of the method on the same inputs (forward on the FP8 tensor cores):
    step time and its stages (timed like the headline, shorter) and CosSim against FP32 attention."""
    other = Step(step.w, dev, inputs=step.host, fp8=True)
    total, stage = time_device(other, max(10, args.steps // 5), 3, flush, lambda: None)
    ms = sum(total) / len(total)
    st = [sum(x) / len(x) for x in stage]
    w = step.w
    out = {"ms_per_step": round(ms, 4), "tops": round((w.flops_fwd() + w.flops_bwd()) / (ms * 1e-3) / 1e12, 2),
           "breakdown_ms": {"quantize": round(st[0], 4), "fwd": round(st[1], 4), "bwd": round(st[3], 4)},
           "fwd_kernel_tflops": round(w.flops_fwd() / (st[1] * 1e-3) / 1e12, 1),
           "cossim_vs_torch_fp32": cossim_vs_torch(other),
           "note": "E4M3 values scaled to 448 at the INT8 granularity; forward S and PV on tcgen05 kind::f8f6f4, "
                   "backward on the same values in BF16 operands"}
    code0, _ = sb.sagebwd_check_status(other.ws0)
    code1, _ = sb.sagebwd_check_status(other.ws1)
    out["status"] = [code0, code1]
    del other
    return out


def error_attribution(step: Step, dev):
    """CosSim against FP32 attention with one quantizer at a time storing BF16 of its scaled values
    instead of INT8 codes (SAGEBWD_FLAG_BF16_*): which quantizer carries the error, on this workload
    at full size (untimed)."""
    out = {"none": cossim_vs_torch(step)}
    for name, flag in sb.FLAG_BF16.items():
        other = Step(step.w, dev, inputs=step.host, flags=flag, balance_qk=bool(step.prob.balance_qk),
                     qk_subexp=bool(step.prob.qk_subexp))
        other.run()
        torch.cuda.synchronize()
        code0, _ = sb.sagebwd_check_status(other.ws0)
        code1, _ = sb.sagebwd_check_status(other.ws1)
        out[name] = {**cossim_vs_torch(other), "status": [code0, code1]}
        del other
    return out


def time_device(step: Step, steps: int, warmup: int, flush: torch.Tensor, dist_barrier, on_timed=None):
    for _ in range(warmup):
        flush.zero_()
        step.run()
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(steps)]
    dist_barrier()
    torch.cuda.synchronize()
    if on_timed is not None:
        on_timed()  # the timed region starts here
    for i in range(steps):
        flush.zero_()  # L2 flush between timed steps, outside the events
        step.run(evs[i])
    torch.cuda.synchronize()
    dist_barrier()
    stage = [[evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(steps)] for j in range(5)]
    total = [evs[i][0].elapsed_time(evs[i][5]) for i in range(steps)]
    return total, stage


OPTIONS = ("balance_qk", "qk_subexp", "ds_subexp")


def other_settings(step: Step, args, dev, flush):
    """The same workload with the library's optional quantizer refinements (Q/K channel balancing,
    Q/K sub-scales, dS sub-scales) in other combinations -- none, each alone, all -- skipping the
    timed one: shorter timings (reported, not the headline) and their cosine similarities."""
    mine = tuple(bool(getattr(step.prob, o)) for o in OPTIONS)
    combos = [(False,) * 3] + [tuple(i == j for j in range(3)) for i in range(3)] + [(True,) * 3]
    out = []
    for combo in combos:
        if combo == mine and not step.prob.smooth_q:
            continue
        kw = dict(zip(OPTIONS, combo))
        other = Step(step.w, dev, inputs=step.host, **kw)
        total, stage = time_device(other, max(5, args.steps // 5), 3, flush, lambda: None)
        out.append({**kw, "ms_per_step": round(sum(total) / len(total), 4),
                    "quantize_ms": round(sum(stage[0]) / len(stage[0]), 4),
                    "bwd_ms": round(sum(stage[3]) / len(stage[3]), 4), "cossim_vs_torch_fp32": cossim_vs_torch(other)})
        del other
    return out


def time_e2e(step: Step, steps: int, warmup: int, flush: torch.Tensor, dist_barrier):
    """Public API (sagebwd_fwd + sagebwd_bwd) with pinned host inputs and outputs: every step uploads
    its Q, K, V, dO and downloads its O, dQ, dK, dV.  As a training loop that prefetches its next batch
    would, the device buffers are double-buffered and the copies run on two more streams (uploads,
    downloads; the link is full duplex): step i+1's inputs go up and step i-1's results come down
    while step i computes.  Step i is timed from the end
    of the L2 flush that precedes it to the end of its compute (the last step also waits for its own
    results to arrive on the host), so every copy is inside some step's interval or hidden behind its
    compute; the copy stream starts a step's copies only after that step's interval has begun."""
    p = step.prob
    hin = {k: v.pin_memory() for k, v in step.host.items()}
    sets = []
    for _ in range(2):
        sets.append({"in": {k: torch.empty_like(step.x[k]) for k in ("q", "k", "v", "do")},
                     "o": torch.empty_like(step.o), "lse": torch.empty_like(step.lse), "dq": torch.empty_like(step.dq),
                     "dk": torch.empty_like(step.dk), "dv": torch.empty_like(step.dv)})
    hout = {k: torch.empty(step.__dict__[k].shape, dtype=step.__dict__[k].dtype, pin_memory=True)
            for k in ("o", "dq", "dk", "dv")}
    s = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()

    def run(n, timed):
        ev_start = [torch.cuda.Event(enable_timing=timed) for _ in range(n)]
        ev_end = [torch.cuda.Event(enable_timing=timed) for _ in range(n)]
        ev_in = [torch.cuda.Event() for _ in range(n)]
        ev_comp = [torch.cuda.Event() for _ in range(n)]
        ev_down = [torch.cuda.Event() for _ in range(n)]

        def upload(j):  # on the upload stream, into set j % 2
            with torch.cuda.stream(up):
                up.wait_event(ev_start[j - 1 if j > 0 else 0])  # inside the step whose compute hides it
                if j >= 2:
                    up.wait_event(ev_comp[j - 2])  # the set's previous reader (step j-2) has finished
                for k in ("q", "k", "v", "do"):
                    sets[j % 2]["in"][k].copy_(hin[k], non_blocking=True)
                ev_in[j].record(up)

        def download(j, after):  # on the download stream, after step j's compute and step `after`'s start
            with torch.cuda.stream(down):
                down.wait_event(ev_start[after])
                down.wait_event(ev_comp[j])
                for k in ("o", "dq", "dk", "dv"):
                    hout[k].copy_(sets[j % 2][k], non_blocking=True)
                ev_down[j].record(down)

        up.wait_stream(s)
        down.wait_stream(s)
        for i in range(n):
            B = sets[i % 2]
            flush.zero_()
            ev_start[i].record(s)
            if i == 0:
                upload(0)
            if i >= 1:
                download(i - 1, i)
            if i + 1 < n:
                upload(i + 1)
            s.wait_event(ev_in[i])
            if i >= 2:
                s.wait_event(ev_down[i - 2])  # step i-2's results, in this set, have reached the host
            x = B["in"]
            sb.sagebwd_fwd(p, x["q"], x["k"], x["v"], B["o"], B["lse"], step.saved, step.ws0, s)
            sb.sagebwd_bwd(p, x["q"], x["k"], x["v"], B["o"], x["do"], B["lse"], step.saved, B["dq"], B["dk"], B["dv"],
                           step.ws1, s)
            ev_comp[i].record(s)
            if i == n - 1:
                download(i, i)
                s.wait_event(ev_down[i])
            ev_end[i].record(s)
        torch.cuda.synchronize()
        return [ev_start[i].elapsed_time(ev_end[i]) for i in range(n)] if timed else []

    run(warmup, False)
    dist_barrier()
    torch.cuda.synchronize()
    ms = run(steps, True)
    dist_barrier()
    h2d = sum(v.numel() * v.element_size() for v in hin.values())
    d2h = sum(v.numel() * v.element_size() for v in hout.values())
    return ms, h2d, d2h


# ---------------------------------------------------------------------------- layer-stack timing
LLAMA_1B = {"layers": 16, "hidden": 2048, "inter": 8192, "hq": 32, "hkv": 8, "d": 64}


def _rms(x, eps=1e-6):
    return x * torch.rsqrt(x.float().pow(2).mean(-1, keepdim=True) + eps).to(x.dtype)


class _LlamaShapedStack:
    """Random-weight decoder layers of Llama-3.2-1B's shapes (RMSNorm, fused QKV projection,
    QK-norm, grouped-query attention, output projection, SwiGLU MLP, residuals; no RoPE), BF16.
    Only timing: the weights are random, so nothing here is a trained model."""

    def __init__(self, cfg, dev, seed=0):
        g = torch.Generator(device="cpu").manual_seed(seed)
        h, f, hq, hkv, d = cfg["hidden"], cfg["inter"], cfg["hq"], cfg["hkv"], cfg["d"]
        self.cfg = cfg

        def w(i, o):
            return (torch.randn(o, i, generator=g) * i ** -0.5).to(torch.bfloat16).to(dev).requires_grad_(True)
        self.layers = [{"qkv": w(h, (hq + 2 * hkv) * d), "o": w(hq * d, h), "up": w(h, f), "gate": w(h, f),
                        "down": w(f, h)} for _ in range(cfg["layers"])]

    def params(self):
        return [t for layer in self.layers for t in layer.values()]

    def forward(self, x, attn):
        c = self.cfg
        B, N, _ = x.shape
        for L in self.layers:
            qkv = torch.nn.functional.linear(_rms(x), L["qkv"])
            q, k, v = qkv.split([c["hq"] * c["d"], c["hkv"] * c["d"], c["hkv"] * c["d"]], dim=-1)
            q = _rms(q.view(B, N, c["hq"], c["d"])).transpose(1, 2).contiguous()  # QK-norm over d
            k = _rms(k.view(B, N, c["hkv"], c["d"])).transpose(1, 2).contiguous()
            v = v.view(B, N, c["hkv"], c["d"]).transpose(1, 2).contiguous()
            o = attn(q, k, v).transpose(1, 2).reshape(B, N, c["hq"] * c["d"])
            x = x + torch.nn.functional.linear(o, L["o"])
            hmid = _rms(x)
            mlp = torch.nn.functional.silu(torch.nn.functional.linear(hmid, L["gate"])) * \
                torch.nn.functional.linear(hmid, L["up"])
            x = x + torch.nn.functional.linear(mlp, L["down"])
        return x


def time_layer_stack(n_tokens: int, steps: int, warmup: int, dev):
    """Forward + backward of a Llama-1B-shaped layer stack (random weights, batch 1) with the
    attention from this library against PyTorch's BF16 SDPA; everything else identical (cuBLAS
    GEMMs through torch).  The pages' end-to-end claim is about this kind of step (Llama 1B at
    8K/16K tokens per step, 2.1 s -> 1.9 s per iteration on an RTX4090)."""
    cfg = LLAMA_1B
    stack = _LlamaShapedStack(cfg, dev)
    g = torch.Generator(device="cpu").manual_seed(1)
    x0 = torch.randn(1, n_tokens, cfg["hidden"], generator=g).to(torch.bfloat16).to(dev)
    gy = torch.randn(1, n_tokens, cfg["hidden"], generator=g).to(torch.bfloat16).to(dev)
    attns = {
        "sagebwd": lambda q, k, v: sb.attention(q, k, v, causal=True),
        "torch_sdpa_bf16": lambda q, k, v: torch.nn.functional.scaled_dot_product_attention(
            q, k, v, is_causal=True, enable_gqa=True),
    }
    out = {}
    for name, attn in attns.items():
        def one():
            x = x0.detach().requires_grad_(True)
            stack.forward(x, attn).backward(gy)
            for t in stack.params():
                t.grad = None
        for _ in range(warmup):
            one()
        torch.cuda.synchronize()
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
        for i in range(steps):
            ev[i][0].record()
            one()
            ev[i][1].record()
        torch.cuda.synchronize()
        out[name + "_ms"] = round(statistics.median(e[0].elapsed_time(e[1]) for e in ev), 3)
    out["speedup"] = round(out["torch_sdpa_bf16_ms"] / out["sagebwd_ms"], 4)
    out["workload"] = (f"Llama-3.2-1B-shaped stack: {cfg['layers']} layers, hidden {cfg['hidden']}, "
                       f"{cfg['hq']}/{cfg['hkv']} heads, d {cfg['d']}, SwiGLU {cfg['inter']}, QK-norm, no RoPE, "
                       f"batch 1, {n_tokens} tokens, causal, BF16, random weights; forward + backward, no optimizer")
    return out


# ---------------------------------------------------------------------------- the oracle (CPU) arm
def oracle_sample_run(w: W.Workload, n_tokens: int, opts: dict):
    """Time the oracle on the first n_tokens tokens of the workload's own inputs (all heads, full
    forward + backward of that prefix), with the library arm's quantizer settings (opts).
    Returns (seconds, algorithmic ops of the sample, threads)."""
    import oracle  # the CPU baseline leg is the one place bench.py runs the oracle
    x = W.make_inputs(w)
    sub = {k: v[:, :, :n_tokens].contiguous() for k, v in x.items()}
    ws = w.with_(N=n_tokens)
    op = oracle.problem(ws.B, ws.Hq, ws.Hkv, ws.N, ws.d, ws.causal, **opts)
    t0 = time.perf_counter()
    oracle.pipeline(op, sub["q"], sub["k"], sub["v"], sub["do"])
    dt = time.perf_counter() - t0
    return dt, ws.flops_fwd() + ws.flops_bwd(), oracle.max_threads()


def oracle_opts(args) -> dict:
    """The oracle's settings for the quantizer configuration the library arm times."""
    fp8 = bool(getattr(args, "fp8", False))
    return {"qk_subexp": not (args.qk_plain or fp8), "ds_subexp": bool(args.ds_subexp),
            "balance_qk": bool(args.balance_qk), "smooth_q": bool(args.smooth_q), "fp8": fp8}


def pick_sample_tokens(w: W.Workload, budget_s: float, opts: dict):
    """Largest multiple of 128 tokens whose oracle run should take about budget_s seconds (quadratic cost)."""
    n = min(256, w.N)
    dt, _, _ = oracle_sample_run(w, n, opts)
    target = int(n * (budget_s / max(dt, 1e-3)) ** 0.5)
    return max(128, min(w.N, target // 128 * 128))


def cpu_baseline(w: W.Workload, budget_s: float, opts: dict):
    n = pick_sample_tokens(w, budget_s, opts)
    dt, ops, cores = oracle_sample_run(w, n, opts)
    return {"value": round(ops / dt / 1e12, 6), "unit": "TOPS", "cores": cores, "kind": "oracle",
            "sample": f"first {n} of {w.N} tokens of the same inputs, all {w.B}x{w.Hq} heads, full forward + "
                      f"backward of that prefix ({ops:.3e} ops in {dt:.2f} s)"}


def run_reference(args, w):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    # each step a bounded sample: at most reference_step_s seconds, and the whole warm-up +
    # timed run within reference_total_s
    step_s = min(args.reference_step_s, args.reference_total_s / max(1, args.steps + args.warmup))
    opts = oracle_opts(args)
    n = pick_sample_tokens(w, step_s, opts)
    for _ in range(args.warmup):
        oracle_sample_run(w, n, opts)
    times, ops, cores = [], 0.0, 1
    for _ in range(args.steps):
        dt, ops, cores = oracle_sample_run(w, n, opts)
        times.append(dt)
    mean = sum(times) / len(times)
    value = ops / mean / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TOPS", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(mean * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64 (codes decided in f32)", "data": "synthetic",
        "config": {"workload": describe(w), "sample": f"first {n} tokens"},
        "cpu_baseline": {"value": round(value, 6), "unit": "TOPS", "cores": cores, "kind": "oracle",
                         "sample": f"first {n} of {w.N} tokens of the same inputs, all heads, full forward + backward"},
        "e2e": {"value": round(value, 6), "unit": "TOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def max_over_ranks(vals, dist, device):
    """Each value's maximum over the ranks (the slowest replica sets the step time); identity
    without a process group."""
    if dist is None:
        return list(vals)
    t = torch.tensor([float(v) for v in vals], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def whole_job_tops(ops_per_replica: float, ms_max: float, world: int) -> float:
    """Whole-job throughput: every replica processes its own copy of the workload (weak scaling),
    so the job does world * ops in the slowest replica's time."""
    return world * ops_per_replica / (ms_max * 1e-3) / 1e12


def describe(w: W.Workload) -> str:
    return (f"{w.name}: B={w.B} Hq={w.Hq} Hkv={w.Hkv} N={w.N} d={w.d} {'causal' if w.causal else 'non-causal'}")


# ---------------------------------------------------------------------------- quantize stage bandwidth
def quantize_bandwidth(step: "Step", flush: torch.Tensor, hbm_gbs: float, reps: int = 10):
    """HBM GB/s of the quantize stage and of its kernels, each timed with CUDA events on the launching
    stream: algorithmic bytes per call / time.  Before every call, outside the events, L2 is flushed
    (a buffer larger than L2 written) and then a second buffer larger than L2 is read, so that the
    flush's dirty lines are written back before the call starts and the call's own traffic is timed.
    Algorithmic bytes: every input element read once per pass that must read it (K twice with
    K-smoothing: its channel sums, then its codes), every output written once; the quantized values
    are 2-byte integer-valued BF16 (the tensor cores' operand form).
      stage      sagebwd_fwd_quantize: K's block sums, their channel means, then one persistent launch
                 of Q's, V's and K's codes (the last two launched as programmatic dependents: the Q
                 and V blocks run beside the K-mean pass, the K blocks wait for the means)
      quantize_q sagebwd_quantize(Q): one persistent quantizer launch on Q alone
      quantize_v sagebwd_quantize(V): one persistent quantizer launch on V alone
      k_path     sagebwd_quantize(K): the single-operand K path (K mean pair, then K's codes)"""
    w, p, x = step.w, step.prob, step.x
    nb = (w.N + 127) // 128
    qe, ke = w.B * w.Hq * w.N * w.d, w.B * w.Hkv * w.N * w.d
    s = torch.cuda.current_stream()
    dev = x["q"].device
    xq = torch.empty_like(x["q"])
    sq = torch.empty(w.B * w.Hq * nb, dtype=torch.float32, device=dev)
    mu = torch.empty(w.B * w.Hkv * w.d, dtype=torch.float32, device=dev)
    calls = {
        "stage": (lambda: sb.sagebwd_fwd_quantize(p, x["q"], x["k"], x["v"], step.saved, step.ws0, s),
                  4 * qe + (6 if p.smooth_k else 4) * ke + 4 * ke + 4 * nb * (w.B * w.Hq + 2 * w.B * w.Hkv)),
        "quantize_q": (lambda: sb.sagebwd_quantize(p, sb.SAGEBWD_Q, x["q"], xq, sq, None, step.ws0, s),
                       4 * qe + 4 * nb * w.B * w.Hq),
        "quantize_v": (lambda: sb.sagebwd_quantize(p, sb.SAGEBWD_V, x["v"], xq, sq, None, step.ws0, s),
                       4 * ke + 4 * nb * w.B * w.Hkv),
        "k_path": (lambda: sb.sagebwd_quantize(p, sb.SAGEBWD_K, x["k"], xq, sq, mu, step.ws0, s),
                   (6 if p.smooth_k else 4) * ke + 4 * nb * w.B * w.Hkv),
    }
    out = {}
    evict = torch.empty(flush.numel() // 4, dtype=torch.float32, device=dev)
    evict.zero_()
    for name, (fn, nbytes) in calls.items():
        if p.smooth_q and name in ("stage", "quantize_q"):
            continue  # Q-smoothing's stage adds the logit terms; its Q path is the fused one only
        ts = []
        for r in range(reps + 2):
            flush.zero_()
            evict.sum()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            fn()
            e1.record(s)
            torch.cuda.synchronize()
            if r >= 2:
                ts.append(e0.elapsed_time(e1))
        us = statistics.median(ts) * 1e3
        gbs = nbytes / (us * 1e-6) / 1e9
        out[name] = {"bytes": int(nbytes), "us": round(us, 2), "gb_per_s": round(gbs, 1),
                     "frac_of_hbm": round(gbs / hbm_gbs, 3)}
    return out


def roofline_peak(peaks: dict, clocks: dict):
    """The BF16 dense denominator for the backward kernel: the burst figure, unless the clock record
    of the timed region shows the power cap (then the seconds-long sustained figure)."""
    capped = "sw_power_cap" in (clocks.get("reasons") or [])
    return (peaks["bf16_sustained"], "sustained") if capped else (peaks["bf16_burst"], "burst")


def config_summary(w: W.Workload, dev, args, flush, peaks):
    """A second configuration of the metric (the 8K-token GQA layer), timed like the headline:
    ms and TOPS of the step, the backward kernel's fraction of the BF16 peaks, CosSim vs FP32."""
    step = Step(w, dev, balance_qk=args.balance_qk, ds_subexp=args.ds_subexp,
                qk_subexp=not (args.qk_plain or args.fp8), smooth_q=args.smooth_q, fp8=args.fp8)
    total, stage = time_device(step, max(10, args.steps // 2), max(3, args.warmup), flush, lambda: None)
    ms = sum(total) / len(total)
    st = [sum(x) / len(x) for x in stage]
    bwd_tf = w.flops_bwd() / (st[3] * 1e-3) / 1e12
    fwd_tf = w.flops_fwd() / (st[1] * 1e-3) / 1e12
    out = {"workload": describe(w), "ms_per_step": round(ms, 4),
           "tops": round((w.flops_fwd() + w.flops_bwd()) / (ms * 1e-3) / 1e12, 2),
           "breakdown_ms": {"quantize": round(st[0], 4), "fwd": round(st[1], 4), "bwd_prepare": round(st[2], 4),
                            "bwd": round(st[3], 4), "grad_convert": round(st[4], 4)},
           "bwd_kernel_tflops": round(bwd_tf, 1), "bwd_frac_bf16_burst": round(bwd_tf / peaks["bf16_burst"], 4),
           "fwd_kernel_tflops": round(fwd_tf, 1), "fwd_frac_bf16_burst": round(fwd_tf / peaks["bf16_burst"], 4),
           "cossim_vs_torch_fp32": None if args.no_cossim else cossim_vs_torch(step)}
    code0, _ = sb.sagebwd_check_status(step.ws0)
    code1, _ = sb.sagebwd_check_status(step.ws1)
    out["status"] = [code0, code1]
    del step
    torch.cuda.empty_cache()
    return out


# ---------------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="qwen15b", choices=sorted(W.WORKLOADS))
    ap.add_argument("--impl", default="library", choices=["library", "reference"])
    ap.add_argument("--cpu-budget-s", type=float, default=15.0, help="oracle CPU-baseline sample size (seconds)")
    ap.add_argument("--reference-step-s", type=float, default=8.0, help="oracle seconds per reference-arm step")
    ap.add_argument("--reference-total-s", type=float, default=150.0,
                    help="oracle seconds for the whole reference-arm run (warm-up + timed steps)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end pass (profiling runs)")
    ap.add_argument("--no-cossim", action="store_true", help="skip the cosine-similarity reference (profiling runs)")
    ap.add_argument("--no-extras", action="store_true",
                    help="profiling runs: skip the second configuration, the layer stack, the per-kernel times "
                         "and the other option settings")
    ap.add_argument("--compare-sdpa", action="store_true",
                    help="also time PyTorch's BF16 SDPA forward + backward on the same inputs (context)")
    ap.add_argument("--balance-qk", action="store_true",
                    help="time the library's optional Q/K channel balancing (the other settings are reported beside)")
    ap.add_argument("--ds-subexp", action="store_true",
                    help="time the library's optional dS sub-scales (the other settings are reported beside)")
    ap.add_argument("--qk-plain", action="store_true",
                    help="time the plain one-scale-per-block Q/K mode instead of the default Q/K sub-scales")
    ap.add_argument("--fp8", action="store_true",
                    help="time the FP8 E4M3 variant instead of INT8 (forward on the FP8 tensor cores; no sub-scales)")
    ap.add_argument("--smooth-q", action="store_true",
                    help="time the library's optional Q-smoothing (block means of Q subtracted, logit term added)")
    ap.add_argument("--layer-step", type=int, default=8192, metavar="TOKENS",
                    help="also time a Llama-1B-shaped 16-layer stack forward + backward at TOKENS tokens with this "
                         "library's attention and with torch SDPA (context; 0 skips it)")
    ap.add_argument("--second-config", default="llama1b", choices=sorted(W.WORKLOADS) + ["none"],
                    help="the metric's other sequence length, reported as per_config (not the headline)")
    ap.add_argument("--seq", type=int, default=0,
                    help="profiling only: override the workload's sequence length (the line then names it)")
    args = ap.parse_args()
    w = W.WORKLOADS[args.workload]
    if args.seq > 0:
        w = dataclasses.replace(w, N=args.seq)

    if args.impl == "reference":
        run_reference(args, w)
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if dist is not None:
            dist.barrier()

    # the CPU baseline first (before any GPU work), rank 0 at N = 1 only
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, args.cpu_budget_s, oracle_opts(args))

    sb.load_library()
    step = Step(w, dev, balance_qk=args.balance_qk, ds_subexp=args.ds_subexp,
                qk_subexp=not (args.qk_plain or args.fp8), smooth_q=args.smooth_q, fp8=args.fp8)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    sampler = ClockSampler(local)
    sampler.wait()
    mark = [0]
    total, stage = time_device(step, args.steps, args.warmup, flush, barrier,
                               on_timed=lambda: mark.__setitem__(0, sampler.mark()))
    end = sampler.mark()
    clocks = sampler.stop(mark[0], end + 1)  # and the sample in flight when the region ended
    if args.no_e2e:
        e2e_ms, h2d, d2h = None, 0, 0
    else:
        e2e_ms, h2d, d2h = time_e2e(step, max(3, args.steps // 5), max(3, args.warmup), flush, barrier)
    code0, _ = sb.sagebwd_check_status(step.ws0)
    code1, _ = sb.sagebwd_check_status(step.ws1)

    ms = sum(total) / len(total)
    e2e = sum(e2e_ms) / len(e2e_ms) if e2e_ms else 0.0
    ms, e2e = max_over_ranks([ms, e2e], dist, dev)
    ops = w.flops_fwd() + w.flops_bwd()
    value = whole_job_tops(ops, ms, world)
    stage_ms = [sum(s) / len(s) for s in stage]
    peaks = load_peaks()
    peak, peak_kind = roofline_peak(peaks, clocks)
    bwd_ms = stage_ms[3]
    achieved = w.flops_bwd() / (bwd_ms * 1e-3) / 1e12
    fwd_achieved = w.flops_fwd() / (stage_ms[1] * 1e-3) / 1e12
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "TOPS", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": ("fp8 e4m3 (forward on tcgen05 kind::f8f6f4; backward e4m3 values in bf16 operands) + bf16 dP"
                  if args.fp8 else "int8 (integer-valued bf16 on tcgen05, fp32 accumulate) + bf16 dP"),
        "data": "synthetic",
        "config": {"workload": describe(w), "l2": "flushed between timed steps (256 MB write)",
                   "qk_granularity": "per-block scale + 8-channel power-of-two sub-scales (library default)"
                   if not (args.qk_plain or args.fp8) else "one scale per 128-token block",
                   "parallelism": f"{world} independent replicas" if world > 1 else "single GPU"},
        "breakdown_ms": {"quantize": round(stage_ms[0], 4), "fwd": round(stage_ms[1], 4),
                         "bwd_prepare": round(stage_ms[2], 4), "bwd": round(stage_ms[3], 4),
                         "grad_convert": round(stage_ms[4], 4)},
        "tops": {"fwd_incl_quantize": round(w.flops_fwd() / ((stage_ms[0] + stage_ms[1]) * 1e-3) / 1e12, 2),
                 "bwd_incl_prepare": round(w.flops_bwd() / (sum(stage_ms[2:]) * 1e-3) / 1e12, 2)},
        "roofline": {"kernel": "sagebwd bwd_kernel", "bound": "tensor", "achieved": round(achieved, 2),
                     "peak": peak, "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "traffic": bwd_traffic(w),
                     "traffic_unit": "bytes per launch (ncu dram__bytes_read.sum + dram__bytes_write.sum)",
                     "peak_kind": f"bf16 dense, {peak_kind} ({peaks['source']}): burst unless the timed "
                                  "region's clock record shows sw_power_cap",
                     "frac_of_burst": round(achieved / peaks["bf16_burst"], 4),
                     "frac_of_sustained": round(achieved / peaks["bf16_sustained"], 4),
                     "fwd_kernel": {"achieved": round(fwd_achieved, 2),
                                    "frac_of_burst": round(fwd_achieved / peaks["bf16_burst"], 4)}},
        "int8_peak_frac": {"vs_mma_sync_s8_ratio": round(value / world / INT8_MMA_SYNC_TOPS, 3),
                           "vs_torch_int_mm_ratio": round(value / world / INT8_TORCH_INT_MM_TOPS, 3),
                           "vs_bf16_dense_burst": round(value / world / peaks["bf16_burst"], 4),
                           "note": "ratios to the legacy INT8 paths measured on this GPU (mma.sync s8, "
                                   "torch._int_mm), not peak fractions: tcgen05 kind::i8 does not exist on "
                                   "sm_103a; the BF16 fraction is the peak of the instructions used"},
        "e2e": None if e2e_ms is None else {
            "value": round(world * ops / (e2e * 1e-3) / 1e12, 3), "unit": "TOPS", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e, 4),
            "copies": "double-buffered on two copy streams: step i+1's inputs up and step i-1's results down while "
                      "step i computes; each step timed from the end of its L2 flush"},
        "balance_qk": bool(args.balance_qk), "qk_subexp": bool(step.prob.qk_subexp),
        "ds_subexp": bool(args.ds_subexp), "smooth_q": bool(args.smooth_q), "fp8": bool(args.fp8),
        "gpu_launches": step.launches() * args.steps,
        "clocks": clocks,
        "status": [code0, code1],
    }
    if rank == 0:
        line["cossim_vs_torch_fp32"] = None if args.no_cossim else cossim_vs_torch(step)
        if not args.no_extras:
            line["quantize_hbm"] = quantize_bandwidth(step, flush, peaks["hbm_gbs"])
            if not args.no_cossim and not args.fp8:
                line["other_settings"] = other_settings(step, args, dev, flush)
                line["fp8_variant"] = fp8_variant(step, args, dev, flush)
                if not (args.ds_subexp or args.smooth_q):
                    line["error_attribution"] = error_attribution(step, dev)
        if args.compare_sdpa:
            line["torch_sdpa_bf16"] = time_torch_sdpa(step, max(5, args.steps // 2), args.warmup, flush)
        if not args.no_extras and args.second_config != "none" and args.second_config != w.name:
            del step
            torch.cuda.empty_cache()
            line["per_config"] = {args.second_config: config_summary(W.WORKLOADS[args.second_config], dev, args,
                                                                     flush, peaks)}
        if not args.no_extras and args.layer_step > 0:
            line["layer_step"] = time_layer_stack(args.layer_step, max(3, args.steps // 5), 2, dev)
        line["cpu_baseline"] = cpu
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
