"""Seeded synthetic attention inputs (BF16 Q, K, V, dO) for tests and the bench.

This module only draws and shapes random inputs; it holds none of the
attention method's arithmetic.  The five named workloads follow the shapes of
the attention layers the SageBwd pages train and fine-tune ("SageBwd: A
Trainable Low-bit Attention", Abstract: QK-norm upstream of attention,
K-smoothing; "SageAttention3 ... An Exploration of 8-Bit Training", Key
results: Llama-1B training at 8K/16K tokens, Qwen2.5-1.5B fine-tuning, 400M
pre-training, CogVideoX video DiT):

  tiny       B=1 Hq=2  Hkv=2 N=128   d=64  non-causal  QK-norm, K offset sd 2
  pretrain   B=8 Hq=16 Hkv=16 N=2048 d=64  causal      QK-norm, K offset sd 2
  llama1b    B=1 Hq=32 Hkv=8 N=8192  d=64  causal      QK-norm, K offset sd 2
  qwen15b    B=1 Hq=12 Hkv=2 N=16384 d=128 causal      1% of Q and K channels x20
  videodit   B=2 Hq=30 Hkv=30 N=17776 d=64 non-causal  K offset sd 3

Recipe (all draws in FP32 on the CPU from one torch.Generator, cast to BF16
once at the end): Q, K, V, dO ~ N(0, 1); QK-norm is an RMSNorm over d (weight
1, eps 1e-6) of Q and K; the K offset is one N(0, sd^2) value per (kv head,
channel), shared by batch and tokens, added after the norm; outliers multiply
ceil(1% of heads*d) randomly chosen (head, channel) pairs of Q and of K by 20.
"""
from __future__ import annotations

import dataclasses
import math

import torch

SEED_BASE = 20260302


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    N: int
    d: int
    causal: bool
    qk_norm: bool = False
    k_offset_sd: float = 0.0
    outlier_frac: float = 0.0
    seed: int = SEED_BASE
    q_offset_sd: float = 0.0  # per (query head, channel) offset of Q (none in the named workloads)

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    def flops_fwd(self) -> float:
        """Dense attention forward FLOPs, 4*B*Hq*N^2*d, halved when causal."""
        f = 4.0 * self.B * self.Hq * self.N * self.N * self.d
        return f * 0.5 if self.causal else f

    def flops_bwd(self) -> float:
        """Backward = 2.5 x forward (five N^2 d products against two)."""
        return 2.5 * self.flops_fwd()


WORKLOADS = {
    "tiny": Workload("tiny", 1, 2, 2, 128, 64, False, qk_norm=True, k_offset_sd=2.0, seed=SEED_BASE + 0),
    "pretrain": Workload("pretrain", 8, 16, 16, 2048, 64, True, qk_norm=True, k_offset_sd=2.0, seed=SEED_BASE + 1),
    "llama1b": Workload("llama1b", 1, 32, 8, 8192, 64, True, qk_norm=True, k_offset_sd=2.0, seed=SEED_BASE + 2),
    "qwen15b": Workload("qwen15b", 1, 12, 2, 16384, 128, True, outlier_frac=0.01, seed=SEED_BASE + 3),
    "videodit": Workload("videodit", 2, 30, 30, 17776, 64, False, k_offset_sd=3.0, seed=SEED_BASE + 4),
}


def _rms_norm(x: torch.Tensor, eps: float = 1e-6) -> torch.Tensor:
    return x * torch.rsqrt(x.pow(2).mean(dim=-1, keepdim=True) + eps)


def _outliers(x: torch.Tensor, frac: float, g: torch.Generator) -> torch.Tensor:
    B, H, N, d = x.shape
    count = math.ceil(frac * H * d)
    pick = torch.randperm(H * d, generator=g)[:count]
    scale = torch.ones(H * d)
    scale[pick] = 20.0
    return x * scale.view(1, H, 1, d)


def make_inputs(w: Workload, seed: int | None = None) -> dict:
    """Return dict(q, k, v, do) of contiguous BF16 CPU tensors [B, H, N, d]."""
    g = torch.Generator().manual_seed(w.seed if seed is None else seed)
    q = torch.randn(w.B, w.Hq, w.N, w.d, generator=g)
    k = torch.randn(w.B, w.Hkv, w.N, w.d, generator=g)
    v = torch.randn(w.B, w.Hkv, w.N, w.d, generator=g)
    do = torch.randn(w.B, w.Hq, w.N, w.d, generator=g)
    if w.qk_norm:
        q = _rms_norm(q)
        k = _rms_norm(k)
    if w.k_offset_sd > 0:
        off = torch.randn(1, w.Hkv, 1, w.d, generator=g) * w.k_offset_sd
        k = k + off
    if w.outlier_frac > 0:
        q = _outliers(q, w.outlier_frac, g)
        k = _outliers(k, w.outlier_frac, g)
    if w.q_offset_sd > 0:  # drawn last, so the other draws do not depend on it
        q = q + torch.randn(1, w.Hq, 1, w.d, generator=g) * w.q_offset_sd
    bf = torch.bfloat16
    return {"q": q.to(bf).contiguous(), "k": k.to(bf).contiguous(), "v": v.to(bf).contiguous(),
            "do": do.to(bf).contiguous()}


def small(name: str, B: int, Hq: int, Hkv: int, N: int, d: int, causal: bool, seed: int, **recipe) -> Workload:
    """A test-sized workload with the same recipe knobs as the named ones."""
    return Workload(name, B, Hq, Hkv, N, d, causal, seed=seed, **recipe)
