"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This module holds no attention arithmetic: it only draws i.i.d. normal
numbers from a seeded generator, scales them and rounds them to bf16 (round to
nearest even). Both sides then read the very same bf16 bits.

Workloads (the five synthetic shapes the attention-backward measurements are
quoted on; Q/K/V/dO are i.i.d. normal, tau = 1/sqrt(d)):

  tiny        B=1 H=2  H_kv=2  N=256   d=64  non-causal
  causal_mha  B=4 H=16 H_kv=16 N=2048  d=128 causal
  causal_gqa  B=2 H=32 H_kv=8  N=4096  d=128 causal (4 query heads per KV head)
  long_causal B=1 H=16 H_kv=16 N=16384 d=128 causal, dO ~ N(0, 0.1^2)
  softcap     B=8 H=16 H_kv=16 N=1024  d=64  non-causal, Q/K/V ~ N(0, 2^2),
              softcap 30 applied as S = 30 tanh(S_raw / 30)
"""
from dataclasses import dataclass, replace
import math

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    H_kv: int
    N: int
    d: int
    causal: bool
    softcap: float = 0.0
    sigma_qkv: float = 1.0
    sigma_do: float = 1.0
    seed_base: int = 20261202

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def G(self) -> int:
        return self.H // self.H_kv

    def flops(self) -> float:
        """Backward work: 5 GEMMs of 2 N^2 d per head, halved when causal."""
        f = self.B * self.H * 5.0 * 2.0 * self.N * self.N * self.d
        return f / 2.0 if self.causal else f

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    "tiny": Workload("tiny", 1, 2, 2, 256, 64, False, seed_base=20261202 + 1000),
    "causal_mha": Workload("causal_mha", 4, 16, 16, 2048, 128, True,
                           seed_base=20261202 + 2000),
    "causal_gqa": Workload("causal_gqa", 2, 32, 8, 4096, 128, True,
                           seed_base=20261202 + 3000),
    "long_causal": Workload("long_causal", 1, 16, 16, 16384, 128, True,
                            sigma_do=0.1, seed_base=20261202 + 4000),
    "softcap": Workload("softcap", 8, 16, 16, 1024, 64, False, softcap=30.0,
                        sigma_qkv=2.0, seed_base=20261202 + 5000),
}


def _normal_bf16(shape, sigma, seed):
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    x = torch.randn(shape, generator=g, dtype=torch.float32)
    if sigma != 1.0:
        x = x * sigma
    return x.to(torch.bfloat16)


def make_inputs(w: Workload):
    """bf16 CPU tensors q [B,H,N,d], k, v [B,H_kv,N,d], do [B,H,N,d].

    One seed per tensor: seed_base + {0: q, 1: k, 2: v, 3: do}.
    """
    qs = (w.B, w.H, w.N, w.d)
    ks = (w.B, w.H_kv, w.N, w.d)
    return {
        "q": _normal_bf16(qs, w.sigma_qkv, w.seed_base + 0),
        "k": _normal_bf16(ks, w.sigma_qkv, w.seed_base + 1),
        "v": _normal_bf16(ks, w.sigma_qkv, w.seed_base + 2),
        "do": _normal_bf16(qs, w.sigma_do, w.seed_base + 3),
    }


def sample_slices(w: Workload, count: int, seed: int = 7):
    """A seeded sample of distinct (batch, kv_head) slices of a workload."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    total = w.B * w.H_kv
    count = min(count, total)
    perm = torch.randperm(total, generator=g)[:count].tolist()
    return sorted((p // w.H_kv, p % w.H_kv) for p in perm)
