"""Seeded synthetic inputs for the Memory Caching forward, shared by the tests,
the smoke check and the benchmark.

This module holds none of the method's arithmetic: it only draws q, k, v, u
with the distributions of the workloads the method is measured on, and names
those workloads.  Draw order is q, k, v, u from one numpy PCG64 stream:
  q, k ~ N(0, 1), then each row scaled to unit L2 norm (in fp32);
  v ~ N(0, 1);  u ~ N(0, 1) / sqrt(d).
The values are then cast to the workload's input dtype (bf16 rounds to
nearest-even); every consumer, the oracle included, receives the cast values.

The SWLA workloads also draw per-token scalars (fp32, [B, H, L]) from a second
PCG64 stream (seed + 1000), in the order alpha, beta, lambda, with z ~ N(0, 1):
  alpha = 1 - 0.1 sigmoid(z)  (a decay in (0.9, 1)),  beta = sigmoid(z),  lambda = sigmoid(z).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

RESIDUAL, GRM, SOUP, SSC, MEAN = 0, 1, 2, 3, 4
MODE_NAMES = {RESIDUAL: "residual", GRM: "grm", SOUP: "soup", SSC: "ssc", MEAN: "mean"}


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    L: int
    d: int
    seg_len: int
    mode: int
    dtype: str  # "f32" or "bf16"
    topk: int = 0
    seed: int = 0
    swla: bool = False  # sliding-window linear attention (c = 2) update instead of M += v k^T

    @property
    def N(self) -> int:
        return (self.L + self.seg_len - 1) // self.seg_len

    @property
    def tokens(self) -> int:
        return self.B * self.L

    def with_(self, **kw) -> "Workload":
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)


# The synthetic workloads, each with its own seed (tiny = 0).
TINY = Workload("tiny-grm B1 H1 L256 d16 C64 fp32", 1, 1, 256, 16, 64, GRM, "f32", seed=0)
GRM_D64 = Workload("grm B4 H8 L4096 d64 C256 bf16", 4, 8, 4096, 64, 256, GRM, "bf16", seed=1)
SWEEP = tuple(
    Workload(f"sweep B8 H16 L8192 d128 C{c} bf16", 8, 16, 8192, 128, c, GRM, "bf16", seed=2)
    for c in (8192, 2048, 512, 128))
SSC_D128 = Workload("ssc B2 H16 L16384 d128 C256 k4 bf16", 2, 16, 16384, 128, 256, SSC, "bf16",
                    topk=4, seed=3)
LONG_GRM = Workload("long-grm B1 H16 L65536 d128 C1024 bf16", 1, 16, 65536, 128, 1024, GRM, "bf16",
                    seed=4)

SWLA_LONG = Workload("swla-grm B1 H16 L65536 d128 C1024 bf16", 1, 16, 65536, 128, 1024, GRM, "bf16",
                     seed=5, swla=True)

# Short segments (seg_len < d / 2), where the cached readout runs in the factorised form:
# the sweep's batch, heads, length and head dimension at seg_len 32 (N = 256).
FACT_C32 = Workload("fact-grm B8 H16 L8192 d128 C32 bf16", 8, 16, 8192, 128, 32, GRM, "bf16", seed=8)
# The long-context workload with twice as many, shorter segments (N = 128).
LONG_C512 = Workload("long-grm B1 H16 L65536 d128 C512 bf16", 1, 16, 65536, 128, 512, GRM, "bf16", seed=9)

ALL = (TINY, GRM_D64) + SWEEP + (SSC_D128, LONG_GRM, SWLA_LONG, FACT_C32, LONG_C512)


def _np_inputs(B: int, H: int, L: int, d: int, seed: int):
    rng = np.random.default_rng(seed)
    shape = (B, H, L, d)
    q = rng.standard_normal(shape, dtype=np.float32)
    k = rng.standard_normal(shape, dtype=np.float32)
    v = rng.standard_normal(shape, dtype=np.float32)
    u = rng.standard_normal(shape, dtype=np.float32)
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    u *= np.float32(1.0 / math.sqrt(d))
    return q, k, v, u


def make_inputs(B: int, H: int, L: int, d: int, seed: int, dtype: str = "bf16",
                device: str | torch.device = "cpu"):
    """Return (q, k, v, u) as contiguous torch tensors [B, H, L, d] of ``dtype``."""
    tdt = {"bf16": torch.bfloat16, "f32": torch.float32}[dtype]
    out = []
    for a in _np_inputs(B, H, L, d, seed):
        t = torch.from_numpy(a).to(tdt)
        out.append(t.to(device).contiguous())
    return tuple(out)


def workload_inputs(w: Workload, device="cpu"):
    return make_inputs(w.B, w.H, w.L, w.d, w.seed, w.dtype, device)


def make_swla_scalars(B: int, H: int, L: int, seed: int, device: str | torch.device = "cpu"):
    """Return (alpha, beta, lambda) as contiguous fp32 torch tensors [B, H, L]."""
    rng = np.random.default_rng(seed + 1000)
    shape = (B, H, L)
    za = rng.standard_normal(shape, dtype=np.float32)
    zb = rng.standard_normal(shape, dtype=np.float32)
    zl = rng.standard_normal(shape, dtype=np.float32)
    sig = lambda z: (1.0 / (1.0 + np.exp(-z.astype(np.float64)))).astype(np.float32)
    alpha = (np.float32(1.0) - np.float32(0.1) * sig(za)).astype(np.float32)
    return tuple(torch.from_numpy(np.ascontiguousarray(a)).to(device) for a in (alpha, sig(zb), sig(zl)))


def workload_swla_scalars(w: Workload, device="cpu"):
    return make_swla_scalars(w.B, w.H, w.L, w.seed, device)
