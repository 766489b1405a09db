"""Seeded synthetic inputs and the workload table.

This module holds no arithmetic of the method: it only draws weights, prefix KV caches and
clean token canvases with fixed seeds, and names the workloads.  Both the CUDA path and the
CPU oracle receive the arrays it makes.

Workloads (canvas length 256 and vocabulary 262,144 as in "DiffusionGemma 완전분석",
section "스펙 정리"; the model dimensions are those of a Gemma-4-sized attention layer):

  tiny      B=1,  prefix 256 (global),       d 256,  4q/4kv x 64,  V 4,096,  12 steps, linear
  window1k  B=1,  prefix 1,024 (window 1,024), d 2,048, 16q/8kv x 128, V 262,144, 12 steps, cosine
  batch16   B=16, prefix 8,192 (global),     same dims, 48 steps, linear, lock at top-1 >= 0.9
  long128k  B=1,  prefix 131,072 (global),   same dims, 12 steps, linear
  sweep4k   B in {1, 8, 32, 64}, prefix 4,096 (global), same dims, cap 48 steps, linear,
            lock at 0.9, stop when every position is locked; plus noising of 64 x 256
            Zipf(1.1) tokens at t ~ U(0, 1)

Values: weights N(0, 0.02) and prefix K/V N(0, 1), stored in bfloat16; the canvas starts
uniform over the vocabulary (drawn by the method's own noising stream on each side).
"""

from __future__ import annotations

import dataclasses

import numpy as np
import torch

SCHED_LINEAR = 0
SCHED_COSINE = 1


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    L: int
    P: int
    window: int
    d: int
    H: int
    Hkv: int
    hd: int
    V: int
    T: int
    schedule: int
    lock_theta: float | None
    stop_when_all_locked: bool
    seed: int
    inv_tau: float = 1.0

    @property
    def canvas_tokens(self) -> int:
        return self.B * self.L

    def with_batch(self, B: int) -> "Workload":
        return dataclasses.replace(self, B=B, name=f"{self.name}-b{B}")

    def describe(self) -> str:
        win = f"window {self.window}" if self.window else "global"
        lock = f", lock at top-1 >= {self.lock_theta}" if self.lock_theta else ""
        stop = ", stop when all locked" if self.stop_when_all_locked else ""
        sched = "cosine" if self.schedule == SCHED_COSINE else "linear"
        return (f"{self.name}: batch {self.B}, canvas {self.L}, prefix {self.P} ({win}), "
                f"d_model {self.d}, {self.H}q/{self.Hkv}kv x {self.hd}, vocab {self.V}, "
                f"{sched} kappa, {self.T} Euler steps{lock}{stop}")


TINY = Workload("tiny", 1, 256, 256, 0, 256, 4, 4, 64, 4096, 12, SCHED_LINEAR, None, False, 0)
WINDOW1K = Workload("window1k", 1, 256, 1024, 1024, 2048, 16, 8, 128, 262144, 12, SCHED_COSINE,
                    None, False, 1)
BATCH16 = Workload("batch16", 16, 256, 8192, 0, 2048, 16, 8, 128, 262144, 48, SCHED_LINEAR,
                   0.9, False, 2)
LONG128K = Workload("long128k", 1, 256, 131072, 0, 2048, 16, 8, 128, 262144, 12, SCHED_LINEAR,
                    None, False, 3)
SWEEP4K = Workload("sweep4k", 1, 256, 4096, 0, 2048, 16, 8, 128, 262144, 48, SCHED_LINEAR,
                   0.9, True, 4)
SWEEP_BATCHES = (1, 8, 32, 64)
WORKLOADS = {w.name: w for w in (TINY, WINDOW1K, BATCH16, LONG128K, SWEEP4K)}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal_bf16(shape, std: float, seed: int, device="cpu") -> torch.Tensor:
    """N(0, std^2) drawn in float32 with a seeded generator, stored as bfloat16."""
    g = _gen(seed, device)
    x = torch.empty(shape, dtype=torch.float32, device=device)
    x.normal_(0.0, std, generator=g)
    return x.to(torch.bfloat16)


def make_model(w: Workload, device="cpu") -> dict:
    """Embedding / tied LM head E [V, d], fused Wqkv [(H + 2 Hkv) hd, d] (q rows, then k,
    then v) and Wo [d, H hd], all N(0, 0.02) in bfloat16."""
    s = 1000 * w.seed
    return {
        "E": normal_bf16((w.V, w.d), 0.02, s + 1, device),
        "Wqkv": normal_bf16(((w.H + 2 * w.Hkv) * w.hd, w.d), 0.02, s + 2, device),
        "Wo": normal_bf16((w.d, w.H * w.hd), 0.02, s + 3, device),
        "H": w.H, "Hkv": w.Hkv, "hd": w.hd,
    }


def make_prefix_kv(w: Workload, device="cpu", B: int | None = None):
    """Per-canvas prefix K and V caches [B, P, Hkv, hd], N(0, 1) in bfloat16."""
    B = w.B if B is None else B
    s = 1000 * w.seed
    shape = (B, w.P, w.Hkv, w.hd)
    return normal_bf16(shape, 1.0, s + 4, device), normal_bf16(shape, 1.0, s + 5, device)


def zipf_tokens(B: int, L: int, V: int, a: float, seed: int) -> np.ndarray:
    """Clean tokens with P(rank k) proportional to k^-a over ranks 1..V; token id = rank - 1."""
    ranks = np.arange(1, V + 1, dtype=np.float64)
    cdf = np.cumsum(ranks ** -a)
    cdf /= cdf[-1]
    u = np.random.Generator(np.random.Philox(seed)).random((B, L))
    return np.minimum(np.searchsorted(cdf, u, side="right"), V - 1).astype(np.int32)


def uniform_times(B: int, seed: int) -> np.ndarray:
    """Per-canvas noise levels t ~ U(0, 1) for training-style noising."""
    return np.random.Generator(np.random.Philox(seed + 17)).random(B)


def random_tokens(shape, V: int, seed: int) -> np.ndarray:
    """Tokens uniform over [0, V) from a seeded host generator (test inputs)."""
    return np.random.Generator(np.random.Philox(seed + 29)).integers(0, V, size=shape,
                                                                    dtype=np.int64).astype(np.int32)
