"""Inference-efficiency metrics of adaptive canvas denoising (host-side helpers).

Definitions from "DiffusionGemma Technical Report 정리", section "추론 효율 지표": with K
canvases, s_k denoising steps of canvas k and n_k valid tokens of canvas k (up to the first
end-of-sequence token):

  Total Tokens              = sum_k n_k
  Total Denoising Steps     = sum_k s_k
  Effective Denoising Steps = sum_k n_k s_k / sum_k n_k
  TPF (tokens per forward)  = sum_k n_k / (sum_k s_k + K - 1)
  TPS                       = TPF / t_fwd   (t_fwd: time of one denoising step)

The K - 1 term counts the extra forward pass that encodes each finished canvas into the
cache before the next one starts.
"""

from __future__ import annotations

from typing import Sequence

import numpy as np


def valid_tokens(canvas, eos_id: int = 1) -> int:
    """n_k: tokens before the first end-of-sequence id (the whole canvas if none)."""
    c = np.asarray(canvas).reshape(-1)
    hits = np.flatnonzero(c == eos_id)
    return int(hits[0]) if hits.size else int(c.size)


def total_tokens(n: Sequence[int]) -> int:
    return int(np.sum(n))


def total_denoising_steps(s: Sequence[int]) -> int:
    return int(np.sum(s))


def effective_denoising_steps(n: Sequence[int], s: Sequence[int]) -> float:
    n = np.asarray(n, np.float64)
    s = np.asarray(s, np.float64)
    return float((n * s).sum() / n.sum())


def tokens_per_forward(n: Sequence[int], s: Sequence[int]) -> float:
    K = len(n)
    return float(np.sum(n) / (np.sum(s) + K - 1))


def tokens_per_second(tpf: float, t_fwd_s: float) -> float:
    return float(tpf / t_fwd_s)


def canvas_token_steps_per_s(L: int, B: int, steps: int, seconds: float) -> float:
    """Throughput of the denoising core: canvas tokens x steps per second (L x B x steps / s)."""
    return float(L * B * steps / seconds)
