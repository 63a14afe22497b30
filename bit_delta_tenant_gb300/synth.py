"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module draws random numbers and rounds them to the storage types; it holds
none of the method's arithmetic (no delta, sign, scale or linear).  Both the GPU
path and the CPU oracle receive exactly the tensors made here.

Recipe (all draws from one ``torch.Generator`` seeded per case, on the device the
caller names; fp32 draws, then round-to-nearest-even to bf16):
  * W_base ~ N(0, sigma^2), rounded to bf16.
  * delta ~ Laplace(0, b) as b * Exp(1) * (+1 or -1 with probability 1/2), fp32;
    b is a scalar or one value per output row.
  * W_ft = bf16(fp32(W_base) + delta).
  * x ~ N(0, 1), rounded to bf16.
  * variant ids: uniform over [0, V), or Zipf(s) segment sizes (p_i ~ i^-s,
    floor plus largest-remainder rounding) with the tokens shuffled.
These stand in for the page's 70B base and its fine-tuned variants: no weights,
datasets or evaluation items are used.
"""
from __future__ import annotations

import numpy as np
import torch


def generator(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(int(seed))
    return g


def bf16_normal(shape, std: float, g: torch.Generator, device) -> torch.Tensor:
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    t.mul_(std)
    return t.to(torch.bfloat16)


def laplace_f32(shape, b, g: torch.Generator, device) -> torch.Tensor:
    """Laplace(0, b) draws in fp32; ``b`` is a float or a [rows] tensor (per-row scale)."""
    mag = torch.empty(shape, device=device, dtype=torch.float32).exponential_(1.0, generator=g)
    flip = torch.randint(0, 2, shape, generator=g, device=device, dtype=torch.int8)
    mag.mul_(flip.to(torch.float32).mul_(2.0).sub_(1.0))
    if isinstance(b, torch.Tensor):
        mag.mul_(b.to(device=device, dtype=torch.float32).reshape(-1, *([1] * (len(shape) - 1))))
    else:
        mag.mul_(float(b))
    return mag


def matrix_pair(n_out: int, n_in: int, sigma: float, b, seed: int, device="cpu"):
    """(W_base, W_ft) as bf16 [n_out, n_in].  ``b='row:lo:hi'`` draws b_j ~ U[lo, hi] per row."""
    g = generator(seed, device)
    w_base = bf16_normal((n_out, n_in), sigma, g, device)
    if isinstance(b, str) and b.startswith("row:"):
        _, lo, hi = b.split(":")
        lo, hi = float(lo), float(hi)
        bj = torch.rand((n_out,), generator=g, device=device, dtype=torch.float32) * (hi - lo) + lo
        d = laplace_f32((n_out, n_in), bj, g, device)
    else:
        d = laplace_f32((n_out, n_in), float(b), g, device)
    w_ft = (w_base.to(torch.float32) + d).to(torch.bfloat16)
    del d
    return w_base, w_ft


def activations(m: int, n_in: int, seed: int, device="cpu") -> torch.Tensor:
    g = generator(seed, device)
    return bf16_normal((m, n_in), 1.0, g, device)


def uniform_ids(m: int, n_variants: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return rng.integers(0, n_variants, size=m, dtype=np.int64).astype(np.int32)


def zipf_sizes(m: int, n_variants: int, s: float) -> list[int]:
    """Segment sizes proportional to i^-s (i = 1..V), floored, remainder by largest fraction."""
    p = np.array([(i + 1) ** (-s) for i in range(n_variants)], dtype=np.float64)
    p /= p.sum()
    raw = p * m
    sizes = np.floor(raw).astype(np.int64)
    short = m - int(sizes.sum())
    order = np.argsort(-(raw - sizes), kind="stable")
    sizes[order[:short]] += 1
    return [int(v) for v in sizes]


def zipf_ids(m: int, n_variants: int, s: float, seed: int) -> np.ndarray:
    """Segment i (size from zipf_sizes) belongs to variant i; tokens are shuffled."""
    sizes = zipf_sizes(m, n_variants, s)
    ids = np.concatenate([np.full(n, v, dtype=np.int32) for v, n in enumerate(sizes)])
    rng = np.random.default_rng(seed)
    return ids[rng.permutation(m)]


def as_u16(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (host copy)."""
    if t.dtype != torch.bfloat16:
        raise TypeError("expected bf16")
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def from_u16(a: np.ndarray, device="cpu") -> torch.Tensor:
    """numpy uint16 bf16 bit patterns -> bf16 tensor on ``device``."""
    a = np.ascontiguousarray(a, dtype=np.uint16)
    return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16).to(device)
