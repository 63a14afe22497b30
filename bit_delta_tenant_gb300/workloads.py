"""Shapes and input distributions of the benchmarked and tested workloads.

Stand-ins for the page's 70B base with 14 fine-tuned variants (no weights or
datasets are used): Llama-style layer linears, 70B-shape linears, a
14-variant batch over one 8192x8192 base, and a full Llama-3-8B-shape stack.
Each matrix gets its own seed derived from the workload seed and its index.
"""
from __future__ import annotations

TINY = dict(name="tiny_256x512", n_out=256, n_in=512, m=8, sigma=0.02, b=1e-3, mode=0, seed=0)

LLAMA7B_LAYER = dict(
    name="llama7b_layer_decode",
    matrices=[("q", 4096, 4096), ("k", 4096, 4096), ("v", 4096, 4096), ("o", 4096, 4096),
              ("gate", 11008, 4096), ("up", 11008, 4096), ("down", 4096, 11008)],
    ms=(1, 4, 16), sigma=0.02, b=1e-3, mode=0, seed=1)

LLAMA70B_PREFILL = dict(
    name="llama70b_linears_prefill",
    matrices=[("attn_sq", 8192, 8192), ("mlp_up", 28672, 8192), ("mlp_down", 8192, 28672)],
    ms=(512, 2048, 8192), sigma=0.015, b="row:5e-4:2e-3", mode=1, seed=2)

GROUPED_14 = dict(
    name="grouped_14_variants_8192",
    n_out=8192, n_in=8192, n_variants=14, sigma=0.015, b_lo=5e-4, b_hi=2e-3, mode=0,
    decode_m=64, prefill_m=2048, zipf_s=1.1, seed=3)

LLAMA3_8B_STACK = dict(
    name="llama3_8b_stack",
    layers=32,
    matrices=[("q", 4096, 4096), ("k", 1024, 4096), ("v", 1024, 4096), ("o", 4096, 4096),
              ("gate", 14336, 4096), ("up", 14336, 4096), ("down", 4096, 14336)],
    ms=(1, 2048), sigma=0.02, b=1e-3, mode=0, seed=4)


def matrix_seed(workload_seed: int, index: int) -> int:
    return workload_seed * 100003 + index


def variant_scales(cfg=GROUPED_14) -> list[float]:
    n = cfg["n_variants"]
    lo, hi = cfg["b_lo"], cfg["b_hi"]
    return [lo + (hi - lo) * i / (n - 1) for i in range(n)]
