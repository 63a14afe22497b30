"""Shared test helpers: seeded cases on the device, oracle expectations, tolerance checks.

Expected values always come from the fp64 oracle (``oracle``), fed the same
synthetic inputs as the GPU; nothing here computes the method itself.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from bit_delta_tenant_gb300 import bitdelta as bd
from bit_delta_tenant_gb300 import synth

# Acceptance bounds: relative Frobenius error of y, per-element bound scaled by
# sum_k |x_tk| |W_eff,jk| (covers bf16 rounding of W_eff and of y), alpha.
Y_FROB_REL = 5e-3
Y_ELEM_SCALE = 2.0 ** -7
Y_ELEM_ABS = 1e-6
ALPHA_REL = 1e-6


def bf16_to_f64(u16: np.ndarray) -> np.ndarray:
    return (np.asarray(u16, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def y_host(y: torch.Tensor) -> np.ndarray:
    return bf16_to_f64(synth.as_u16(y))


def assert_y_close(y_gpu: np.ndarray, y_ref: np.ndarray, mag: np.ndarray, what: str = "y") -> None:
    assert y_gpu.shape == y_ref.shape, (y_gpu.shape, y_ref.shape)
    assert np.all(np.isfinite(y_gpu)), f"{what}: non-finite output"
    err = np.abs(y_gpu - y_ref)
    bound = Y_ELEM_SCALE * mag + Y_ELEM_ABS
    bad = err > bound
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {int(bad.sum())} elements out of bound; first at {tuple(i)}: "
                             f"gpu={y_gpu[tuple(i)]!r} ref={y_ref[tuple(i)]!r} bound={bound[tuple(i)]!r}")
    den = np.linalg.norm(y_ref)
    if den > 0:
        rel = np.linalg.norm(y_gpu - y_ref) / den
        assert rel <= Y_FROB_REL, f"{what}: relative Frobenius error {rel:.3e}"


class LinearCase:
    """One matrix: inputs on the device plus their host bit patterns and the oracle's compression."""

    def __init__(self, n_out, n_in, m, sigma=0.02, b=1e-3, mode=0, seed=0, device="cuda"):
        self.n_out, self.n_in, self.m, self.mode = n_out, n_in, m, mode
        self.w_base, self.w_ft = synth.matrix_pair(n_out, n_in, sigma, b, seed, device)
        self.x = synth.activations(m, n_in, seed + 7919, device) if m > 0 else \
            torch.empty((0, n_in), dtype=torch.bfloat16, device=device)
        self.wb_h = synth.as_u16(self.w_base)
        self.wf_h = synth.as_u16(self.w_ft)
        self.x_h = synth.as_u16(self.x)
        self.bits_h, self.alpha32_h, self.alpha64_h = oracle.compress(self.wb_h, self.wf_h, mode)
        self.bits = torch.from_numpy(self.bits_h).to(device)
        self.alpha = torch.from_numpy(self.alpha32_h).to(device)

    def set_m(self, m: int, seed: int) -> None:
        """Replace the activations by a fresh seeded [m, n_in] batch (same matrix)."""
        self.m = m
        self.x = synth.activations(m, self.n_in, seed, self.w_base.device)
        self.x_h = synth.as_u16(self.x)

    def run_linear(self, stream=None) -> torch.Tensor:
        y = torch.empty((self.m, self.n_out), dtype=torch.bfloat16, device=self.x.device)
        bd.bd_linear(self.x, self.w_base, self.bits, self.alpha, self.mode, y, stream)
        return y

    def reference(self):
        return oracle.linear(self.x_h, self.wb_h, self.bits_h, self.alpha32_h, self.mode)

    def reference_sampled(self, ts, js):
        return oracle.linear_sampled(self.x_h, self.wb_h, self.bits_h, self.alpha32_h, self.mode, ts, js)


def sample_outputs(m: int, n_out: int, count: int, seed: int = 0):
    """Output coordinates to check at full size: corners, tails and a seeded spread."""
    rng = np.random.default_rng(seed)
    ts = [0, m - 1, 0, m - 1, m // 2]
    js = [0, 0, n_out - 1, n_out - 1, n_out // 2]
    ts += list(rng.integers(0, m, count))
    js += list(rng.integers(0, n_out, count))
    return np.array(ts, np.int64), np.array(js, np.int64)


def with_linear_path(path: int):
    """Context manager forcing bd_linear's kernel choice (0 auto, 1 streaming, 2 tensor core, 3 register-fed streaming)."""
    class _Ctx:
        def __enter__(self):
            self.prev = bd.bd_set_linear_path(path)

        def __exit__(self, *exc):
            bd.bd_set_linear_path(self.prev)
    return _Ctx()
