"""GPU reconstruct-only pass (bd_reconstruct) against the oracle, and the
"standard matmul" reading of decode: W_eff materialised once, then an
ordinary GEMM (cuBLAS through torch), checked against the fp64 oracle and
against the fused linear.

The stored W_eff is bf16, formed in fp32 and rounded once to nearest even on
both sides, so the comparison is bit-exact."""
import numpy as np
import pytest
import torch

import oracle
from bit_delta_tenant_gb300 import bitdelta as bd
from bit_delta_tenant_gb300 import synth, workloads
from helpers import LinearCase, assert_y_close, y_host

pytestmark = pytest.mark.gpu


def reconstruct(case: LinearCase, alpha=None):
    out = torch.empty_like(case.w_base)
    bd.bd_reconstruct(case.w_base, case.bits, case.alpha if alpha is None else alpha, case.mode, out)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("n_out,n_in", [(1, 8), (7, 8), (129, 264), (300, 1024), (64, 4104), (513, 2048)])
@pytest.mark.parametrize("mode", [0, 1])
def test_reconstruct_is_bit_exact(n_out, n_in, mode):
    case = LinearCase(n_out, n_in, 0, mode=mode, seed=n_out + n_in)
    got = synth.as_u16(reconstruct(case))
    exp = oracle.w_eff_bf16(case.wb_h, case.bits_h, case.alpha32_h, mode)
    assert np.array_equal(got, exp), f"{int((got != exp).sum())} of {got.size} differ"


def test_reconstruct_alpha_zero_is_the_base():
    case = LinearCase(200, 512, 0, seed=3)
    got = reconstruct(case, alpha=torch.zeros(1, dtype=torch.float32, device="cuda"))
    assert torch.equal(got.view(torch.int16), case.w_base.view(torch.int16))


@pytest.mark.parametrize("idx", [0, 4])
def test_reconstruct_full_size_sampled_rows(idx):
    c = workloads.LLAMA7B_LAYER
    name, n_out, n_in = c["matrices"][idx]
    case = LinearCase(n_out, n_in, 0, c["sigma"], c["b"], c["mode"], workloads.matrix_seed(c["seed"], idx))
    got = synth.as_u16(reconstruct(case))
    rows = np.unique(np.concatenate([[0, n_out - 1], np.random.default_rng(idx).integers(0, n_out, 200)]))
    exp = oracle.w_eff_bf16(case.wb_h[rows], case.bits_h[rows], case.alpha32_h, case.mode)
    assert np.array_equal(got[rows], exp), name


@pytest.mark.parametrize("m", [1, 16, 300])
def test_standard_matmul_over_reconstructed_weight(m):
    """The page's decode reading: rebuild once, then a standard matmul.  Both it
    and the fused linear meet the same tolerance against the fp64 oracle."""
    case = LinearCase(384, 1024, m, mode=1, seed=40 + m)
    w_eff = reconstruct(case)
    y_std = (case.x.float() @ w_eff.float().t()).to(torch.bfloat16)
    y_fused = case.run_linear()
    torch.cuda.synchronize()
    y_ref, mag = case.reference()
    assert_y_close(y_host(y_std), y_ref, mag, f"reconstruct + matmul m={m}")
    assert_y_close(y_host(y_fused), y_ref, mag, f"fused m={m}")
