"""bd_compress_noalloc: compression for callers that cannot allocate device memory.

Some callers can hand the library their inputs and outputs but no workspace --
a framework that owns all device memory through a pre-planned arena, or a
latency-critical path that must not call cudaMalloc.  bd_compress_noalloc
serves them from a fixed scratch array inside the library.  These tests call it
through the C ABI and check that two calls in a row give the same bits and
alpha as bd_compress with a caller-provided workspace (bits bit-exact, alpha
within the suite's 1e-6 relative tolerance).  The file name sorts last so a
run that stops at the first failure has run every other test already; it also
passes on its own in a fresh process (the first call sets the scratch up).
"""
import numpy as np
import pytest
import torch

from bit_delta_tenant_gb300 import bitdelta as bd
from bit_delta_tenant_gb300 import synth
from helpers import ALPHA_REL

pytestmark = pytest.mark.gpu


def _with_workspace(w_base, w_ft, mode):
    n_out, n_in = w_base.shape
    bits = torch.empty((n_out, n_in // 8), dtype=torch.uint8, device="cuda")
    alpha = torch.empty((n_out if mode else 1,), dtype=torch.float32, device="cuda")
    ws = torch.empty((bd.bd_compress_workspace_size(n_out, n_in, mode),), dtype=torch.uint8, device="cuda")
    bd.bd_compress(w_base, w_ft, mode, bits, alpha, ws)
    return bits, alpha


def _no_alloc(w_base, w_ft, mode):
    n_out, n_in = w_base.shape
    bits = torch.empty((n_out, n_in // 8), dtype=torch.uint8, device="cuda")
    alpha = torch.empty((n_out if mode else 1,), dtype=torch.float32, device="cuda")
    bd.bd_compress_noalloc(w_base, w_ft, mode, bits, alpha)
    return bits, alpha


def _same(got, ref):
    (gb, ga), (rb, ra) = got, ref
    assert torch.equal(gb, rb), "packed bits differ from bd_compress"
    g = ga.double().cpu().numpy()
    r = ra.double().cpu().numpy()
    assert np.all(np.abs(g - r) <= ALPHA_REL * np.abs(r)), "alpha differs from bd_compress"


@pytest.mark.parametrize("mode", [0, 1])
def test_two_calls_in_a_row_match_bd_compress(mode):
    # A large shape first, then a smaller one: the second call must not be
    # affected by what the first left in the shared scratch.  Both split their
    # rows into several segments in either mode (n_in > 8192), so the second
    # call reads partial-sum slots that the first one wrote.
    a = synth.matrix_pair(4096, 11008, 0.02, 1e-3, seed=101, device="cuda")
    b = synth.matrix_pair(300, 8320, 0.02, "row:5e-4:2e-3", seed=102, device="cuda")
    first = _no_alloc(*a, mode)
    second = _no_alloc(*b, mode)
    torch.cuda.synchronize()
    assert bd.bd_get_device_status() == bd.BD_OK
    _same(first, _with_workspace(*a, mode))
    _same(second, _with_workspace(*b, mode))


def test_repeated_call_on_same_input_is_identical():
    a = synth.matrix_pair(2048, 4096, 0.015, 1e-3, seed=103, device="cuda")
    r1 = _no_alloc(*a, 0)
    r2 = _no_alloc(*a, 0)
    torch.cuda.synchronize()
    assert torch.equal(r1[0], r2[0]) and torch.equal(r1[1].view(torch.int32), r2[1].view(torch.int32))
    _same(r1, _with_workspace(*a, 0))


def test_shape_beyond_the_built_in_scratch_is_rejected():
    # per-row alpha with 65537 rows of 8200 inputs (1025 chunks: two segments per row) needs
    # 131074 partial sums > BD_NOALLOC_MAX_PARTIALS; rejected on the host before any launch,
    # so these fake pointers are never touched.
    lib = bd.load_library()
    rows = bd.BD_NOALLOC_MAX_PARTIALS // 2 + 1
    rc = lib.bd_compress_noalloc(0x10000, 0x10000, rows, 8200, 1, 0x10000, 0x10000, None)
    assert rc == bd.BD_ERR_WORKSPACE
