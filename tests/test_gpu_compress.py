"""GPU compression (bd_compress) against the fp64 oracle: packed bits bit-exact,
alpha within 1e-6 relative, bitwise-reproducible alpha, on the workload shapes
and on ragged shapes."""
import os

import numpy as np
import pytest
import torch

import oracle
from bit_delta_tenant_gb300 import bitdelta as bd
from bit_delta_tenant_gb300 import synth, workloads
from helpers import ALPHA_REL

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def gpu_compress(w_base, w_ft, mode):
    n_out, n_in = w_base.shape
    bits = torch.empty((n_out, n_in // 8), dtype=torch.uint8, device=w_base.device)
    alpha = torch.empty((n_out if mode == 1 else 1,), dtype=torch.float32, device=w_base.device)
    ws = torch.empty((max(1, bd.bd_compress_workspace_size(n_out, n_in, mode)),), dtype=torch.uint8,
                     device=w_base.device)
    bd.bd_compress(w_base, w_ft, mode, bits, alpha, ws)
    torch.cuda.synchronize()
    return bits, alpha


def check_against_oracle(w_base, w_ft, mode):
    bits, alpha = gpu_compress(w_base, w_ft, mode)
    wb, wf = synth.as_u16(w_base), synth.as_u16(w_ft)
    ref_bits = oracle.sign_bits(wb, wf)
    got = bits.cpu().numpy()
    if not np.array_equal(got, ref_bits):
        bad = np.argwhere(got != ref_bits)
        raise AssertionError(f"{len(bad)} packed bytes differ; first at {tuple(bad[0])}")
    a64 = oracle.alpha(wb, wf, mode)
    a32 = alpha.cpu().numpy().astype(np.float64)
    rel = np.abs(a32 - a64) / np.abs(a64)
    assert rel.max() <= ALPHA_REL, f"alpha relative error {rel.max():.3e}"
    return bits, alpha


def _read_cases():
    with open(os.path.join(GOLDEN, "sign_bytes.txt"), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield [p.strip() for p in line.split(";")]


@pytest.mark.parametrize("case", list(_read_cases()), ids=lambda c: c[0])
def test_hand_worked_bytes_on_gpu(case):
    """The page-derived golden bytes, straight through the GPU kernel."""
    _, rows, cols, wb, wf, expect = case
    rows, cols = int(rows), int(cols)
    wb = np.array([int(h, 16) for h in wb.split(",")], np.uint16).reshape(rows, cols)
    wf = np.array([int(h, 16) for h in wf.split(",")], np.uint16).reshape(rows, cols)
    expect = np.array([int(h, 16) for h in expect.split(",")], np.uint8).reshape(rows, cols // 8)
    bits, _ = gpu_compress(synth.from_u16(wb, "cuda"), synth.from_u16(wf, "cuda"), 0)
    assert np.array_equal(bits.cpu().numpy(), expect)


@pytest.fixture(params=["direct", "ring"])
def compress_form(request):
    """Both forms of pass 1 (the default direct one, and the persistent ring one)."""
    with bd.option(bd.BD_OPT_COMPRESS_FORM, 1 if request.param == "ring" else 0):
        yield request.param


@pytest.mark.parametrize("n_out,n_in", [(1, 8), (7, 24), (33, 120), (129, 136), (128, 4096), (3, 16392)])
@pytest.mark.parametrize("mode", [0, 1])
def test_ragged_shapes(n_out, n_in, mode, compress_form):
    w_base, w_ft = synth.matrix_pair(n_out, n_in, 0.02, 1e-3, seed=n_out * 31 + n_in, device="cuda")
    check_against_oracle(w_base, w_ft, mode)


def test_tiny_workload():
    c = workloads.TINY
    w_base, w_ft = synth.matrix_pair(c["n_out"], c["n_in"], c["sigma"], c["b"], c["seed"], "cuda")
    check_against_oracle(w_base, w_ft, c["mode"])


@pytest.mark.parametrize("idx", range(len(workloads.LLAMA7B_LAYER["matrices"])))
def test_llama7b_layer_matrices(idx):
    c = workloads.LLAMA7B_LAYER
    _, n_out, n_in = c["matrices"][idx]
    w_base, w_ft = synth.matrix_pair(n_out, n_in, c["sigma"], c["b"], workloads.matrix_seed(c["seed"], idx), "cuda")
    check_against_oracle(w_base, w_ft, c["mode"])


@pytest.mark.parametrize("idx", range(len(workloads.LLAMA70B_PREFILL["matrices"])))
def test_llama70b_matrices_per_row_alpha(idx):
    c = workloads.LLAMA70B_PREFILL
    _, n_out, n_in = c["matrices"][idx]
    w_base, w_ft = synth.matrix_pair(n_out, n_in, c["sigma"], c["b"], workloads.matrix_seed(c["seed"], idx), "cuda")
    check_against_oracle(w_base, w_ft, c["mode"])
    # the same matrix with a scalar alpha as well
    check_against_oracle(w_base, w_ft, 0)


@pytest.mark.parametrize("mode", [0, 1])
def test_alpha_is_bitwise_reproducible(mode):
    w_base, w_ft = synth.matrix_pair(4096, 11008, 0.02, 1e-3, seed=5, device="cuda")
    b1, a1 = gpu_compress(w_base, w_ft, mode)
    b2, a2 = gpu_compress(w_base, w_ft, mode)
    assert torch.equal(b1, b2)
    assert torch.equal(a1.view(torch.int32), a2.view(torch.int32))


@pytest.mark.parametrize("mode", [0, 1])
def test_direct_and_ring_forms_agree_bitwise(mode):
    """The two forms of pass 1 take the same summation tree, so their alpha agree to the bit."""
    w_base, w_ft = synth.matrix_pair(2048, 11008, 0.02, 1e-3, seed=8, device="cuda")
    with bd.option(bd.BD_OPT_COMPRESS_FORM, 0):
        b1, a1 = gpu_compress(w_base, w_ft, mode)
    with bd.option(bd.BD_OPT_COMPRESS_FORM, 1):
        b2, a2 = gpu_compress(w_base, w_ft, mode)
    assert torch.equal(b1, b2)
    assert torch.equal(a1.view(torch.int32), a2.view(torch.int32))


def test_zero_delta_packs_all_ones_and_alpha_zero():
    w_base = synth.bf16_normal((64, 256), 0.02, synth.generator(1, "cuda"), "cuda")
    bits, alpha = gpu_compress(w_base, w_base.clone(), 1)
    assert torch.all(bits == 255)
    assert torch.all(alpha == 0)


def gpu_compress_batch(mats):
    """bd_compress_batch over [(w_base, w_ft, mode)]; returns [(bits, alpha)]."""
    outs, probs = [], []
    for w_base, w_ft, mode in mats:
        n_out, n_in = w_base.shape
        bits = torch.full((n_out, n_in // 8), 0xAA, dtype=torch.uint8, device=w_base.device)
        alpha = torch.full((n_out if mode == 1 else 1,), float("nan"), dtype=torch.float32, device=w_base.device)
        outs.append((bits, alpha))
        probs.append((w_base, w_ft, mode, bits, alpha))
    descs = bd.compress_descs(probs)
    ws = torch.empty((max(1, bd.bd_compress_batch_workspace_size(descs)),), dtype=torch.uint8, device="cuda")
    bd.bd_compress_batch(descs, ws)
    torch.cuda.synchronize()
    return outs


BATCH_SHAPES = [  # scalar (many segments: block pass 2), per-row one segment, per-row 2..32 segments, ragged
    (256, 512, 0), (33, 120, 1), (3, 16392, 1), (129, 136, 0), (1000, 8192, 1), (7, 24, 0), (64, 65536, 1),
    (300, 4096, 0), (1, 8, 1), (2048, 11008, 0),
]


@pytest.mark.parametrize("count", [1, 3, 8, 10])
def test_batched_compression_equals_single_calls_and_oracle(count):
    """Every matrix of a batch gets the bits and alpha of its own bd_compress call (bitwise), and the
    oracle's bits and alpha; 10 matrices take two launches of each pass."""
    mats = []
    for i, (n_out, n_in, mode) in enumerate(BATCH_SHAPES[:count]):
        w_base, w_ft = synth.matrix_pair(n_out, n_in, 0.02, 1e-3, seed=40 + i, device="cuda")
        mats.append((w_base, w_ft, mode))
    outs = gpu_compress_batch(mats)
    for i, ((w_base, w_ft, mode), (bits, alpha)) in enumerate(zip(mats, outs)):
        b1, a1 = check_against_oracle(w_base, w_ft, mode)
        assert torch.equal(bits, b1), f"matrix {i}: bits differ from bd_compress"
        assert torch.equal(alpha.view(torch.int32), a1.view(torch.int32)), f"matrix {i}: alpha differs"


def test_batched_compression_of_the_llama7b_layer():
    c = workloads.LLAMA7B_LAYER
    mats = []
    for i, (_, n_out, n_in) in enumerate(c["matrices"]):
        w_base, w_ft = synth.matrix_pair(n_out, n_in, c["sigma"], c["b"], workloads.matrix_seed(c["seed"], i), "cuda")
        mats.append((w_base, w_ft, c["mode"]))
    outs = gpu_compress_batch(mats)
    for (w_base, w_ft, mode), (bits, alpha) in zip(mats, outs):
        b1, a1 = gpu_compress(w_base, w_ft, mode)
        assert torch.equal(bits, b1)
        assert torch.equal(alpha.view(torch.int32), a1.view(torch.int32))
        wb, wf = synth.as_u16(w_base), synth.as_u16(w_ft)
        a64 = oracle.alpha(wb, wf, mode)
        assert abs(float(alpha[0]) - a64[0]) / abs(a64[0]) <= ALPHA_REL


def test_batched_compression_workspace_errors():
    w_base, w_ft = synth.matrix_pair(64, 8192, 0.02, 1e-3, seed=3, device="cuda")
    bits = torch.empty((64, 1024), dtype=torch.uint8, device="cuda")
    alpha = torch.empty((1,), dtype=torch.float32, device="cuda")
    descs = bd.compress_descs([(w_base, w_ft, 0, bits, alpha)])
    need = bd.bd_compress_batch_workspace_size(descs)
    assert need == (bd.bd_compress_workspace_size(64, 8192, 0) + 255) // 256 * 256
    with pytest.raises(bd.BitDeltaError) as e:
        bd.bd_compress_batch(descs, torch.empty(need - 256, dtype=torch.uint8, device="cuda"))
    assert e.value.status == bd.BD_ERR_WORKSPACE
    assert bd.bd_compress_batch_workspace_size((bd.CompressDesc * 0)()) == 0


def test_batched_compression_of_the_llama3_8b_stack_shapes():
    """One layer of the Llama-3-8B-shape stack (q, k, v, o, gate, up, down) in one batched call."""
    c = workloads.LLAMA3_8B_STACK
    mats = []
    for i, (_, n_out, n_in) in enumerate(c["matrices"]):
        w_base, w_ft = synth.matrix_pair(n_out, n_in, c["sigma"], c["b"], workloads.matrix_seed(c["seed"], i), "cuda")
        mats.append((w_base, w_ft, c["mode"]))
    outs = gpu_compress_batch(mats)
    for (w_base, w_ft, mode), (bits, alpha) in zip(mats, outs):
        wb, wf = synth.as_u16(w_base), synth.as_u16(w_ft)
        assert np.array_equal(bits.cpu().numpy(), oracle.sign_bits(wb, wf))
        a64 = oracle.alpha(wb, wf, mode)
        assert abs(float(alpha[0]) - a64[0]) / abs(a64[0]) <= ALPHA_REL


def test_stalled_wait_ring_form_reports_timeout_and_context_survives():
    """The persistent ring form of pass 1, its consumers made to wait first on a barrier that
    nothing completes (BD_OPT_TEST_STALL) under a 1 ms wait limit, gives up: it records a
    timeout, its producer drains the copies it issued, and the next call is correct.  (A zero
    wait limit alone does not force this: the hardware's suspended try-wait outlasts the
    copy of one ring slot.)"""
    w_base, w_ft = synth.matrix_pair(2048, 8192, 0.02, 1e-3, seed=61, device="cuda")
    assert bd.bd_get_device_status() == bd.BD_OK
    with bd.option(bd.BD_OPT_COMPRESS_FORM, 1):
        prev = bd.bd_set_wait_limit_ns(1_000_000)
        try:
            with bd.option(bd.BD_OPT_TEST_STALL, 1):
                gpu_compress(w_base, w_ft, 0)
            status = bd.bd_get_device_status()
        finally:
            bd.bd_set_wait_limit_ns(prev)
        assert status == bd.BD_ERR_DEVICE_TIMEOUT
        assert bd.bd_get_device_status() == bd.BD_OK
        check_against_oracle(w_base, w_ft, 0)
