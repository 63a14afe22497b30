"""GPU fused linear (bd_linear) against the fp64 oracle, through the C ABI.

Both kernels are exercised: the HBM-streaming one (forced path 1, m <= 64) and
the tcgen05 tensor-core one (forced path 2, any m), plus the automatic choice.
Small cases compare every output; the full workload sizes compare sampled
outputs that the oracle computes one by one."""
import numpy as np
import pytest
import torch

from bit_delta_tenant_gb300 import bitdelta as bd
from bit_delta_tenant_gb300 import synth, workloads
from helpers import LinearCase, assert_y_close, sample_outputs, with_linear_path, y_host

pytestmark = pytest.mark.gpu

AUTO, STREAM, TENSOR, STREAM_REG = 0, 1, 2, 3


def full_check(case: LinearCase, path: int, what: str):
    with with_linear_path(path):
        y = case.run_linear()
    torch.cuda.synchronize()
    assert bd.bd_get_device_status() == bd.BD_OK
    y_ref, mag = case.reference()
    assert_y_close(y_host(y), y_ref, mag, what)


def sampled_check(case: LinearCase, path: int, count: int, what: str):
    with with_linear_path(path):
        y = case.run_linear()
    torch.cuda.synchronize()
    assert bd.bd_get_device_status() == bd.BD_OK
    yh = y_host(y)
    assert np.all(np.isfinite(yh)), f"{what}: non-finite output"
    ts, js = sample_outputs(case.m, case.n_out, count, seed=case.m + case.n_out)
    y_ref, mag = case.reference_sampled(ts, js)
    assert_y_close(yh[ts, js], y_ref, mag, what)


@pytest.mark.parametrize("path", [AUTO, STREAM, TENSOR])
def test_tiny_workload(path):
    c = workloads.TINY
    case = LinearCase(c["n_out"], c["n_in"], c["m"], c["sigma"], c["b"], c["mode"], c["seed"])
    full_check(case, path, f"tiny path={path}")


STREAM_SHAPES = [  # (n_out, n_in, m): ragged K (not multiples of 128), odd rows, every token-tile count
    (1, 8, 1), (7, 16, 2), (129, 24, 3), (128, 120, 15), (33, 136, 16), (200, 4096, 17), (64, 1000, 33),
    (130, 520, 64), (256, 4096, 8), (1, 11008, 4), (300, 264, 40),
]
TMA_STREAM_SHAPES = [  # n_in multiples of 128 (TMA-fed variant): ragged rows, slices, tokens
    (64, 128, 1), (65, 256, 9), (300, 384, 33), (129, 1152, 64), (7, 2048, 16), (1000, 8192, 2),
    (4096, 4096, 16), (63, 16384, 5), (2000, 640, 24),
]


@pytest.mark.parametrize("n_out,n_in,m", STREAM_SHAPES + TMA_STREAM_SHAPES)
@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("path", [STREAM, STREAM_REG])
def test_streaming_kernel_shapes(n_out, n_in, m, mode, path):
    case = LinearCase(n_out, n_in, m, 0.02, "row:5e-4:2e-3" if mode else 1e-3, mode, seed=n_out + 7 * n_in + m)
    full_check(case, path, f"stream path={path} {n_out}x{n_in} m={m}")


TENSOR_SHAPES = [  # ragged in every dimension: rows vs 128/256, tokens vs 256, K vs 64
    (128, 64, 256), (129, 64, 1), (7, 8, 5), (128, 72, 257), (300, 136, 100), (256, 1024, 511),
    (200, 520, 512), (384, 4096, 513), (129, 24, 65), (64, 4104, 300), (257, 640, 9), (513, 192, 16),
    (1000, 2048, 263), (520, 4096, 1024),
]
# the tensor-core kernels: one CTA per 128 x 256 tile, and CTA pairs on 256 x 256 tiles
# (BD_OPT_PREFILL_KERNEL, BD_OPT_PAIR_RING): single-CTA tiles, and the CTA-pair kernel in both of
# its shapes (5-deep ring with the whole output tile staged, 6-deep with two staged halves)
PREFILL_KERNELS = {"single": (1, 0), "pair5": (2, 1), "pair6": (2, 2)}


@pytest.fixture(params=list(PREFILL_KERNELS))
def prefill_kernel(request):
    kernel, ring = PREFILL_KERNELS[request.param]
    with bd.option(bd.BD_OPT_PREFILL_KERNEL, kernel), bd.option(bd.BD_OPT_PAIR_RING, ring):
        yield request.param


@pytest.mark.parametrize("n_out,n_in,m", TENSOR_SHAPES)
@pytest.mark.parametrize("mode", [0, 1])
def test_tensor_core_kernel_shapes(n_out, n_in, m, mode, prefill_kernel):
    case = LinearCase(n_out, n_in, m, 0.02, "row:5e-4:2e-3" if mode else 1e-3, mode, seed=3 * n_out + n_in + m)
    full_check(case, TENSOR, f"tcgen05 {prefill_kernel} {n_out}x{n_in} m={m}")


@pytest.mark.parametrize("ring", [1, 2])
@pytest.mark.parametrize("n_out,n_in,m", [(8192, 72, 4096), (2000, 200, 3000), (4096, 8, 2048), (700, 1000, 5000)])
def test_pair_kernel_many_tiles_per_pair(n_out, n_in, m, ring):
    """The persistent pair kernel: several tiles per pair (up to ~7 here on 76 pairs), tiles of 1, 2,
    4 or 16 K blocks so that tile boundaries fall at every position of the K-block ring, ragged W
    rows and token tiles, both kernel shapes."""
    case = LinearCase(n_out, n_in, m, 0.02, "row:5e-4:2e-3" if ring == 2 else 1e-3, ring - 1, seed=n_out + m)
    with bd.option(bd.BD_OPT_PREFILL_KERNEL, 2), bd.option(bd.BD_OPT_PAIR_RING, ring):
        full_check(case, TENSOR, f"pair ring {ring} {n_out}x{n_in} m={m}")


@pytest.mark.parametrize("n_out,n_in,m,mode", [(3000, 1000, 2500, 1), (8192, 640, 1300, 0), (700, 8200, 600, 0)])
def test_pair_kernel_shapes_give_identical_bits(n_out, n_in, m, mode):
    """The pair kernel's two shapes differ only in ring depth and in how the output tile is staged,
    not in the arithmetic or its order: their outputs are bit-identical (and match the oracle)."""
    case = LinearCase(n_out, n_in, m, 0.02, "row:5e-4:2e-3" if mode else 1e-3, mode, seed=n_out + 3 * m)
    ys = []
    for ring in (1, 2):
        with bd.option(bd.BD_OPT_PREFILL_KERNEL, 2), bd.option(bd.BD_OPT_PAIR_RING, ring):
            ys.append(case.run_linear())
    torch.cuda.synchronize()
    assert bd.bd_get_device_status() == bd.BD_OK
    assert torch.equal(ys[0], ys[1]), "the 5-deep and 6-deep shapes differ"
    ts, js = sample_outputs(m, n_out, 600, seed=m)
    y_ref, mag = case.reference_sampled(ts, js)
    assert_y_close(y_host(ys[0])[ts, js], y_ref, mag, f"pair shapes {n_out}x{n_in} m={m}")


@pytest.mark.parametrize("ring", [1, 2])
@pytest.mark.parametrize("m", [1, 8, 9, 16, 17, 120, 128, 129, 255, 256])
def test_pair_kernel_last_token_tile_split(m, ring):
    """The pair's MMA N is the tile's token count rounded to 16, each CTA holding half of it:
    a last tile of few tokens leaves the odd CTA's half partly or wholly past the end."""
    case = LinearCase(300, 512, 256 + m, seed=40 + m)
    with bd.option(bd.BD_OPT_PREFILL_KERNEL, 2), bd.option(bd.BD_OPT_PAIR_RING, ring):
        full_check(case, TENSOR, f"pair ring {ring} m={256 + m}")


@pytest.mark.parametrize("path", [STREAM, STREAM_REG, TENSOR])
def test_alpha_zero_is_plain_base_linear(path, prefill_kernel):
    case = LinearCase(96, 256, 16, seed=11)
    case.alpha.zero_()
    case.alpha32_h[:] = 0
    full_check(case, path, "alpha=0")


@pytest.mark.parametrize("path", [STREAM, STREAM_REG, TENSOR])
@pytest.mark.parametrize("n_in", [32, 128])
def test_zero_base_unit_alpha_is_exact_sign_product(path, n_in, prefill_kernel):
    """W_base = 0, alpha = 1, integer x: y = x . S^T exactly (|y| <= 2*n_in fits bf16 exactly here)."""
    rng = np.random.default_rng(3)
    n_out, m = 64, 8
    s = rng.choice(np.array([-1, 1]), size=(n_out, n_in))
    xi = rng.integers(-2, 3, size=(m, n_in))
    case = LinearCase(n_out, n_in, m, seed=1)
    case.w_base.zero_()
    case.wb_h[:] = 0
    case.bits_h[:] = np.packbits(s > 0, axis=1, bitorder="little")
    case.bits.copy_(torch.from_numpy(case.bits_h))
    case.alpha.fill_(1.0)
    case.alpha32_h[:] = 1.0
    case.x.copy_(torch.from_numpy(xi.astype(np.float32)).to(torch.bfloat16))
    case.x_h = synth.as_u16(case.x)
    with with_linear_path(path):
        y = case.run_linear()
    torch.cuda.synchronize()
    assert np.array_equal(y_host(y), (xi @ s.T).astype(np.float64))


def test_empty_batch_is_a_no_op():
    case = LinearCase(64, 128, 0, seed=2)
    y = case.run_linear()
    assert y.shape == (0, 64)


@pytest.mark.parametrize("idx", range(len(workloads.LLAMA7B_LAYER["matrices"])))
def test_llama7b_layer_decode_full_size(idx):
    c = workloads.LLAMA7B_LAYER
    name, n_out, n_in = c["matrices"][idx]
    case = LinearCase(n_out, n_in, 1, c["sigma"], c["b"], c["mode"], workloads.matrix_seed(c["seed"], idx))
    for m in c["ms"]:
        case.set_m(m, seed=1000 + m)
        sampled_check(case, AUTO, 1500, f"{name} m={m}")


@pytest.mark.parametrize("idx", range(len(workloads.LLAMA70B_PREFILL["matrices"])))
def test_llama70b_prefill_full_size(idx):
    c = workloads.LLAMA70B_PREFILL
    name, n_out, n_in = c["matrices"][idx]
    case = LinearCase(n_out, n_in, 1, c["sigma"], c["b"], c["mode"], workloads.matrix_seed(c["seed"], idx))
    for m in c["ms"]:
        case.set_m(m, seed=2000 + m)
        sampled_check(case, AUTO, 1500, f"{name} m={m}")
    del case
    torch.cuda.empty_cache()


# the distinct matrix shapes of the Llama-3-8B-shape stack (k and v share one, gate and up another)
STACK_SHAPES = sorted({(n, a, b) for (n, a, b) in workloads.LLAMA3_8B_STACK["matrices"] if n in ("q", "k", "gate", "down")})


@pytest.mark.parametrize("idx", range(len(STACK_SHAPES)))
def test_llama3_8b_stack_shapes_full_size(idx):
    c = workloads.LLAMA3_8B_STACK
    name, n_out, n_in = STACK_SHAPES[idx]
    case = LinearCase(n_out, n_in, 1, c["sigma"], c["b"], c["mode"], workloads.matrix_seed(c["seed"], idx))
    for m in c["ms"]:
        case.set_m(m, seed=3000 + m)
        sampled_check(case, AUTO, 1500, f"{name} m={m}")
    del case
    torch.cuda.empty_cache()


def test_both_kernels_agree_with_oracle_at_the_dispatch_boundary():
    for m in (63, 64, 65):
        case = LinearCase(512, 2048, m, seed=m)
        y_ref, mag = case.reference()
        for path in (STREAM, STREAM_REG, TENSOR) if m <= 64 else (TENSOR,):
            with with_linear_path(path):
                y = case.run_linear()
            torch.cuda.synchronize()
            assert_y_close(y_host(y), y_ref, mag, f"m={m} path={path}")


def test_repeated_calls_on_a_side_stream():
    case = LinearCase(256, 1024, 300, seed=4)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        y1 = case.run_linear(s)
        y2 = case.run_linear(s)
    s.synchronize()
    assert torch.equal(y1, y2)
    y_ref, mag = case.reference()
    assert_y_close(y_host(y1), y_ref, mag, "side stream")


def test_wait_limit_zero_reports_timeout_and_context_survives(prefill_kernel):
    """A zero wait limit makes the tensor-core kernel give up at its first
    unsatisfied wait: it records a timeout, drains its own copies and returns.
    The context stays usable and a normal call afterwards is correct."""
    case = LinearCase(256, 4096, 512, seed=9)
    assert bd.bd_get_device_status() == bd.BD_OK
    prev = bd.bd_set_wait_limit_ns(0)
    try:
        with with_linear_path(TENSOR):
            case.run_linear()
        status = bd.bd_get_device_status()
    finally:
        bd.bd_set_wait_limit_ns(prev)
    assert status == bd.BD_ERR_DEVICE_TIMEOUT
    assert bd.bd_get_device_status() == bd.BD_OK      # read-and-clear
    with with_linear_path(TENSOR):
        y = case.run_linear()
    torch.cuda.synchronize()
    assert bd.bd_get_device_status() == bd.BD_OK
    y_ref, mag = case.reference()
    assert_y_close(y_host(y), y_ref, mag, "after timeout")


def with_weight_prefetch(enable: int):
    class _Ctx:
        def __enter__(self):
            self.prev = bd.bd_set_weight_prefetch(enable)

        def __exit__(self, *exc):
            bd.bd_set_weight_prefetch(self.prev)
    return _Ctx()


@pytest.mark.parametrize("m", [1, 16, 64])
def test_weight_prefetch_chain_in_a_graph(m):
    """Back-to-back streaming linears captured in a CUDA graph with weight
    prefetch on: each kernel may read its weights while the previous one
    drains, but its activations only after that kernel completes.  The chain
    feeds y of the first linear into the second (a read-after-write through x),
    so a stale read would show up in the second output."""
    a = LinearCase(384, 1024, m, seed=21)
    b = LinearCase(640, 384, 0, seed=22)
    c = LinearCase(512, 2048, m, seed=23)
    s = torch.cuda.Stream()

    def chain(prefetch):
        y1 = torch.full((m, 384), float("nan"), dtype=torch.bfloat16, device="cuda")
        y2 = torch.full((m, 640), float("nan"), dtype=torch.bfloat16, device="cuda")
        y3 = torch.full((m, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
        torch.cuda.synchronize()
        with with_linear_path(STREAM), with_weight_prefetch(prefetch):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                bd.bd_linear(a.x, a.w_base, a.bits, a.alpha, 0, y1, s)
                bd.bd_linear(y1, b.w_base, b.bits, b.alpha, 0, y2, s)
                bd.bd_linear(c.x, c.w_base, c.bits, c.alpha, 0, y3, s)
        g.replay()
        torch.cuda.synchronize()
        assert bd.bd_get_device_status() == bd.BD_OK
        return y1, y2, y3

    p1, p2, p3 = chain(1)
    q1, q2, q3 = chain(0)
    for y, case in ((p1, a), (p3, c)):
        y_ref, mag = case.reference()
        assert_y_close(y_host(y), y_ref, mag, f"prefetch m={m}")
    # the same kernels in the same order: identical bits with and without prefetch
    assert torch.equal(p1, q1) and torch.equal(p3, q3)
    assert torch.equal(p2, q2), "the dependent linear read its activations before they were written"
