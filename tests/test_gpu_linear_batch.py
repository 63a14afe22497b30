"""GPU batched fused linear (bd_linear_batch) against the fp64 oracle, through the C ABI.

Each problem of a batch must match the oracle's fused linear on the same seeded
inputs; small problems compare every output, full-size ones sampled outputs.
Both kernels a launch can run are exercised, by the library's choice and forced:
the cluster-split one (64-row CTAs, K split over a cluster, partials pushed to the
owning CTA) and the evenly split one (one 128-column K step of one 64-row block per
work item, split evenly over the CTAs), the latter also with forced grids that make
row blocks shared by many CTAs or by none."""
import os

import pytest
import torch

import oracle
from bit_delta_tenant_gb300 import bitdelta as bd
from bit_delta_tenant_gb300 import synth, workloads
from helpers import LinearCase, assert_y_close, sample_outputs, y_host

pytestmark = pytest.mark.gpu


def make_cases(shapes, seed0=0, mode=0):
    return [LinearCase(n_out, n_in, m, sigma=0.02, b=1e-3, mode=mode, seed=seed0 + i)
            for i, (n_out, n_in, m) in enumerate(shapes)]


def run_batch(cases, workspace=None, stream=None, fill=float("nan")):
    ys = [torch.full((c.m, c.n_out), fill, dtype=torch.bfloat16, device="cuda") for c in cases]
    descs = bd.linear_descs([(c.x, c.w_base, c.bits, c.alpha, c.mode, y) for c, y in zip(cases, ys)])
    need = bd.bd_linear_batch_workspace_size(descs)
    if workspace is None:
        workspace = torch.zeros(max(need, 1), dtype=torch.uint8, device="cuda")
    assert workspace.numel() >= need
    bd.bd_linear_batch(descs, workspace, stream)
    return ys, workspace


def assert_reusable(cases, ys, ws, what):
    """A second call on the same workspace (its counters must be back at zero) gives identical bits."""
    ys2, _ = run_batch(cases, workspace=ws)
    torch.cuda.synchronize()
    assert bd.bd_get_device_status() == bd.BD_OK
    for i, (a, b) in enumerate(zip(ys, ys2)):
        assert torch.equal(a, b), f"{what}: problem {i} differs on a reused workspace"


def check_all(cases, ys, what):
    torch.cuda.synchronize()
    assert bd.bd_get_device_status() == bd.BD_OK
    for i, (c, y) in enumerate(zip(cases, ys)):
        y_ref, mag = c.reference()
        assert_y_close(y_host(y), y_ref, mag, f"{what} problem {i} ({c.n_out}x{c.n_in}, m={c.m})")


KERNELS = ["auto", "cluster", "streamk"]


BATCH_KERNEL_VALUE = {"auto": 0, "cluster": 1, "streamk": 2}


@pytest.fixture(params=KERNELS)
def batch_kernel(request):
    """The kernel a launch of the batch runs: the library's choice (the cluster-split kernel when
    its CTAs fit in one wave, else the evenly split one) or either one forced (BD_OPT_BATCH_KERNEL)."""
    with bd.option(bd.BD_OPT_BATCH_KERNEL, BATCH_KERNEL_VALUE[request.param]):
        yield request.param


def grid_override(grid):
    """Forces the number of CTAs of the batched kernel (BD_OPT_BATCH_GRID)."""
    return bd.option(bd.BD_OPT_BATCH_GRID, grid)


BATCHES = {  # ragged rows (not multiples of 64), several K lengths, both token tiles
    "qkv_like": [(256, 512, 1), (256, 512, 1), (256, 512, 1)],
    "ragged": [(200, 384, 3), (65, 1152, 8), (1, 128, 5), (1000, 640, 2)],
    "two_tiles": [(300, 768, 16), (129, 256, 9), (64, 2048, 12)],
    "mixed_tiles": [(96, 1024, 1), (96, 1024, 16), (333, 384, 4), (70, 896, 11)],
    # m <= 8 with 64-row blocks between one and two per SM: taller CTAs (80 / 96 rows on 152 SMs)
    # split in two along K, last blocks partial
    "tall_ctas_r5": [(4000, 512, 2), (4000, 384, 5), (2000, 256, 1)],
    "tall_ctas_r6": [(4000, 512, 1), (4000, 512, 3), (4000, 640, 8), (200, 256, 6)],
}


@pytest.mark.parametrize("name", list(BATCHES))
@pytest.mark.parametrize("mode", [0, 1])
def test_batches_match_oracle(name, mode, batch_kernel):
    cases = make_cases(BATCHES[name], seed0=100, mode=mode)
    ys, ws = run_batch(cases)
    check_all(cases, ys, f"{name} mode={mode}")
    assert_reusable(cases, ys, ws, name)


@pytest.mark.parametrize("grid", [1, 2, 3, 7, 50, 1000, 100000])
def test_forced_grids(grid):
    """Few CTAs (every block in one CTA's range, several linears per CTA) to far
    more CTAs than items (capped at one item per CTA: every block split K-step by K-step)."""
    cases = make_cases([(200, 1280, 3), (64, 384, 8), (130, 2048, 1)], seed0=300, mode=1)
    with bd.option(bd.BD_OPT_BATCH_KERNEL, 2):
        with grid_override(grid):
            ys, ws = run_batch(cases)
        check_all(cases, ys, f"grid={grid}")
        with grid_override(grid):
            assert_reusable(cases, ys, ws, f"grid={grid}")


@pytest.mark.parametrize("shape", [(200, 1280, 3), (4096, 4096, 16), (65, 128, 1), (1000, 8192, 9)])
def test_single_linear_launch(shape):
    """A batch of one runs as bd_linear unless BD_OPT_BATCH_SINGLE keeps it on the batched kernel."""
    cases = make_cases([shape], seed0=350, mode=1)
    with bd.option(bd.BD_OPT_BATCH_SINGLE, 1):
        ys, ws = run_batch(cases)
        check_all(cases, ys, f"single {shape}")
        assert_reusable(cases, ys, ws, f"single {shape}")


def test_deterministic_and_equal_across_repeats(batch_kernel):
    cases = make_cases([(512, 4096, 16), (512, 4096, 16), (1000, 2048, 5)], seed0=400)
    ys1, ws = run_batch(cases)
    ys2, _ = run_batch(cases, workspace=ws)
    torch.cuda.synchronize()
    for a, b in zip(ys1, ys2):
        assert torch.equal(a, b)
    check_all(cases, ys1, "repeat")


def test_more_problems_than_one_launch_and_problems_that_run_alone(batch_kernel):
    """11 problems: two launches of the batched kernel plus problems it does not take
    (m > 16: tensor-core kernel; n_in not a multiple of 128: register-fed kernel; m = 0)."""
    shapes = [(128, 256, 1 + i % 8) for i in range(9)] + [(200, 512, 40), (96, 520, 3), (64, 256, 0)]
    cases = make_cases(shapes, seed0=500)
    ys, ws = run_batch(cases)
    torch.cuda.synchronize()
    assert bd.bd_get_device_status() == bd.BD_OK
    for i, (c, y) in enumerate(zip(cases, ys)):
        if c.m == 0:
            continue
        y_ref, mag = c.reference()
        assert_y_close(y_host(y), y_ref, mag, f"problem {i}")
    assert_reusable(cases, ys, ws, "11 problems")


@pytest.mark.parametrize("m", [1, 16])
def test_llama7b_layer_batches_full_size(m, batch_kernel):
    """q, k, v (4096 x 4096) in one batch and gate, up (11008 x 4096) in another, sampled outputs."""
    c = workloads.LLAMA7B_LAYER
    for group in (("q", "k", "v"), ("gate", "up")):
        shapes = [(n_out, n_in) for (name, n_out, n_in) in c["matrices"] if name in group]
        cases = [LinearCase(n_out, n_in, m, c["sigma"], c["b"], c["mode"], seed=700 + i)
                 for i, (n_out, n_in) in enumerate(shapes)]
        ys, ws = run_batch(cases)
        torch.cuda.synchronize()
        assert bd.bd_get_device_status() == bd.BD_OK
        for i, (case, y) in enumerate(zip(cases, ys)):
            yh = y_host(y)
            ts, js = sample_outputs(case.m, case.n_out, 400, seed=i)
            y_ref, mag = case.reference_sampled(ts, js)
            assert_y_close(yh[ts, js], y_ref, mag, f"{group} problem {i} m={m}")
        assert_reusable(cases, ys, ws, f"{group} m={m}")


@pytest.mark.parametrize("m", [1, 9])
def test_llama3_8b_qkv_batch_full_size_per_row_alpha(m, batch_kernel):
    """q (4096 x 4096) with k and v (1024 x 4096) in one batch, per-row alpha, sampled outputs."""
    shapes = [(4096, 4096), (1024, 4096), (1024, 4096)]
    cases = [LinearCase(n_out, n_in, m, 0.02, 1e-3, 1, seed=750 + i) for i, (n_out, n_in) in enumerate(shapes)]
    ys, ws = run_batch(cases)
    torch.cuda.synchronize()
    assert bd.bd_get_device_status() == bd.BD_OK
    for i, (case, y) in enumerate(zip(cases, ys)):
        yh = y_host(y)
        ts, js = sample_outputs(case.m, case.n_out, 400, seed=10 + i)
        y_ref, mag = case.reference_sampled(ts, js)
        assert_y_close(yh[ts, js], y_ref, mag, f"qkv problem {i} m={m}")
    assert_reusable(cases, ys, ws, f"qkv m={m}")


def test_in_a_graph_with_weight_prefetch_and_a_dependent_batch(batch_kernel):
    """Two batches captured in a graph with weight prefetch on; the second batch
    reads the first one's output as its activations (a read-after-write that a
    premature activation load would miss)."""
    a = make_cases([(384, 1024, 8), (384, 1024, 8)], seed0=800)
    b = LinearCase(256, 384, 0, seed=810)
    s = torch.cuda.Stream()
    ya = [torch.full((8, 384), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in a]
    yb = torch.full((8, 256), float("nan"), dtype=torch.bfloat16, device="cuda")
    da = bd.linear_descs([(c.x, c.w_base, c.bits, c.alpha, 0, y) for c, y in zip(a, ya)])
    db = bd.linear_descs([(ya[0], b.w_base, b.bits, b.alpha, 0, yb)])
    ws = torch.zeros(max(bd.bd_linear_batch_workspace_size(da), bd.bd_linear_batch_workspace_size(db), 1),
                     dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    prev = bd.bd_set_weight_prefetch(1)
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            bd.bd_linear_batch(da, ws, s)
            bd.bd_linear_batch(db, ws, s)
        g.replay()
        g.replay()
        torch.cuda.synchronize()
    finally:
        bd.bd_set_weight_prefetch(prev)
    assert bd.bd_get_device_status() == bd.BD_OK
    check_all(a, ya, "graph batch 1")
    y_ref, mag = oracle.linear(synth.as_u16(ya[0]), b.wb_h, b.bits_h, b.alpha32_h, 0)
    assert_y_close(y_host(yb), y_ref, mag, "graph batch 2 (dependent)")


def test_wait_limit_zero_reports_timeout_and_context_survives(batch_kernel):
    """A zero wait limit makes the batched kernel give up at its first unsatisfied
    wait; it records a timeout, drains its copies and returns.  After zeroing the
    workspace again a normal call is correct."""
    cases = make_cases([(4096, 4096, 4), (4096, 4096, 4)], seed0=900)
    assert bd.bd_get_device_status() == bd.BD_OK
    prev = bd.bd_set_wait_limit_ns(0)
    try:
        _, ws = run_batch(cases)
        torch.cuda.synchronize()
        status = bd.bd_get_device_status()
    finally:
        bd.bd_set_wait_limit_ns(prev)
    assert status == bd.BD_ERR_DEVICE_TIMEOUT
    assert bd.bd_get_device_status() == bd.BD_OK
    ws.zero_()
    ys, ws = run_batch(cases, workspace=ws)
    check_all(cases, ys, "after timeout")
    assert_reusable(cases, ys, ws, "after timeout")


def test_workspace_errors():
    cases = make_cases([(256, 512, 2), (128, 512, 2)], seed0=950)
    ys = [torch.empty((2, c.n_out), dtype=torch.bfloat16, device="cuda") for c in cases]
    descs = bd.linear_descs([(c.x, c.w_base, c.bits, c.alpha, 0, y) for c, y in zip(cases, ys)])
    need = bd.bd_linear_batch_workspace_size(descs)
    assert need > 0
    with pytest.raises(bd.BitDeltaError) as e:
        bd.bd_linear_batch(descs, None)
    assert e.value.status == bd.BD_ERR_WORKSPACE
    small = torch.zeros(need - 1, dtype=torch.uint8, device="cuda")
    with pytest.raises(bd.BitDeltaError) as e:
        bd.bd_linear_batch(descs, small)
    assert e.value.status == bd.BD_ERR_WORKSPACE
    # a single linear runs as bd_linear and needs no workspace
    assert bd.bd_linear_batch_workspace_size(bd.linear_descs(
        [(cases[0].x, cases[0].w_base, cases[0].bits, cases[0].alpha, 0, ys[0])])) == 0
    assert bd.bd_linear_batch_workspace_size((bd.LinearDesc * 0)()) == 0


# Tensor-core problems launched together on the pair kernel: ragged rows (vs 256), ragged token
# tiles, different K per linear, several linears per pair wave; each batch has at least 76 pair
# tiles (256 W rows x 256 tokens), so that together they fill the 152 SMs and share one launch.
PAIR_BATCHES = {
    "qkv_like": [(4096, 1024, 1000), (1024, 1024, 1000), (1024, 1024, 1000)],
    "ragged": [(1000, 640, 300), (2570, 4096, 777), (3000, 192, 300), (130, 520, 2048)],
    "gate_up_like": [(3584, 1024, 513), (3584, 1024, 513)],
}


@pytest.mark.parametrize("name", list(PAIR_BATCHES))
@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("ring", [0, 1, 2])
def test_tensor_core_problems_on_the_pair_kernel(name, mode, ring):
    cases = make_cases(PAIR_BATCHES[name], seed0=700, mode=mode)
    with bd.option(bd.BD_OPT_PAIR_RING, ring):
        ys, ws = run_batch(cases)
    check_all(cases, ys, f"pair batch {name} mode={mode}")
    assert_reusable(cases, ys, ws, f"pair batch {name}")
    # the same problems one by one on the pair kernel: identical bits
    with bd.option(bd.BD_OPT_PREFILL_KERNEL, 2):
        for c, y in zip(cases, ys):
            y1 = torch.empty_like(y)
            bd.bd_linear(c.x, c.w_base, c.bits, c.alpha, c.mode, y1)
            torch.cuda.synchronize()
            assert torch.equal(y1, y), f"{name}: {c.n_out}x{c.n_in} m={c.m} differs from bd_linear"


def test_llama3_8b_layer_prefill_batches_full_size():
    """A stack layer's q/k/v and gate/up at 2048 tokens, each group in one bd_linear_batch call (one
    pair-kernel launch each), sampled outputs against the oracle."""
    c = workloads.LLAMA3_8B_STACK
    mats = dict((n, (a, b)) for n, a, b in c["matrices"])
    for group in (("q", "k", "v"), ("gate", "up")):
        cases = [LinearCase(mats[g][0], mats[g][1], 2048, c["sigma"], c["b"], c["mode"],
                            seed=workloads.matrix_seed(c["seed"], 900 + j)) for j, g in enumerate(group)]
        x = cases[0].x
        for cs in cases[1:]:  # the group shares its input, as in a layer
            cs.x, cs.x_h = x, cases[0].x_h
        ys, _ = run_batch(cases)
        torch.cuda.synchronize()
        assert bd.bd_get_device_status() == bd.BD_OK
        for g, cs, y in zip(group, cases, ys):
            ts, js = sample_outputs(cs.m, cs.n_out, 800, seed=cs.n_out)
            y_ref, mag = cs.reference_sampled(ts, js)
            assert_y_close(y_host(y)[ts, js], y_ref, mag, f"{g} m=2048")
        del cases, ys
        torch.cuda.empty_cache()
