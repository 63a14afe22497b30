"""GPU multi-tenant fused linear (bd_linear_grouped) against the fp64 oracle.

Each token carries its own variant id over one shared W_base; the expected
output of token t is the oracle's fused linear with variant ids[t]'s packed
bits and alpha.  Covers the 14-variant workload (uniform decode ids, Zipf
prefill segments), empty variants, one variant, mixed alpha modes, ragged
shapes and out-of-range ids."""
import numpy as np
import pytest
import torch

import oracle
from bit_delta_tenant_gb300 import bitdelta as bd
from bit_delta_tenant_gb300 import synth, workloads
from helpers import assert_y_close, sample_outputs, y_host

pytestmark = pytest.mark.gpu


class GroupedCase:
    def __init__(self, n_out, n_in, n_var, ids, scales=None, modes=None, sigma=0.015, seed=0):
        dev = "cuda"
        self.n_out, self.n_in, self.n_var = n_out, n_in, n_var
        g = synth.generator(seed, dev)
        self.w_base = synth.bf16_normal((n_out, n_in), sigma, g, dev)
        self.wb_h = synth.as_u16(self.w_base)
        scales = scales or [5e-4 + 1.5e-3 * v / max(1, n_var - 1) for v in range(n_var)]
        self.modes = list(modes) if modes is not None else [0] * n_var
        self.bits_h, self.alpha_h, self.bits, self.alpha = [], [], [], []
        for v in range(n_var):
            d = synth.laplace_f32((n_out, n_in), scales[v], g, dev)
            wf = (self.w_base.float() + d).to(torch.bfloat16)
            b, a, _ = oracle.compress(self.wb_h, synth.as_u16(wf), self.modes[v])
            self.bits_h.append(b), self.alpha_h.append(a)
            self.bits.append(torch.from_numpy(b).to(dev)), self.alpha.append(torch.from_numpy(a).to(dev))
        self.ids_h = np.asarray(ids, np.int32)
        self.m = len(self.ids_h)
        self.ids = torch.from_numpy(self.ids_h).to(dev)
        self.x = synth.activations(self.m, n_in, seed + 1, dev)
        self.x_h = synth.as_u16(self.x)

    def run(self):
        y = torch.zeros((self.m, self.n_out), dtype=torch.bfloat16, device="cuda")
        ws = torch.empty((bd.bd_linear_grouped_workspace_size(self.m, self.n_var, self.n_out, self.n_in),),
                         dtype=torch.uint8, device="cuda")
        bd.bd_linear_grouped(self.x, self.ids, self.w_base, self.bits, self.alpha, self.modes, y, ws)
        torch.cuda.synchronize()
        return y

    def reference(self):
        return oracle.linear_grouped(self.x_h, self.ids_h, self.wb_h, self.bits_h, self.alpha_h,
                                     np.array(self.modes, np.int32))

    def reference_sampled(self, ts, js):
        return oracle.linear_grouped_sampled(self.x_h, self.ids_h, self.wb_h, self.bits_h, self.alpha_h,
                                             np.array(self.modes, np.int32), ts, js)


def check_full(case, what):
    y = case.run()
    assert bd.bd_get_device_status() == bd.BD_OK
    y_ref, mag = case.reference()
    assert_y_close(y_host(y), y_ref, mag, what)
    return y


def test_single_variant_equals_plain_linear():
    case = GroupedCase(192, 256, 1, np.zeros(40, np.int32), seed=1)
    y = check_full(case, "V=1")
    y1 = torch.empty_like(y)
    bd.bd_linear(case.x, case.w_base, case.bits[0], case.alpha[0], 0, y1)
    torch.cuda.synchronize()
    y_ref, mag = oracle.linear(case.x_h, case.wb_h, case.bits_h[0], case.alpha_h[0], 0)
    assert_y_close(y_host(y1), y_ref, mag, "plain")


@pytest.mark.parametrize("m", [1, 7, 64, 65, 300, 2048])
def test_uniform_ids_fourteen_variants(m):
    ids = synth.uniform_ids(m, 14, seed=m)
    case = GroupedCase(256, 512, 14, ids, seed=10 + m)
    check_full(case, f"14 variants m={m}")


@pytest.fixture(params=["single", "pair5", "pair6"])
def prefill_kernel(request):
    """The tensor-core kernel of the per-variant token tiles: one CTA per 128 W rows, or CTA pairs
    on 256 W rows (BD_OPT_PREFILL_KERNEL) in either of the pair kernel's shapes (BD_OPT_PAIR_RING:
    5-deep ring, whole tile staged; 6-deep ring, two staged halves)."""
    kernel, ring = {"single": (1, 0), "pair5": (2, 1), "pair6": (2, 2)}[request.param]
    with bd.option(bd.BD_OPT_PREFILL_KERNEL, kernel), bd.option(bd.BD_OPT_PAIR_RING, ring):
        yield request.param


def test_zipf_segments_fourteen_variants(prefill_kernel):
    ids = synth.zipf_ids(2048, 14, 1.1, seed=5)
    assert sorted(np.bincount(ids, minlength=14).tolist(), reverse=True) == \
        [699, 326, 209, 152, 119, 97, 82, 71, 62, 56, 50, 45, 42, 38]
    case = GroupedCase(200, 520, 14, ids, seed=6)
    check_full(case, f"zipf {prefill_kernel}")


@pytest.mark.parametrize("n_out,n_in,m,n_var", [(257, 640, 300, 5), (513, 192, 1000, 14), (100, 4096, 65, 3),
                                                 (384, 1024, 777, 64)])
def test_tensor_core_tiles_ragged_shapes(n_out, n_in, m, n_var, prefill_kernel):
    """Per-variant token tiles on both tensor-core kernels: ragged W rows (vs 128 and 256), ragged
    K, tiles of a few tokens, up to 64 variants with mixed alpha modes."""
    ids = synth.uniform_ids(m, n_var, seed=n_out + m)
    case = GroupedCase(n_out, n_in, n_var, ids, modes=[v % 2 for v in range(n_var)], seed=n_in + m)
    check_full(case, f"{prefill_kernel} {n_out}x{n_in} m={m} V={n_var}")


def test_empty_variants_and_all_tokens_in_one_variant():
    case = GroupedCase(130, 136, 5, np.full(37, 3, np.int32), seed=7)
    check_full(case, "one busy variant of five")


def test_mixed_alpha_modes_and_ragged_shapes():
    ids = np.array([4, 0, 0, 2, 1, 4, 4, 0, 2, 2, 3, 1, 0] * 5, np.int32)
    case = GroupedCase(129, 24, 5, ids, modes=[0, 1, 0, 1, 1], seed=8)
    check_full(case, "mixed modes")


def test_permuted_batch_gives_permuted_output():
    ids = synth.uniform_ids(96, 6, seed=3)
    case = GroupedCase(128, 256, 6, ids, seed=9)
    y = check_full(case, "original order")
    perm = np.random.default_rng(1).permutation(case.m)
    case.ids_h = case.ids_h[perm]
    case.ids = torch.from_numpy(case.ids_h).to("cuda")
    case.x = case.x[torch.from_numpy(perm).to("cuda")].contiguous()
    case.x_h = synth.as_u16(case.x)
    yp = check_full(case, "permuted order")
    # the same tokens in another order: identical rows up to the kernel's rounding
    np.testing.assert_allclose(y_host(yp), y_host(y)[perm], rtol=2e-2, atol=1e-2)


def test_out_of_range_id_is_reported_and_other_tokens_are_correct():
    ids = np.array([0, 1, 5, 2, -1, 1, 0, 2], np.int32)
    case = GroupedCase(64, 128, 3, ids, seed=11)
    y = case.run()
    assert bd.bd_get_device_status() == bd.BD_ERR_BAD_VARIANT_ID
    assert bd.bd_get_device_status() == bd.BD_OK
    good = np.where((ids >= 0) & (ids < 3))[0]
    y_ref, mag = oracle.linear_grouped(case.x_h[good], ids[good], case.wb_h, case.bits_h, case.alpha_h,
                                       np.array(case.modes, np.int32))
    assert_y_close(y_host(y)[good], y_ref, mag, "good tokens")


@pytest.mark.parametrize("kind", ["decode", "prefill"])
def test_fourteen_variant_workload_full_size(kind, grouped_path):
    c = workloads.GROUPED_14
    m = c["decode_m"] if kind == "decode" else c["prefill_m"]
    ids = synth.uniform_ids(m, c["n_variants"], c["seed"]) if kind == "decode" else \
        synth.zipf_ids(m, c["n_variants"], c["zipf_s"], c["seed"])
    case = GroupedCase(c["n_out"], c["n_in"], c["n_variants"], ids, scales=workloads.variant_scales(c),
                       sigma=c["sigma"], seed=c["seed"])
    y = case.run()
    assert bd.bd_get_device_status() == bd.BD_OK
    yh = y_host(y)
    assert np.all(np.isfinite(yh))
    ts, js = sample_outputs(case.m, case.n_out, 1500, seed=m)
    y_ref, mag = case.reference_sampled(ts, js)
    assert_y_close(yh[ts, js], y_ref, mag, f"14-variant {kind}")


@pytest.mark.parametrize("m", [1, 8, 16])
@pytest.mark.parametrize("path", ["2", "4"], ids=["mma_stream", "base_tc_signs_mma"])
def test_small_batches_on_the_fourteen_variant_shape(m, path):
    """Few tokens over the full 8192 x 8192 shape: 64 K steps per CTA with warps that have no
    sign tile (fewer tiles than warps) running ahead of the others through the ring."""
    c = workloads.GROUPED_14
    ids = synth.uniform_ids(m, c["n_variants"], c["seed"] + m)
    case = GroupedCase(c["n_out"], c["n_in"], c["n_variants"], ids, scales=workloads.variant_scales(c),
                       sigma=c["sigma"], seed=c["seed"])
    with bd.option(bd.BD_OPT_GROUPED_PATH, int(path)):
        y = case.run()
    assert bd.bd_get_device_status() == bd.BD_OK
    ts, js = sample_outputs(case.m, case.n_out, 600, seed=m)
    y_ref, mag = case.reference_sampled(ts, js)
    assert_y_close(y_host(y)[ts, js], y_ref, mag, f"14-variant m={m} path={path}")


@pytest.fixture(params=["1", "2", "3", "4"], ids=["tcgen05_stream", "mma_stream", "per_variant_tiles",
                                                  "base_tc_signs_mma"])
def grouped_path(request):
    """Force one multi-tenant kernel (shapes a kernel cannot take fall through to the next)."""
    with bd.option(bd.BD_OPT_GROUPED_PATH, int(request.param)):
        yield request.param


@pytest.mark.parametrize("n_out,n_in,m,n_var", [(129, 256, 64, 14), (64, 1152, 1, 3), (300, 128, 33, 16),
                                                 (1000, 4096, 9, 5), (65, 640, 64, 12), (7, 384, 17, 2),
                                                 (200, 192, 40, 7), (513, 2048, 64, 14)])
def test_streaming_kernel_shapes_and_mixed_modes(n_out, n_in, m, n_var, grouped_path):
    """Small batches: every kernel against the oracle, ragged rows, mixed alpha modes."""
    ids = synth.uniform_ids(m, n_var, seed=n_out + m)
    modes = [v % 2 for v in range(n_var)]
    case = GroupedCase(n_out, n_in, n_var, ids, modes=modes, seed=n_in + m)
    check_full(case, f"grouped path={grouped_path} {n_out}x{n_in} m={m} V={n_var}")


def test_streaming_kernel_bad_id_and_empty_variants(grouped_path):
    ids = np.array([0, 5, 2, 2, 9, -3, 0, 2, 5, 5, 5], np.int32)  # variants 1, 3, 4 empty; 9 and -3 invalid
    case = GroupedCase(256, 512, 6, ids, modes=[1, 0, 1, 0, 1, 0], seed=12)
    y = case.run()
    assert bd.bd_get_device_status() == bd.BD_ERR_BAD_VARIANT_ID
    good = np.where((ids >= 0) & (ids < 6))[0]
    y_ref, mag = oracle.linear_grouped(case.x_h[good], ids[good], case.wb_h, case.bits_h, case.alpha_h,
                                       np.array(case.modes, np.int32))
    assert_y_close(y_host(y)[good], y_ref, mag, "good tokens (streaming)")


@pytest.mark.parametrize("path", ["1", "2", "4"], ids=["tcgen05_stream", "mma_stream", "base_tc_signs_mma"])
def test_stalled_wait_reports_timeout_and_context_survives(path):
    """Each multi-tenant streaming kernel, made to wait first on a barrier that nothing
    completes (BD_OPT_TEST_STALL) under a 1 ms wait limit, gives up: it records a timeout,
    drains its own copies (and MMAs) and returns.  The status is read and cleared once, the
    context stays usable, and the same call afterwards is correct against the oracle."""
    ids = synth.uniform_ids(16, 5, seed=77)
    case = GroupedCase(1024, 4096, 5, ids, seed=78)
    assert bd.bd_get_device_status() == bd.BD_OK
    with bd.option(bd.BD_OPT_GROUPED_PATH, int(path)):
        prev = bd.bd_set_wait_limit_ns(1_000_000)
        try:
            with bd.option(bd.BD_OPT_TEST_STALL, 1):
                case.run()
            status = bd.bd_get_device_status()
        finally:
            bd.bd_set_wait_limit_ns(prev)
        assert status == bd.BD_ERR_DEVICE_TIMEOUT
        assert bd.bd_get_device_status() == bd.BD_OK  # read-and-clear
        y = case.run()
    assert bd.bd_get_device_status() == bd.BD_OK
    y_ref, mag = case.reference()
    assert_y_close(y_host(y), y_ref, mag, f"after timeout, path {path}")
