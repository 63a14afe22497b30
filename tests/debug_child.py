"""Child process of test_gpu_debug_build: small cases of every kernel family through the
bounds-checked library (libbitdelta_debug.so), each checked against the fp64 oracle, with
the device status word read after each (a failed index check would report
BD_ERR_DEVICE_BOUNDS).  Run as a separate process so that the debug library, not the
release one, is the one loaded.  Prints "debug build ok" on success."""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
for p in (ROOT, HERE):
    if p not in sys.path:
        sys.path.insert(0, p)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from bit_delta_tenant_gb300 import bitdelta as bd  # noqa: E402

bd.load_library(bd.LIB_DEBUG_PATH)

import oracle  # noqa: E402
from bit_delta_tenant_gb300 import synth  # noqa: E402
from helpers import LinearCase, assert_y_close, y_host  # noqa: E402


def status_ok(what):
    torch.cuda.synchronize()
    st = bd.bd_get_device_status()
    assert st == bd.BD_OK, f"{what}: {bd.bd_status_string(st)}"


def main():
    assert bd.bd_build_flags() & 1, "the bounds-checked library is not the one loaded"
    torch.cuda.set_device(0)
    # compression, both forms, both alpha modes, ragged shapes
    for n_out, n_in, mode in ((129, 136, 0), (300, 8320, 1), (7, 24, 1)):
        for form in (0, 1):
            wb, wf = synth.matrix_pair(n_out, n_in, 0.02, 1e-3, seed=n_out + n_in, device="cuda")
            bits = torch.empty((n_out, n_in // 8), dtype=torch.uint8, device="cuda")
            alpha = torch.empty((n_out if mode else 1,), dtype=torch.float32, device="cuda")
            ws = torch.empty((max(16, bd.bd_compress_workspace_size(n_out, n_in, mode)),), dtype=torch.uint8,
                             device="cuda")
            with bd.option(bd.BD_OPT_COMPRESS_FORM, form):
                bd.bd_compress(wb, wf, mode, bits, alpha, ws)
            status_ok(f"compress {n_out}x{n_in} form {form}")
            rb, _, ra = oracle.compress(synth.as_u16(wb), synth.as_u16(wf), mode)
            assert np.array_equal(bits.cpu().numpy(), rb), "bits differ"
            assert np.all(np.abs(alpha.cpu().numpy().astype(np.float64) - ra) <= 1e-6 * np.abs(ra))
    # fused linear on every kernel: register-fed and TMA streaming, single-CTA and pair tensor cores
    for n_out, n_in, m, path, kernel in ((65, 256, 9, 1, 0), (130, 520, 5, 3, 0), (300, 640, 100, 2, 1),
                                         (257, 640, 300, 2, 2), (64, 4104, 70, 2, 1)):
        case = LinearCase(n_out, n_in, m, mode=m % 2, b="row:5e-4:2e-3" if m % 2 else 1e-3, seed=n_out + m)
        prev = bd.bd_set_linear_path(path)
        try:
            with bd.option(bd.BD_OPT_PREFILL_KERNEL, kernel):
                y = case.run_linear()
        finally:
            bd.bd_set_linear_path(prev)
        status_ok(f"linear {n_out}x{n_in} m={m} path {path}")
        y_ref, mag = case.reference()
        assert_y_close(y_host(y), y_ref, mag, f"linear {n_out}x{n_in} m={m}")
    # the persistent pair kernel in both shapes (5-deep ring with the whole tile staged, 6-deep with two
    # staged halves), several tiles per pair, ragged rows and tokens
    for ring in (1, 2):
        case = LinearCase(2000, 1000, 3000, mode=ring - 1, b="row:5e-4:2e-3" if ring == 2 else 1e-3, seed=40 + ring)
        with bd.option(bd.BD_OPT_PREFILL_KERNEL, 2), bd.option(bd.BD_OPT_PAIR_RING, ring):
            y = case.run_linear()
        status_ok(f"pair kernel ring {ring}")
        y_ref, mag = case.reference()
        assert_y_close(y_host(y), y_ref, mag, f"pair kernel ring {ring}")
    # batched linear: the streaming batch kernels and a pair-kernel batch
    for shapes, kern in (([(200, 384, 3), (65, 1152, 8), (1000, 640, 2)], 2),
                         ([(200, 384, 3), (65, 1152, 8)], 1),
                         ([(4096, 1024, 1000), (1024, 1024, 1000)], 0)):
        cases = [LinearCase(a, b, c, seed=11 + i) for i, (a, b, c) in enumerate(shapes)]
        ys = [torch.empty((c.m, c.n_out), dtype=torch.bfloat16, device="cuda") for c in cases]
        descs = bd.linear_descs([(c.x, c.w_base, c.bits, c.alpha, c.mode, y) for c, y in zip(cases, ys)])
        wsb = torch.zeros(max(1, bd.bd_linear_batch_workspace_size(descs)), dtype=torch.uint8, device="cuda")
        with bd.option(bd.BD_OPT_BATCH_KERNEL, kern):
            bd.bd_linear_batch(descs, wsb)
        status_ok(f"batch {shapes}")
        for c, y in zip(cases, ys):
            y_ref, mag = c.reference()
            assert_y_close(y_host(y), y_ref, mag, f"batch {c.n_out}x{c.n_in}")
    # multi-tenant: streaming kernels at 16 tokens, tensor-core tiles (both kernels) at 300 tokens
    g = synth.generator(5, "cuda")
    n_out, n_in, nv = 257, 512, 5
    w_base = synth.bf16_normal((n_out, n_in), 0.015, g, "cuda")
    wb_h = synth.as_u16(w_base)
    bits_h, alpha_h, bits_d, alpha_d = [], [], [], []
    for v in range(nv):
        d = synth.laplace_f32((n_out, n_in), 5e-4 * (v + 1), g, "cuda")
        b_h, a_h, _ = oracle.compress(wb_h, synth.as_u16((w_base.float() + d).to(torch.bfloat16)), v % 2)
        bits_h.append(b_h), alpha_h.append(a_h)
        bits_d.append(torch.from_numpy(b_h).cuda()), alpha_d.append(torch.from_numpy(a_h).cuda())
    modes = [v % 2 for v in range(nv)]
    for m, path, kernel in ((16, 2, 0), (16, 4, 0), (16, 1, 0), (300, 0, 1), (300, 0, 2)):
        ids_h = synth.uniform_ids(m, nv, seed=m + path)
        x = synth.activations(m, n_in, seed=m, device="cuda")
        y = torch.empty((m, n_out), dtype=torch.bfloat16, device="cuda")
        wsg = torch.empty((bd.bd_linear_grouped_workspace_size(m, nv, n_out, n_in),), dtype=torch.uint8,
                          device="cuda")
        with bd.option(bd.BD_OPT_GROUPED_PATH, path), bd.option(bd.BD_OPT_PREFILL_KERNEL, kernel):
            bd.bd_linear_grouped(x, torch.from_numpy(ids_h).cuda(), w_base, bits_d, alpha_d, modes, y, wsg)
        status_ok(f"multi-tenant m={m} path {path} kernel {kernel}")
        y_ref, mag = oracle.linear_grouped(synth.as_u16(x), ids_h, wb_h, bits_h, alpha_h, np.array(modes, np.int32))
        assert_y_close(y_host(y), y_ref, mag, f"multi-tenant m={m} path {path}")
    print("debug build ok")


if __name__ == "__main__":
    main()
