"""Delta cache in CUDA mode: deltas registered from pinned host memory are
loaded into a device arena on first request and used by the fused linear
straight from there; eviction and reload keep results exact against the
oracle, with every copy and kernel ordered on streams (no host sync between
requests)."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from bit_delta_tenant_gb300 import bitdelta as bd
from bit_delta_tenant_gb300 import synth
from helpers import assert_y_close, y_host

pytestmark = pytest.mark.gpu


def variants(n, n_out, n_in, seed=0):
    g = synth.generator(seed, "cuda")
    wb = synth.bf16_normal((n_out, n_in), 0.02, g, "cuda")
    out = []
    for v in range(n):
        d = synth.laplace_f32((n_out, n_in), 5e-4 * (v + 1), g, "cuda")
        wf = (wb.float() + d).to(torch.bfloat16)
        bits, alpha, _ = oracle.compress(synth.as_u16(wb), synth.as_u16(wf), 1)
        out.append((torch.from_numpy(bits).pin_memory(), torch.from_numpy(alpha).pin_memory(), bits, alpha))
    return wb, out


def linear_from_ptrs(x, wb, bits_ptr, alpha_ptr, y, stream):
    lib = bd.load_library()
    m, n_in = x.shape
    n_out = wb.shape[0]
    rc = lib.bd_linear(ctypes.c_void_p(x.data_ptr()), m, ctypes.c_void_p(wb.data_ptr()), ctypes.c_void_p(bits_ptr),
                       ctypes.c_void_p(alpha_ptr), 1, n_out, n_in, ctypes.c_void_p(y.data_ptr()),
                       ctypes.c_void_p(stream.cuda_stream))
    assert rc == bd.BD_OK


def test_requests_through_the_cache_with_eviction():
    n_out, n_in, m = 256, 1024, 4
    wb, vs = variants(3, n_out, n_in, seed=3)
    block = (n_out * n_in // 8 + 255) // 256 * 256 + 1024
    arena = torch.empty(2 * block, dtype=torch.uint8, device="cuda")   # room for two deltas
    cache = bd.DeltaCache(3, arena, half_life_s=5.0)
    for v, (hb, ha, _, _) in enumerate(vs):
        cache.register(v, hb, ha)
    x = synth.activations(m, n_in, 11, "cuda")
    xh = synth.as_u16(x)
    wbh = synth.as_u16(wb)
    s = torch.cuda.Stream()
    seq = [0, 1, 0, 2, 1, 2, 0, 0, 1]
    ys = []
    for i, v in enumerate(seq):
        rc, bp, ap = cache.acquire(v, now_s=float(i), stream=s)
        assert rc == bd.BD_OK
        y = torch.empty((m, n_out), dtype=torch.bfloat16, device="cuda")
        linear_from_ptrs(x, wb, bp, ap, y, s)
        assert cache.release(v, stream=s) == bd.BD_OK
        ys.append(y)
    s.synchronize()
    assert bd.bd_get_device_status() == bd.BD_OK
    for v, y in zip(seq, ys):
        y_ref, mag = oracle.linear(xh, wbh, vs[v][2], vs[v][3], 1)
        assert_y_close(y_host(y), y_ref, mag, f"variant {v} through the cache")
    st = cache.stats()
    assert st.acquires == len(seq) and st.evictions >= 2 and st.loads == st.misses
    cache.close()


def test_second_stream_waits_for_the_load_in_flight():
    n_out, n_in = 4096, 4096
    wb, vs = variants(1, n_out, n_in, seed=4)
    arena = torch.empty(4 << 20, dtype=torch.uint8, device="cuda")
    cache = bd.DeltaCache(1, arena)
    cache.register(0, vs[0][0], vs[0][1])
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    rc1, b1, a1 = cache.acquire(0, stream=s1)
    rc2, b2, a2 = cache.acquire(0, stream=s2)      # queued copy on s1: s2 waits for its event
    assert rc1 == bd.BD_OK and rc2 == bd.BD_OK and (b1, a1) == (b2, a2)
    x = synth.activations(1, n_in, 5, "cuda")
    y = torch.empty((1, n_out), dtype=torch.bfloat16, device="cuda")
    linear_from_ptrs(x, wb, b2, a2, y, s2)
    cache.release(0, stream=s1)
    cache.release(0, stream=s2)
    torch.cuda.synchronize()
    assert cache.stats().loads == 1
    y_ref, mag = oracle.linear(synth.as_u16(x), synth.as_u16(wb), vs[0][2], vs[0][3], 1)
    assert_y_close(y_host(y), y_ref, mag, "second stream")
    cache.close()
