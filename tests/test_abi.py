"""The C-ABI library without a GPU: it builds, loads, exports every declared
symbol, and rejects bad arguments synchronously before any CUDA call."""
import ctypes
import os
import re

import pytest

from bit_delta_tenant_gb300 import bitdelta as bd
from bit_delta_tenant_gb300 import build as bd_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bitdelta.h")

ALIGNED = 0x10000          # fake device addresses: never dereferenced on these paths
MISALIGNED = 0x10008


@pytest.fixture(scope="module")
def lib():
    bd_build.build()
    return bd.load_library()


def declared_functions():
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bd_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for required in ["bd_compress", "bd_compress_workspace_size", "bd_compress_batch",
                     "bd_compress_batch_workspace_size", "bd_linear", "bd_linear_batch",
                     "bd_linear_batch_workspace_size", "bd_linear_grouped",
                     "bd_linear_grouped_workspace_size", "bd_status_string", "bd_get_device_status"]:
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in bitdelta.h but not exported"


def test_library_exports_nothing_else():
    out = os.popen(f"nm -D --defined-only {bd_build.LIB_PATH}").read()
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert exported and all(s.startswith("bd_") for s in exported), sorted(exported)[:10]


def test_status_strings(lib):
    for code in range(8):
        assert bd.bd_status_string(code) and bd.bd_status_string(code) != "unknown status"
    assert bd.bd_status_string(99) == "unknown status"
    assert bd.bd_version() >= 100


def test_workspace_sizes(lib):
    # scalar alpha: one fp64 partial per 1024 chunks of 8 elements
    assert bd.bd_compress_workspace_size(256, 512, 0) == (256 * 64 // 1024) * 8
    assert bd.bd_compress_workspace_size(4096, 4096, 0) == (4096 * 512 // 1024) * 8
    # per-row alpha: rows * segments per row (28672 / 8 = 3584 chunks -> 4 segments)
    assert bd.bd_compress_workspace_size(8192, 28672, 1) == 8192 * 4 * 8
    assert bd.bd_compress_workspace_size(4, 12, 0) == 0          # n_in not a multiple of 8
    assert bd.bd_compress_workspace_size(4, 16, 5) == 0          # unknown mode
    assert bd.bd_linear_grouped_workspace_size(64, 14, 8192, 8192) > 64 * 8192 * 2
    assert bd.bd_linear_grouped_workspace_size(64, 0, 8192, 8192) == 0
    assert bd.bd_linear_grouped_workspace_size(64, 65, 8192, 8192) == 0


def _compress(lib, wb=ALIGNED, wf=ALIGNED, n_out=4, n_in=16, mode=0, bits=ALIGNED, alpha=ALIGNED,
              ws=ALIGNED, ws_bytes=1 << 20):
    return lib.bd_compress(wb, wf, n_out, n_in, mode, bits, alpha, ws, ws_bytes, None)


def test_compress_rejects_bad_arguments(lib):
    assert _compress(lib, wb=0) == bd.BD_ERR_INVALID_ARG
    assert _compress(lib, alpha=0) == bd.BD_ERR_INVALID_ARG
    assert _compress(lib, mode=2) == bd.BD_ERR_INVALID_ARG
    assert _compress(lib, n_out=0) == bd.BD_ERR_INVALID_ARG
    assert _compress(lib, n_in=12) == bd.BD_ERR_UNSUPPORTED_SHAPE
    assert _compress(lib, n_in=1 << 31) == bd.BD_ERR_UNSUPPORTED_SHAPE
    assert _compress(lib, wf=MISALIGNED) == bd.BD_ERR_MISALIGNED
    assert _compress(lib, ws=0) == bd.BD_ERR_WORKSPACE
    assert _compress(lib, ws_bytes=0) == bd.BD_ERR_WORKSPACE


def _linear(lib, x=ALIGNED, m=4, wb=ALIGNED, bits=ALIGNED, alpha=ALIGNED, mode=0, n_out=8, n_in=16, y=ALIGNED):
    return lib.bd_linear(x, m, wb, bits, alpha, mode, n_out, n_in, y, None)


def test_linear_rejects_bad_arguments(lib):
    assert _linear(lib, m=-1) == bd.BD_ERR_INVALID_ARG
    assert _linear(lib, x=0) == bd.BD_ERR_INVALID_ARG
    assert _linear(lib, bits=0) == bd.BD_ERR_INVALID_ARG
    assert _linear(lib, mode=7) == bd.BD_ERR_INVALID_ARG
    assert _linear(lib, n_in=20) == bd.BD_ERR_UNSUPPORTED_SHAPE
    assert _linear(lib, m=1 << 31) == bd.BD_ERR_UNSUPPORTED_SHAPE
    assert _linear(lib, y=MISALIGNED) == bd.BD_ERR_MISALIGNED
    assert _linear(lib, alpha=MISALIGNED) == bd.BD_ERR_MISALIGNED
    # an empty batch is valid and launches nothing
    assert _linear(lib, m=0, x=0, y=0) == bd.BD_OK


def _desc(**kw):
    d = dict(x=ALIGNED, w_base=ALIGNED, bits=ALIGNED, alpha=ALIGNED, y=ALIGNED, m=4, n_out=64, n_in=256,
             alpha_mode=0, reserved=0)
    d.update(kw)
    out = bd.LinearDesc()
    for k, v in d.items():
        setattr(out, k, v)
    return out


def _batch(lib, descs, ws=ALIGNED, ws_bytes=1 << 20, n=None):
    arr = (bd.LinearDesc * len(descs))(*descs)
    return lib.bd_linear_batch(arr, len(descs) if n is None else n, ctypes.c_void_p(ws), ws_bytes, None)


def _cdesc(**kw):
    d = dict(w_base=ALIGNED, w_ft=ALIGNED, bits_out=ALIGNED, alpha_out=ALIGNED, n_out=64, n_in=256,
             alpha_mode=0, reserved=0)
    d.update(kw)
    out = bd.CompressDesc()
    for k, v in d.items():
        setattr(out, k, v)
    return out


def test_compress_batch_rejects_bad_arguments(lib):
    def call(descs, ws=ALIGNED, ws_bytes=1 << 20, n=None):
        arr = (bd.CompressDesc * len(descs))(*descs)
        return lib.bd_compress_batch(arr, len(descs) if n is None else n, ctypes.c_void_p(ws), ws_bytes, None)
    good = _cdesc()
    assert call([good, _cdesc(w_ft=0)]) == bd.BD_ERR_INVALID_ARG
    assert call([_cdesc(alpha_mode=2)]) == bd.BD_ERR_INVALID_ARG
    assert call([_cdesc(reserved=5)]) == bd.BD_ERR_INVALID_ARG
    assert call([good, _cdesc(n_in=12)]) == bd.BD_ERR_UNSUPPORTED_SHAPE
    assert call([_cdesc(bits_out=MISALIGNED)]) == bd.BD_ERR_MISALIGNED
    assert call([good], n=bd.BD_COMPRESS_BATCH_MAX + 1) == bd.BD_ERR_INVALID_ARG
    assert call([good], ws=0) == bd.BD_ERR_WORKSPACE
    assert call([good], ws=ALIGNED + 16) == bd.BD_ERR_WORKSPACE      # not 256-byte aligned
    assert call([good], ws_bytes=8) == bd.BD_ERR_WORKSPACE
    assert call([]) == bd.BD_OK
    arr = (bd.CompressDesc * 2)(good, _cdesc(alpha_mode=1, n_out=3, n_in=16392))
    # scalar 64x256: 2 segments; per-row 16392: 3 segments per row; each region rounded to 256 bytes
    assert lib.bd_compress_batch_workspace_size(arr, 2) == 256 + 256


def test_linear_batch_rejects_bad_arguments(lib):
    """Validation happens before any launch: every problem is checked as bd_linear checks it."""
    good = _desc()
    assert _batch(lib, [good, _desc(m=-1)]) == bd.BD_ERR_INVALID_ARG
    assert _batch(lib, [good, _desc(x=0)]) == bd.BD_ERR_INVALID_ARG
    assert _batch(lib, [_desc(alpha_mode=3)]) == bd.BD_ERR_INVALID_ARG
    assert _batch(lib, [_desc(reserved=1)]) == bd.BD_ERR_INVALID_ARG
    assert _batch(lib, [good, _desc(n_in=20)]) == bd.BD_ERR_UNSUPPORTED_SHAPE
    assert _batch(lib, [_desc(y=MISALIGNED)]) == bd.BD_ERR_MISALIGNED
    assert _batch(lib, [good], n=-1) == bd.BD_ERR_INVALID_ARG
    assert _batch(lib, [good], n=bd.BD_LINEAR_BATCH_MAX + 1) == bd.BD_ERR_INVALID_ARG
    assert lib.bd_linear_batch(None, 2, None, 0, None) == bd.BD_ERR_INVALID_ARG
    # empty batches (no problems, or only m = 0 problems) are valid and launch nothing
    assert _batch(lib, []) == bd.BD_OK
    assert _batch(lib, [_desc(m=0, x=0, y=0)], ws=0, ws_bytes=0) == bd.BD_OK
    arr = (bd.LinearDesc * 1)(_desc(m=-1))
    assert lib.bd_linear_batch_workspace_size(arr, 1) == 0
    assert lib.bd_linear_batch_workspace_size(None, 0) == 0


def test_grouped_rejects_bad_arguments(lib):
    V = ctypes.c_void_p
    bits = (V * 2)(ALIGNED, ALIGNED)
    alph = (V * 2)(ALIGNED, ALIGNED)
    modes = (ctypes.c_int32 * 2)(0, 1)

    def call(x=ALIGNED, ids=ALIGNED, m=4, wb=ALIGNED, b=bits, a=alph, md=modes, nv=2, n_out=8, n_in=16,
             y=ALIGNED, ws=ALIGNED, ws_bytes=1 << 30):
        return lib.bd_linear_grouped(x, ids, m, wb, b, a, md, nv, n_out, n_in, y, ws, ws_bytes, None)

    assert call(nv=0) == bd.BD_ERR_INVALID_ARG
    assert call(nv=65) == bd.BD_ERR_INVALID_ARG
    assert call(ids=0) == bd.BD_ERR_INVALID_ARG
    assert call(b=None) == bd.BD_ERR_INVALID_ARG
    assert call(md=(ctypes.c_int32 * 2)(0, 3)) == bd.BD_ERR_INVALID_ARG
    assert call(b=(V * 2)(ALIGNED, 0)) == bd.BD_ERR_INVALID_ARG
    assert call(n_in=10) == bd.BD_ERR_UNSUPPORTED_SHAPE
    assert call(a=(V * 2)(ALIGNED, MISALIGNED)) == bd.BD_ERR_MISALIGNED
    assert call(ids=MISALIGNED) == bd.BD_ERR_MISALIGNED
    assert call(ws=0) == bd.BD_ERR_WORKSPACE
    assert call(ws_bytes=16) == bd.BD_ERR_WORKSPACE
    assert call(m=0, x=0, y=0, ids=0) == bd.BD_OK


def test_knobs_round_trip(lib):
    prev = bd.bd_set_wait_limit_ns(12345)
    assert bd.bd_set_wait_limit_ns(prev) == 12345
    p = bd.bd_set_linear_path(2)
    assert bd.bd_set_linear_path(p) == 2
    assert bd.bd_set_linear_path(9) == p          # out-of-range values are ignored
    assert bd.bd_set_linear_path(p) == p
    w = bd.bd_set_weight_prefetch(1)
    assert bd.bd_set_weight_prefetch(7) == 1          # any non-zero value enables
    assert bd.bd_set_weight_prefetch(w) == 1


@pytest.mark.parametrize("option,top", [(bd.BD_OPT_COMPRESS_FORM, 1), (bd.BD_OPT_GROUPED_PATH, 4),
                                        (bd.BD_OPT_BATCH_KERNEL, 2), (bd.BD_OPT_BATCH_SINGLE, 1),
                                        (bd.BD_OPT_TEST_STALL, 1), (bd.BD_OPT_PREFILL_KERNEL, 2),
                                        (bd.BD_OPT_PAIR_RING, 2)])
def test_options_accept_their_documented_range_only(lib, option, top):
    prev = bd.bd_set_option(option, top)
    try:
        assert bd.bd_set_option(option, top + 1) == -1     # out of range: nothing changed
        assert bd.bd_set_option(option, -1) == -1
        assert bd.bd_set_option(option, 0) == top
    finally:
        bd.bd_set_option(option, prev)
    assert bd.bd_set_option(0, 0) == -1 and bd.bd_set_option(99, 0) == -1  # unknown options


def test_reconstruct_rejects_bad_arguments(lib):
    def rc(wb=ALIGNED, bits=ALIGNED, alpha=ALIGNED, mode=0, n_out=4, n_in=16, out=ALIGNED):
        return lib.bd_reconstruct(wb, bits, alpha, mode, n_out, n_in, out, None)
    assert rc(wb=0) == bd.BD_ERR_INVALID_ARG
    assert rc(out=0) == bd.BD_ERR_INVALID_ARG
    assert rc(mode=2) == bd.BD_ERR_INVALID_ARG
    assert rc(n_out=0) == bd.BD_ERR_INVALID_ARG
    assert rc(n_in=12) == bd.BD_ERR_UNSUPPORTED_SHAPE
    assert rc(out=ALIGNED + 8) == bd.BD_ERR_MISALIGNED
