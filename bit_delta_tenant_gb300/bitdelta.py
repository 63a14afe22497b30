"""Thin ctypes binding of libbitdelta.so (C ABI in ``include/bitdelta.h``).

Function names match the C entry points.  This module only marshals
arguments: torch tensors become device pointers and sizes, the current torch
CUDA stream is passed as the stream, and a non-zero status raises
``BitDeltaError``.  Every step of the computation runs in the library's CUDA
kernels; there is no fallback, and a missing library is an error.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "lib", "libbitdelta.so")
# the bounds-checked build (``build.build(debug=True)``): load it with load_library(LIB_DEBUG_PATH)
LIB_DEBUG_PATH = os.path.join(_HERE, "lib", "libbitdelta_debug.so")

BD_OK = 0
BD_ERR_INVALID_ARG = 1
BD_ERR_UNSUPPORTED_SHAPE = 2
BD_ERR_MISALIGNED = 3
BD_ERR_WORKSPACE = 4
BD_ERR_CUDA = 5
BD_ERR_DEVICE_TIMEOUT = 6
BD_ERR_BAD_VARIANT_ID = 7
BD_ERR_NO_SPACE = 8
BD_ERR_DEVICE_BOUNDS = 9
BD_ALPHA_SCALAR = 0
BD_ALPHA_PER_ROW = 1
BD_MAX_VARIANTS = 64
BD_NOALLOC_MAX_PARTIALS = 131072
BD_LINEAR_BATCH_MAX = 256
BD_COMPRESS_BATCH_MAX = 4096
BD_COMPRESS_BATCH_PER_LAUNCH = 8
BD_LINEAR_BATCH_PER_LAUNCH = 8
BD_OPT_COMPRESS_FORM = 1
BD_OPT_GROUPED_PATH = 2
BD_OPT_BATCH_KERNEL = 3
BD_OPT_BATCH_SINGLE = 4
BD_OPT_BATCH_GRID = 5
BD_OPT_TEST_STALL = 6
BD_OPT_PREFILL_KERNEL = 7
BD_OPT_PAIR_RING = 8

_lock = threading.Lock()
_lib = None


class LinearDesc(ctypes.Structure):
    """bd_linear_desc: one problem of bd_linear_batch (device pointers and sizes)."""
    _fields_ = [("x", ctypes.c_void_p), ("w_base", ctypes.c_void_p), ("bits", ctypes.c_void_p),
                ("alpha", ctypes.c_void_p), ("y", ctypes.c_void_p), ("m", ctypes.c_int64),
                ("n_out", ctypes.c_int64), ("n_in", ctypes.c_int64), ("alpha_mode", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class CompressDesc(ctypes.Structure):
    """bd_compress_desc: one matrix of bd_compress_batch (device pointers and sizes)."""
    _fields_ = [("w_base", ctypes.c_void_p), ("w_ft", ctypes.c_void_p), ("bits_out", ctypes.c_void_p),
                ("alpha_out", ctypes.c_void_p), ("n_out", ctypes.c_int64), ("n_in", ctypes.c_int64),
                ("alpha_mode", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class BitDeltaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {bd_status_string(status)} (status {status})")


def load_library(path: str | None = None):
    """Open libbitdelta.so (built by ``bit_delta_tenant_gb300.build``); raises if absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"libbitdelta.so not found at {p}; build it with "
                               "`python -m bit_delta_tenant_gb300.build` (nvcc, sm_103a)")
        lib = ctypes.CDLL(p)
        V, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        lib.bd_version.restype = I32
        lib.bd_build_flags.restype = I32
        lib.bd_status_string.argtypes = [I32]
        lib.bd_status_string.restype = ctypes.c_char_p
        lib.bd_set_wait_limit_ns.argtypes = [I64]
        lib.bd_set_wait_limit_ns.restype = I64
        lib.bd_set_linear_path.argtypes = [I32]
        lib.bd_set_linear_path.restype = I32
        lib.bd_reconstruct.argtypes = [V, V, V, I32, I64, I64, V, V]
        lib.bd_reconstruct.restype = I32
        lib.bd_cache_state_size.argtypes = [I32]
        lib.bd_cache_state_size.restype = SZ
        lib.bd_cache_create.argtypes = [V, SZ, I32, V, SZ, ctypes.c_double, I32, ctypes.POINTER(V)]
        lib.bd_cache_create.restype = I32
        lib.bd_cache_destroy.argtypes = [V]
        lib.bd_cache_destroy.restype = I32
        lib.bd_cache_register.argtypes = [V, I32, V, SZ, V, SZ]
        lib.bd_cache_register.restype = I32
        lib.bd_cache_set_pinned.argtypes = [V, I32, I32]
        lib.bd_cache_set_pinned.restype = I32
        lib.bd_cache_acquire.argtypes = [V, I32, ctypes.c_double, V, ctypes.POINTER(V), ctypes.POINTER(V)]
        lib.bd_cache_acquire.restype = I32
        lib.bd_cache_release.argtypes = [V, I32, V]
        lib.bd_cache_release.restype = I32
        lib.bd_cache_get_stats.argtypes = [V, ctypes.POINTER(CacheStats)]
        lib.bd_cache_get_stats.restype = I32
        lib.bd_cache_is_resident.argtypes = [V, I32]
        lib.bd_cache_is_resident.restype = I32
        lib.bd_set_option.argtypes = [I32, I64]
        lib.bd_set_option.restype = I64
        lib.bd_set_weight_prefetch.argtypes = [I32]
        lib.bd_set_weight_prefetch.restype = I32
        lib.bd_get_device_status.argtypes = [V]
        lib.bd_get_device_status.restype = I32
        lib.bd_compress_workspace_size.argtypes = [I64, I64, I32]
        lib.bd_compress_workspace_size.restype = SZ
        lib.bd_compress.argtypes = [V, V, I64, I64, I32, V, V, V, SZ, V]
        lib.bd_compress.restype = I32
        lib.bd_compress_noalloc.argtypes = [V, V, I64, I64, I32, V, V, V]
        lib.bd_compress_noalloc.restype = I32
        lib.bd_linear.argtypes = [V, I64, V, V, V, I32, I64, I64, V, V]
        lib.bd_linear.restype = I32
        lib.bd_compress_batch_workspace_size.argtypes = [ctypes.POINTER(CompressDesc), I32]
        lib.bd_compress_batch_workspace_size.restype = SZ
        lib.bd_compress_batch.argtypes = [ctypes.POINTER(CompressDesc), I32, V, SZ, V]
        lib.bd_compress_batch.restype = I32
        lib.bd_linear_batch_workspace_size.argtypes = [ctypes.POINTER(LinearDesc), I32]
        lib.bd_linear_batch_workspace_size.restype = SZ
        lib.bd_linear_batch.argtypes = [ctypes.POINTER(LinearDesc), I32, V, SZ, V]
        lib.bd_linear_batch.restype = I32
        lib.bd_linear_grouped_workspace_size.argtypes = [I64, I32, I64, I64]
        lib.bd_linear_grouped_workspace_size.restype = SZ
        lib.bd_linear_grouped.argtypes = [V, V, I64, V, V, V, V, I32, I64, I64, V, V, SZ, V]
        lib.bd_linear_grouped.restype = I32
        _lib = lib
        return lib


def _stream(stream=None) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream if hasattr(s, "cuda_stream") else int(s))


def _ptr(t: torch.Tensor | None) -> ctypes.c_void_p:
    if t is None:
        return ctypes.c_void_p(0)
    if not t.is_contiguous():
        raise ValueError("tensors passed to libbitdelta must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _check(rc: int, where: str) -> None:
    if rc != BD_OK:
        raise BitDeltaError(rc, where)


def bd_version() -> int:
    return int(load_library().bd_version())


def bd_build_flags() -> int:
    return int(load_library().bd_build_flags())


def bd_status_string(status: int) -> str:
    return load_library().bd_status_string(int(status)).decode()


def bd_set_wait_limit_ns(limit_ns: int) -> int:
    return int(load_library().bd_set_wait_limit_ns(int(limit_ns)))


def bd_set_linear_path(path: int) -> int:
    return int(load_library().bd_set_linear_path(int(path)))


def bd_set_option(option: int, value: int) -> int:
    """Force one kernel choice (BD_OPT_*); returns the previous value, -1 if rejected."""
    return int(load_library().bd_set_option(int(option), int(value)))


class option:
    """Context manager: bd_set_option(opt, value) inside, the previous value restored after."""

    def __init__(self, opt: int, value: int):
        self.opt, self.value = opt, value

    def __enter__(self):
        self.prev = bd_set_option(self.opt, self.value)
        if self.prev < 0:
            raise ValueError(f"bd_set_option({self.opt}, {self.value}) rejected")
        return self

    def __exit__(self, *exc):
        bd_set_option(self.opt, self.prev)


class CacheStats(ctypes.Structure):
    _fields_ = [("acquires", ctypes.c_int64), ("hits", ctypes.c_int64), ("misses", ctypes.c_int64),
                ("joined", ctypes.c_int64), ("loads", ctypes.c_int64), ("evictions", ctypes.c_int64),
                ("bytes_loaded", ctypes.c_int64), ("resident_bytes", ctypes.c_int64),
                ("resident", ctypes.c_int32), ("in_use", ctypes.c_int32)]


class DeltaCache:
    """Thin owner of a bd_cache: the state buffer (host), the arena (a torch
    tensor on the device, or a host tensor with host_arena=True) and the host
    deltas it registers are kept alive here; every call is the C entry point."""

    def __init__(self, max_variants: int, arena: torch.Tensor, half_life_s: float = 10.0, host_arena: bool = False):
        lib = load_library()
        size = lib.bd_cache_state_size(int(max_variants))
        if size == 0:
            raise ValueError("max_variants out of range")
        self._state = ctypes.create_string_buffer(size)
        self._arena = arena
        self._keep = {}
        self._handle = ctypes.c_void_p()
        self._host = bool(host_arena)
        rc = lib.bd_cache_create(ctypes.addressof(self._state), size, int(max_variants), _ptr(arena),
                                 arena.numel() * arena.element_size(), float(half_life_s), 1 if host_arena else 0,
                                 ctypes.byref(self._handle))
        _check(rc, "bd_cache_create")

    def register(self, variant: int, bits: torch.Tensor, alpha: torch.Tensor) -> None:
        rc = load_library().bd_cache_register(self._handle, int(variant), _ptr(bits), bits.numel(), _ptr(alpha),
                                              alpha.numel() * 4)
        _check(rc, "bd_cache_register")
        self._keep[variant] = (bits, alpha)

    def set_pinned(self, variant: int, pinned: bool) -> None:
        _check(load_library().bd_cache_set_pinned(self._handle, int(variant), 1 if pinned else 0), "bd_cache_set_pinned")

    def acquire(self, variant: int, now_s: float = -1.0, stream=None):
        """(status, bits_ptr, alpha_ptr) -- raw device (or arena) addresses."""
        b, a = ctypes.c_void_p(), ctypes.c_void_p()
        rc = load_library().bd_cache_acquire(self._handle, int(variant), float(now_s), self._s(stream),
                                             ctypes.byref(b), ctypes.byref(a))
        return int(rc), b.value or 0, a.value or 0

    def release(self, variant: int, stream=None) -> int:
        return int(load_library().bd_cache_release(self._handle, int(variant), self._s(stream)))

    def _s(self, stream):
        return ctypes.c_void_p(0) if self._host else _stream(stream)

    def stats(self) -> CacheStats:
        st = CacheStats()
        _check(load_library().bd_cache_get_stats(self._handle, ctypes.byref(st)), "bd_cache_get_stats")
        return st

    def is_resident(self, variant: int) -> bool:
        return bool(load_library().bd_cache_is_resident(self._handle, int(variant)))

    def close(self) -> None:
        if self._handle:
            _check(load_library().bd_cache_destroy(self._handle), "bd_cache_destroy")
            self._handle = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def bd_set_weight_prefetch(enable: int) -> int:
    return int(load_library().bd_set_weight_prefetch(int(enable)))


def bd_get_device_status(stream=None) -> int:
    return int(load_library().bd_get_device_status(_stream(stream)))


def bd_compress_workspace_size(n_out: int, n_in: int, alpha_mode: int) -> int:
    return int(load_library().bd_compress_workspace_size(n_out, n_in, alpha_mode))


def bd_compress(w_base: torch.Tensor, w_ft: torch.Tensor, alpha_mode: int, bits_out: torch.Tensor,
                alpha_out: torch.Tensor, workspace: torch.Tensor, stream=None) -> None:
    """Packed sign bits and alpha of (W_base, W_ft); all tensors on the device."""
    n_out, n_in = w_base.shape
    rc = load_library().bd_compress(_ptr(w_base), _ptr(w_ft), n_out, n_in, int(alpha_mode), _ptr(bits_out),
                                    _ptr(alpha_out), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                    _stream(stream))
    _check(rc, "bd_compress")


def bd_compress_noalloc(w_base: torch.Tensor, w_ft: torch.Tensor, alpha_mode: int, bits_out: torch.Tensor,
                        alpha_out: torch.Tensor, stream=None) -> None:
    """bd_compress without a workspace, for callers that cannot allocate device memory.

    Uses the library's built-in 1 MiB scratch array; shapes needing more partial
    sums than BD_NOALLOC_MAX_PARTIALS raise (status BD_ERR_WORKSPACE).  Calls
    that overlap on the GPU share that array and race: keep them ordered.
    """
    n_out, n_in = w_base.shape
    rc = load_library().bd_compress_noalloc(_ptr(w_base), _ptr(w_ft), n_out, n_in, int(alpha_mode),
                                            _ptr(bits_out), _ptr(alpha_out), _stream(stream))
    _check(rc, "bd_compress_noalloc")


def bd_linear(x: torch.Tensor, w_base: torch.Tensor, bits: torch.Tensor, alpha: torch.Tensor, alpha_mode: int,
              y: torch.Tensor, stream=None) -> None:
    """y[m, n_out] = x[m, n_in] . (W_base + alpha * sign)^T."""
    m = x.shape[0] if x.dim() == 2 else 0
    n_out, n_in = w_base.shape
    rc = load_library().bd_linear(_ptr(x), m, _ptr(w_base), _ptr(bits), _ptr(alpha), int(alpha_mode), n_out, n_in,
                                  _ptr(y), _stream(stream))
    _check(rc, "bd_linear")


def compress_descs(problems) -> ctypes.Array:
    """bd_compress_desc array from (w_base, w_ft, alpha_mode, bits_out, alpha_out) tuples of tensors."""
    arr = (CompressDesc * len(problems))()
    for d, (w_base, w_ft, alpha_mode, bits_out, alpha_out) in zip(arr, problems):
        n_out, n_in = w_base.shape
        d.w_base, d.w_ft, d.bits_out, d.alpha_out = (_ptr(w_base).value, _ptr(w_ft).value, _ptr(bits_out).value,
                                                     _ptr(alpha_out).value)
        d.n_out, d.n_in, d.alpha_mode, d.reserved = n_out, n_in, int(alpha_mode), 0
    return arr


def bd_compress_batch_workspace_size(descs: ctypes.Array) -> int:
    return int(load_library().bd_compress_batch_workspace_size(descs, len(descs)))


def bd_compress_batch(descs: ctypes.Array, workspace: torch.Tensor, stream=None) -> None:
    """Each matrix's (bits, alpha) as bd_compress gives it, several matrices per launch."""
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load_library().bd_compress_batch(descs, len(descs), _ptr(workspace), ws_bytes, _stream(stream))
    _check(rc, "bd_compress_batch")


def linear_descs(problems) -> ctypes.Array:
    """bd_linear_desc array from (x, w_base, bits, alpha, alpha_mode, y) tuples of tensors."""
    arr = (LinearDesc * len(problems))()
    for d, (x, w_base, bits, alpha, alpha_mode, y) in zip(arr, problems):
        n_out, n_in = w_base.shape
        d.x, d.w_base, d.bits, d.alpha, d.y = (_ptr(x).value, _ptr(w_base).value, _ptr(bits).value,
                                               _ptr(alpha).value, _ptr(y).value)
        d.m = x.shape[0] if x.dim() == 2 else 0
        d.n_out, d.n_in, d.alpha_mode, d.reserved = n_out, n_in, int(alpha_mode), 0
    return arr


def bd_linear_batch_workspace_size(descs: ctypes.Array) -> int:
    return int(load_library().bd_linear_batch_workspace_size(descs, len(descs)))


def bd_linear_batch(descs: ctypes.Array, workspace: torch.Tensor | None, stream=None) -> None:
    """Each problem's y = x . (W_base + alpha * sign)^T, independent problems batched per launch.

    `descs` comes from `linear_descs`; `workspace` is a zero-filled device buffer of at
    least `bd_linear_batch_workspace_size(descs)` bytes (left ready for the next call)."""
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load_library().bd_linear_batch(descs, len(descs), _ptr(workspace), ws_bytes, _stream(stream))
    _check(rc, "bd_linear_batch")


def bd_linear_grouped_workspace_size(m: int, n_variants: int, n_out: int, n_in: int) -> int:
    return int(load_library().bd_linear_grouped_workspace_size(m, n_variants, n_out, n_in))


def bd_reconstruct(w_base: torch.Tensor, bits: torch.Tensor, alpha: torch.Tensor, alpha_mode: int,
                   w_eff: torch.Tensor, stream=None) -> None:
    """W_eff = bf16(W_base + alpha * s), materialised (for a standard matmul)."""
    n_out, n_in = w_base.shape
    rc = load_library().bd_reconstruct(_ptr(w_base), _ptr(bits), _ptr(alpha), int(alpha_mode), n_out, n_in,
                                       _ptr(w_eff), _stream(stream))
    _check(rc, "bd_reconstruct")


def bd_linear_grouped(x: torch.Tensor, variant_ids: torch.Tensor, w_base: torch.Tensor, bits_v, alpha_v,
                      alpha_modes_v, y: torch.Tensor, workspace: torch.Tensor, stream=None) -> None:
    """Multi-tenant fused linear: token t uses (bits_v[ids[t]], alpha_v[ids[t]])."""
    n_var = len(bits_v)
    if len(alpha_v) != n_var or len(alpha_modes_v) != n_var:
        raise ValueError("bits_v, alpha_v and alpha_modes_v must have one entry per variant")
    m = x.shape[0]
    n_out, n_in = w_base.shape
    bits_arr = (ctypes.c_void_p * n_var)(*[b.data_ptr() for b in bits_v])
    alpha_arr = (ctypes.c_void_p * n_var)(*[a.data_ptr() for a in alpha_v])
    modes_arr = (ctypes.c_int32 * n_var)(*[int(md) for md in alpha_modes_v])
    rc = load_library().bd_linear_grouped(_ptr(x), _ptr(variant_ids), m, _ptr(w_base), bits_arr, alpha_arr,
                                          modes_arr, n_var, n_out, n_in, _ptr(y), _ptr(workspace),
                                          workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "bd_linear_grouped")
