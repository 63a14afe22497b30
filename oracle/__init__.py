"""BitDelta oracle: the plain fp64 CPU restatement of the method.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  The product
library (``bit_delta_tenant_gb300``) never imports it, and the two share no
source: the arithmetic lives in ``bd_oracle.c`` (plain C, fp64, no GPU code),
built here with gcc and loaded through ctypes.

Method source: the blog page "BitDelta : servir 14 modèles Zen depuis un seul
cluster GPU" (Hanzo blog).  Sections cited: "Le fondement mathématique"
(delta, sign, alpha), "Architecture de service" (fused reconstruction and the
conceptual ``fused_bitdelta_linear`` listing), "Détails d'infrastructure"
(8 bits per byte, fp32 alpha).

Every function here is pinned by the ``-m "not gpu"`` tests against something
other than itself (brute force, library special cases, closed forms, the
page's printed arithmetic); none is "parity unpinned".

Arrays: bf16 tensors are passed as numpy ``uint16`` bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bd_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libbdoracle.so")
_lock = threading.Lock()
_lib = None

ALPHA_SCALAR = 0
ALPHA_PER_ROW = 1


def build(force: bool = False) -> str:
    """Compile bd_oracle.c into a shared library (gcc, OpenMP, strict IEEE)."""
    os.makedirs(_BUILD, exist_ok=True)
    fresh = os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)
    if fresh and not force:
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        I32 = ctypes.c_int32
        lib.bdo_delta.argtypes = [P, P, I64, P]
        lib.bdo_sign_bits.argtypes = [P, P, I64, I64, P]
        lib.bdo_alpha.argtypes = [P, P, I64, I64, ctypes.c_int, P]
        lib.bdo_unpack_signs.argtypes = [P, I64, I64, P]
        lib.bdo_weff.argtypes = [P, P, P, ctypes.c_int, I64, I64, P]
        lib.bdo_weff_bf16.argtypes = [P, P, P, ctypes.c_int, I64, I64, P]
        lib.bdo_linear.argtypes = [P, I64, P, P, P, ctypes.c_int, I64, I64, P, P]
        lib.bdo_linear_sampled.argtypes = [P, P, P, P, ctypes.c_int, I64, I64, P, P, I64, P, P]
        lib.bdo_linear_grouped.argtypes = [P, P, I64, P, P, P, P, I32, I64, I64, P, P]
        lib.bdo_linear_grouped.restype = ctypes.c_int
        lib.bdo_linear_grouped_sampled.argtypes = [P, P, P, P, P, P, I32, I64, I64, P, P, I64, P, P]
        lib.bdo_linear_grouped_sampled.restype = ctypes.c_int
        lib.bdo_packed_bytes.argtypes = [I64, I64]
        lib.bdo_packed_bytes.restype = I64
        _lib = lib
        return lib


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check_bf16_matrix(w: np.ndarray) -> None:
    if w.dtype != np.uint16 or w.ndim != 2:
        raise TypeError("expected a 2-D uint16 array of bf16 bit patterns")


def delta(w_base: np.ndarray, w_ft: np.ndarray) -> np.ndarray:
    """Delta = W_ft - W_base in fp64 ("Le fondement mathématique")."""
    wb, wf = _c(w_base, np.uint16), _c(w_ft, np.uint16)
    out = np.empty(wb.shape, np.float64)
    _load().bdo_delta(_p(wb), _p(wf), wb.size, _p(out))
    return out


def sign_bits(w_base: np.ndarray, w_ft: np.ndarray) -> np.ndarray:
    """Packed sign bits [n_out, n_in/8] uint8, LSB = lowest d_in, bit=1 iff Delta >= 0."""
    _check_bf16_matrix(w_base)
    n_out, n_in = w_base.shape
    if n_in % 8:
        raise ValueError("n_in must be a multiple of 8 (eight signs per byte)")
    wb, wf = _c(w_base, np.uint16), _c(w_ft, np.uint16)
    out = np.empty((n_out, n_in // 8), np.uint8)
    _load().bdo_sign_bits(_p(wb), _p(wf), n_out, n_in, _p(out))
    return out


def alpha(w_base: np.ndarray, w_ft: np.ndarray, mode: int = ALPHA_SCALAR) -> np.ndarray:
    """alpha = mean|Delta| in fp64: shape [1] (scalar) or [n_out] (per-row)."""
    _check_bf16_matrix(w_base)
    n_out, n_in = w_base.shape
    wb, wf = _c(w_base, np.uint16), _c(w_ft, np.uint16)
    out = np.empty(n_out if mode == ALPHA_PER_ROW else 1, np.float64)
    _load().bdo_alpha(_p(wb), _p(wf), n_out, n_in, int(mode), _p(out))
    return out


def alpha_f32(w_base: np.ndarray, w_ft: np.ndarray, mode: int = ALPHA_SCALAR) -> np.ndarray:
    """alpha rounded once (nearest-even) to the fp32 storage type ("Détails d'infrastructure")."""
    return alpha(w_base, w_ft, mode).astype(np.float32)


def compress(w_base: np.ndarray, w_ft: np.ndarray, mode: int = ALPHA_SCALAR):
    """(bits, alpha_fp32, alpha_fp64) for one matrix."""
    a64 = alpha(w_base, w_ft, mode)
    return sign_bits(w_base, w_ft), a64.astype(np.float32), a64


def unpack_signs(bits: np.ndarray, n_in: int) -> np.ndarray:
    """[n_out, n_in] int8 in {-1, +1} from packed bits."""
    b = _c(bits, np.uint8)
    out = np.empty((b.shape[0], n_in), np.int8)
    _load().bdo_unpack_signs(_p(b), b.shape[0], n_in, _p(out))
    return out


def w_eff(w_base: np.ndarray, bits: np.ndarray, alpha32: np.ndarray, mode: int) -> np.ndarray:
    """W_eff = W_base + alpha * sign in fp64 ("Architecture de service")."""
    wb = _c(w_base, np.uint16)
    n_out, n_in = wb.shape
    b = _c(bits, np.uint8)
    a = _c(alpha32, np.float32)
    out = np.empty((n_out, n_in), np.float64)
    _load().bdo_weff(_p(wb), _p(b), _p(a), int(mode), n_out, n_in, _p(out))
    return out


def w_eff_bf16(w_base: np.ndarray, bits: np.ndarray, alpha32: np.ndarray, mode: int) -> np.ndarray:
    """bf16 bit patterns of W_eff formed in fp32 and rounded once to nearest even (reading R5)."""
    wb = _c(w_base, np.uint16)
    n_out, n_in = wb.shape
    b = _c(bits, np.uint8)
    a = _c(alpha32, np.float32)
    out = np.empty((n_out, n_in), np.uint16)
    _load().bdo_weff_bf16(_p(wb), _p(b), _p(a), int(mode), n_out, n_in, _p(out))
    return out


def linear(x: np.ndarray, w_base: np.ndarray, bits: np.ndarray, alpha32: np.ndarray,
           mode: int):
    """Fused linear y = x . (W_base + alpha*sign)^T in fp64, and sum |x||W_eff| per output."""
    xx = _c(x, np.uint16)
    wb = _c(w_base, np.uint16)
    m, n_in = xx.shape
    n_out = wb.shape[0]
    if wb.shape[1] != n_in:
        raise ValueError("x and W_base disagree on n_in")
    b = _c(bits, np.uint8)
    a = _c(alpha32, np.float32)
    y = np.empty((m, n_out), np.float64)
    mag = np.empty((m, n_out), np.float64)
    _load().bdo_linear(_p(xx), m, _p(wb), _p(b), _p(a), int(mode), n_out, n_in, _p(y), _p(mag))
    return y, mag


def linear_sampled(x, w_base, bits, alpha32, mode, ts, js):
    """Fused linear at the (ts[i], js[i]) outputs only."""
    xx = _c(x, np.uint16)
    wb = _c(w_base, np.uint16)
    n_out, n_in = wb.shape
    b = _c(bits, np.uint8)
    a = _c(alpha32, np.float32)
    t = _c(ts, np.int64)
    j = _c(js, np.int64)
    y = np.empty(t.size, np.float64)
    mag = np.empty(t.size, np.float64)
    _load().bdo_linear_sampled(_p(xx), _p(wb), _p(b), _p(a), int(mode), n_out, n_in,
                               _p(t), _p(j), t.size, _p(y), _p(mag))
    return y, mag


def _ptr_array(arrays):
    ptrs = (ctypes.c_void_p * len(arrays))(*[a.ctypes.data for a in arrays])
    return ptrs


def linear_grouped(x, ids, w_base, bits_v, alpha32_v, modes_v):
    """Multi-tenant fused linear: token t uses variant ids[t]'s (bits, alpha)."""
    xx = _c(x, np.uint16)
    idv = _c(ids, np.int32)
    wb = _c(w_base, np.uint16)
    n_out, n_in = wb.shape
    m = xx.shape[0]
    bl = [_c(b, np.uint8) for b in bits_v]
    al = [_c(a, np.float32) for a in alpha32_v]
    md = _c(modes_v, np.int32)
    y = np.empty((m, n_out), np.float64)
    mag = np.empty((m, n_out), np.float64)
    rc = _load().bdo_linear_grouped(_p(xx), _p(idv), m, _p(wb), _ptr_array(bl), _ptr_array(al),
                                    _p(md), len(bl), n_out, n_in, _p(y), _p(mag))
    if rc != 0:
        raise ValueError("variant id out of range")
    return y, mag


def linear_grouped_sampled(x, ids, w_base, bits_v, alpha32_v, modes_v, ts, js):
    xx = _c(x, np.uint16)
    idv = _c(ids, np.int32)
    wb = _c(w_base, np.uint16)
    n_out, n_in = wb.shape
    bl = [_c(b, np.uint8) for b in bits_v]
    al = [_c(a, np.float32) for a in alpha32_v]
    md = _c(modes_v, np.int32)
    t = _c(ts, np.int64)
    j = _c(js, np.int64)
    y = np.empty(t.size, np.float64)
    mag = np.empty(t.size, np.float64)
    rc = _load().bdo_linear_grouped_sampled(_p(xx), _p(idv), _p(wb), _ptr_array(bl), _ptr_array(al),
                                            _p(md), len(bl), n_out, n_in, _p(t), _p(j), t.size,
                                            _p(y), _p(mag))
    if rc != 0:
        raise ValueError("variant id out of range")
    return y, mag


def packed_bytes(n_out: int, n_in: int) -> int:
    """Bytes of packed sign storage for an [n_out, n_in] matrix."""
    return int(_load().bdo_packed_bytes(n_out, n_in))
