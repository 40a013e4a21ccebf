"""CPU oracle for y = FP16(x . W^T) + b -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path never does, and the
two share no code: this module compiles ``oracle_linear.c`` with gcc (no
CUDA, no torch) and calls it through ctypes on numpy arrays of binary16 bit
patterns (``np.uint16``).

The arithmetic follows "Tensor Programs, Part 1", section "One Program and
One Numerical Contract" (the proj formula, rules 1 and 2, and the
Figure 1.1 caption): binary32 sum of exact products in ascending k, RN16 of
the sum, then RN16(proj + b[n]).  See ``oracle_linear.c`` for the details
and the pins in ``tests/test_oracle_*.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle_linear.c")
_BUILD = os.path.join(_HERE, "_build")
_LOCK = threading.Lock()
_LIBS: dict[int, ctypes.CDLL] = {}

# gcc flags: no fast-math, no contraction into FMA (an FMA would give the
# same result here because every product is exact, but the plain form is
# what a reader checks), position independent, portable (no -march).
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
          "-fno-fast-math", "-pthread"]


def lib_path(mutation: int = 0) -> str:
    name = "liboracle_linear.so" if mutation == 0 else f"liboracle_linear_mut{mutation}.so"
    return os.path.join(_BUILD, name)


def build(mutation: int = 0, force: bool = False) -> str:
    """Compile the oracle (gcc) into ``oracle/_build``; return the .so path."""
    out = lib_path(mutation)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(_SRC)):
        return out
    os.makedirs(_BUILD, exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", *CFLAGS, f"-DORACLE_MUTATION={int(mutation)}", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _lib(mutation: int = 0) -> ctypes.CDLL:
    with _LOCK:
        lib = _LIBS.get(mutation)
        if lib is None:
            lib = ctypes.CDLL(build(mutation))
            u16p = ctypes.POINTER(ctypes.c_uint16)
            f32p = ctypes.POINTER(ctypes.c_float)
            lib.oracle_linear_f16.argtypes = [u16p, u16p, u16p, u16p, u16p,
                                              ctypes.c_int64, ctypes.c_int64,
                                              ctypes.c_int64, ctypes.c_int]
            lib.oracle_linear_f16.restype = ctypes.c_int
            lib.oracle_f16_to_f32.argtypes = [ctypes.c_uint16]
            lib.oracle_f16_to_f32.restype = ctypes.c_float
            lib.oracle_f32_to_f16_rn.argtypes = [ctypes.c_float]
            lib.oracle_f32_to_f16_rn.restype = ctypes.c_uint16
            lib.oracle_f16_to_f32_array.argtypes = [u16p, f32p, ctypes.c_int64]
            lib.oracle_f16_to_f32_array.restype = None
            lib.oracle_f32_to_f16_rn_array.argtypes = [f32p, u16p, ctypes.c_int64]
            lib.oracle_f32_to_f16_rn_array.restype = None
            _LIBS[mutation] = lib
        return lib


def _u16(a: np.ndarray) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype == np.float16:
        a = a.view(np.uint16)
    if a.dtype != np.uint16:
        raise TypeError("oracle inputs are binary16 bit patterns (uint16 or float16)")
    return np.ascontiguousarray(a)


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def linear_f16(x, w, b, *, nthreads: int | None = None, want_proj: bool = False,
               mutation: int = 0):
    """y = RN16(RN16(sum_k x[m,k] W[n,k]) + b[n]); returns uint16 bit patterns.

    x: [M,K], w: [N,K] ([out_features, in_features]), b: [N]; uint16 bits or
    float16.  With ``want_proj`` also returns proj = RN16(sum).
    """
    x, w, b = _u16(x), _u16(w), _u16(b)
    if x.ndim != 2 or w.ndim != 2 or b.ndim != 1:
        raise ValueError("x [M,K], w [N,K], b [N] expected")
    M, K = x.shape
    N, K2 = w.shape
    if K2 != K or b.shape[0] != N:
        raise ValueError(f"shape mismatch x{x.shape} w{w.shape} b{b.shape}")
    y = np.zeros((M, N), dtype=np.uint16)
    proj = np.zeros((M, N), dtype=np.uint16) if want_proj else None
    nt = default_threads() if nthreads is None else int(nthreads)
    lib = _lib(mutation)
    rc = lib.oracle_linear_f16(_ptr(x, ctypes.c_uint16), _ptr(w, ctypes.c_uint16),
                               _ptr(b, ctypes.c_uint16), _ptr(y, ctypes.c_uint16),
                               _ptr(proj, ctypes.c_uint16) if proj is not None else None,
                               M, N, K, nt)
    if rc != 0:
        raise RuntimeError(f"oracle_linear_f16 returned {rc}")
    return (y, proj) if want_proj else y


def f16_to_f32(h) -> np.ndarray:
    """binary16 bits -> binary32 values (the oracle's own conversion)."""
    h = _u16(h).ravel()
    out = np.empty(h.shape, dtype=np.float32)
    _lib().oracle_f16_to_f32_array(_ptr(h, ctypes.c_uint16), _ptr(out, ctypes.c_float), h.size)
    return out


def f32_to_f16_rn(v) -> np.ndarray:
    """binary32 values -> binary16 bits, ties to even (the oracle's own RN16)."""
    v = np.ascontiguousarray(np.asarray(v, dtype=np.float32)).ravel()
    out = np.empty(v.shape, dtype=np.uint16)
    _lib().oracle_f32_to_f16_rn_array(_ptr(v, ctypes.c_float), _ptr(out, ctypes.c_uint16), v.size)
    return out
