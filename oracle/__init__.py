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

``contraction`` widens it (``oracle_contraction.c``): a bfloat16 head, no
bias, FP32 output without the head rounding, and epilogue steps (add or
multiply an [M,N] tensor, SiLU, GELU in its tanh and erf forms) of which
every primitive rounds to the head dtype ("ML compiler internals", the
ContractionEpilogue and DenseContraction rows of the OpKind table and the
section "SwiGLU and GeLU FFN").
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle_linear.c")
_SRCS = [_SRC, os.path.join(_HERE, "oracle_contraction.c")]
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
            and all(os.path.getmtime(out) >= os.path.getmtime(src) for src in _SRCS)):
        return out
    os.makedirs(_BUILD, exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", *CFLAGS, f"-DORACLE_MUTATION={int(mutation)}", *_SRCS, "-lm", "-o", tmp]
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
            f64p = ctypes.POINTER(ctypes.c_double)
            i32p = ctypes.POINTER(ctypes.c_int)
            i64p = ctypes.POINTER(ctypes.c_int64)
            u16pp = ctypes.POINTER(u16p)
            lib.oracle_contraction.argtypes = [u16p, u16p, u16p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                               u16p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                               ctypes.c_int, i32p, u16pp, i64p, ctypes.c_int]
            lib.oracle_contraction.restype = ctypes.c_int
            lib.oracle_epilogue.argtypes = [u16p, u16p, ctypes.c_int, u16p, ctypes.c_int64, ctypes.c_int64,
                                            ctypes.c_int, i32p, u16pp, i64p, ctypes.c_int]
            lib.oracle_epilogue.restype = ctypes.c_int
            lib.oracle_f64_to_f16_rn_array.argtypes = [f64p, u16p, ctypes.c_int64]
            lib.oracle_f64_to_f16_rn_array.restype = None
            lib.oracle_f64_to_bf16_rn_array.argtypes = [f64p, u16p, ctypes.c_int64]
            lib.oracle_f64_to_bf16_rn_array.restype = None
            lib.oracle_bf16_to_f32_array.argtypes = [u16p, f32p, ctypes.c_int64]
            lib.oracle_bf16_to_f32_array.restype = None
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


# ---- the widened contraction (oracle_contraction.c) ---------------------------
DTYPES = {"f16": 0, "bf16": 1}
STEP_OPS = {"add": 1, "mul": 2, "silu": 3, "gelu_tanh": 4, "gelu_erf": 5}


def _u16any(a) -> np.ndarray:
    """binary16 / bfloat16 bit patterns as uint16 (float16 arrays are viewed)."""
    a = np.asarray(a)
    if a.dtype == np.float16:
        a = a.view(np.uint16)
    if a.dtype != np.uint16:
        raise TypeError("head-dtype inputs are bit patterns (uint16), or float16 for binary16")
    return np.ascontiguousarray(a)


def _steps(steps, M, N):
    """(ops, operand pointer array, lds, keep-alive list) for the C call."""
    steps = list(steps)
    ops = (ctypes.c_int * max(1, len(steps)))()
    ptrs = (ctypes.POINTER(ctypes.c_uint16) * max(1, len(steps)))()
    lds = (ctypes.c_int64 * max(1, len(steps)))()
    keep = []
    for i, st in enumerate(steps):
        name, operand = (st, None) if isinstance(st, str) else st
        if name not in STEP_OPS:
            raise ValueError(f"unknown epilogue step {name!r}")
        ops[i] = STEP_OPS[name]
        if name in ("add", "mul"):
            r = _u16any(operand)
            if r.ndim != 2 or r.shape[0] != M or r.shape[1] < N:
                raise ValueError(f"step {name}: operand [M, >=N] expected, got {r.shape}")
            keep.append(r)
            ptrs[i] = _ptr(r, ctypes.c_uint16)
            lds[i] = r.shape[1]
        else:
            lds[i] = N
    return len(steps), ops, ptrs, lds, keep


def contraction(x, w, b=None, *, dtype: str = "f16", out_f32: bool = False, steps=(),
                want_proj: bool = False, nthreads: int | None = None, mutation: int = 0):
    """The widened contraction; returns head-dtype bits (uint16) or float32 values.

    x [M,K], w [N,K] ([out, in], read in place), b [N] or None, all bit
    patterns of the head dtype ("f16" or "bf16").  ``out_f32``: y is the
    binary32 sum (+ b in binary32), no head rounding and no steps.
    ``steps``: sequence of "silu" / "gelu_tanh" / "gelu_erf" or
    ("add" | "mul", operand [M,N] bits).  ``want_proj`` also returns RN_h of
    the sum.
    """
    if dtype not in DTYPES:
        raise ValueError(f"dtype must be one of {list(DTYPES)}")
    x, w = _u16any(x), _u16any(w)
    if x.ndim != 2 or w.ndim != 2 or x.shape[1] != w.shape[1]:
        raise ValueError(f"x [M,K] and w [N,K] expected, got {x.shape} {w.shape}")
    M, K = x.shape
    N = w.shape[0]
    bb = None if b is None else _u16any(b)
    if bb is not None and (bb.ndim != 1 or bb.shape[0] != N):
        raise ValueError(f"b [N] expected, got {bb.shape}")
    ns, ops, ptrs, lds, keep = _steps(steps, M, N)
    if out_f32 and ns:
        raise ValueError("the FP32 output takes no epilogue steps")
    y = np.zeros((M, N), dtype=np.float32 if out_f32 else np.uint16)
    proj = np.zeros((M, N), dtype=np.uint16) if (want_proj and not out_f32) else None
    nt = default_threads() if nthreads is None else int(nthreads)
    rc = _lib(mutation).oracle_contraction(
        _ptr(x, ctypes.c_uint16), _ptr(w, ctypes.c_uint16),
        _ptr(bb, ctypes.c_uint16) if bb is not None else None, DTYPES[dtype], int(bool(out_f32)),
        y.ctypes.data_as(ctypes.c_void_p), _ptr(proj, ctypes.c_uint16) if proj is not None else None,
        M, N, K, ns, ops, ptrs, lds, nt)
    if rc != 0:
        raise RuntimeError(f"oracle_contraction returned {rc}")
    return (y, proj) if want_proj else y


def epilogue(t, b=None, *, dtype: str = "f16", steps=(), nthreads: int | None = None, mutation: int = 0):
    """steps(RN_h(t + b[n])) for head values t [M,N] (bits); returns bits."""
    t = _u16any(t)
    M, N = t.shape
    bb = None if b is None else _u16any(b)
    ns, ops, ptrs, lds, keep = _steps(steps, M, N)
    y = np.zeros((M, N), dtype=np.uint16)
    nt = default_threads() if nthreads is None else int(nthreads)
    rc = _lib(mutation).oracle_epilogue(_ptr(t, ctypes.c_uint16),
                                        _ptr(bb, ctypes.c_uint16) if bb is not None else None,
                                        DTYPES[dtype], _ptr(y, ctypes.c_uint16), M, N, ns, ops, ptrs, lds, nt)
    if rc != 0:
        raise RuntimeError(f"oracle_epilogue returned {rc}")
    return y


def f64_to_f16_rn(v, mutation: int = 0) -> np.ndarray:
    """binary64 values -> binary16 bits, ties to even (one rounding)."""
    v = np.ascontiguousarray(np.asarray(v, dtype=np.float64)).ravel()
    out = np.empty(v.shape, dtype=np.uint16)
    _lib(mutation).oracle_f64_to_f16_rn_array(_ptr(v, ctypes.c_double), _ptr(out, ctypes.c_uint16), v.size)
    return out


def f64_to_bf16_rn(v, mutation: int = 0) -> np.ndarray:
    """binary64 values -> bfloat16 bits, ties to even (one rounding)."""
    v = np.ascontiguousarray(np.asarray(v, dtype=np.float64)).ravel()
    out = np.empty(v.shape, dtype=np.uint16)
    _lib(mutation).oracle_f64_to_bf16_rn_array(_ptr(v, ctypes.c_double), _ptr(out, ctypes.c_uint16), v.size)
    return out


def bf16_to_f32(h) -> np.ndarray:
    """bfloat16 bits -> binary32 values (exact)."""
    h = _u16any(h).ravel()
    out = np.empty(h.shape, dtype=np.float32)
    _lib().oracle_bf16_to_f32_array(_ptr(h, ctypes.c_uint16), _ptr(out, ctypes.c_float), h.size)
    return out


def contraction_grouped(x, w, b=None, *, dtype: str = "f16", out_f32: bool = False, steps=(),
                        nthreads: int | None = None):
    """G independent contractions ("ML compiler internals", the
    GroupedDenseContraction row): x [G,M,K], w [G*N,K] read as G blocks of
    N rows, b [G*N] or None, step operands [G,M,N]; y [G,M,N].  Each group
    is ``contraction`` of its own blocks."""
    x = _u16any(x)
    if x.ndim != 3:
        raise ValueError("x [G,M,K] expected")
    G = x.shape[0]
    w = _u16any(w)
    if w.shape[0] % G:
        raise ValueError("w must hold G blocks of N rows")
    N = w.shape[0] // G
    outs = []
    for g in range(G):
        st = [s if isinstance(s, str) else (s[0], _u16any(s[1])[g]) for s in steps]
        bg = None if b is None else _u16any(b)[g * N:(g + 1) * N]
        outs.append(contraction(x[g], w[g * N:(g + 1) * N], bg, dtype=dtype, out_f32=out_f32, steps=st,
                                nthreads=nthreads))
    return np.stack(outs)
