"""ctypes binding of libpoot_linear.so: argument marshalling only.

The functions named like the C entry points (include/poot_linear.h) take raw
device pointers and sizes and return the status code.  ``linear`` is the
tensor-level call: it checks torch tensors, allocates y with torch, and
calls ``poot_linear_f16`` on the current stream.  Every step of the
computation runs in the CUDA library; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

# status codes and variants (mirror include/poot_linear.h)
POOT_OK = 0
POOT_ERR_INVALID_ARG = 1
POOT_ERR_MISALIGNED = 2
POOT_ERR_UNSUPPORTED_DEVICE = 3
POOT_ERR_CUDA = 4
POOT_ERR_DEVICE_TIMEOUT = 5

VARIANT_AUTO = -1
VARIANT_NONE = 0
VARIANT_BIAS_ONLY = 1
VARIANT_GEMV = 2
VARIANT_GEMV_SCALAR = 3
VARIANT_GEMM_TMA = 4
VARIANT_GEMM_CPASYNC = 5
VARIANT_GEMM_REG = 6
VARIANT_GEMM_PACKED = 7
VARIANT_NAMES = {
    VARIANT_NONE: "none", VARIANT_BIAS_ONLY: "bias_only", VARIANT_GEMV: "gemv",
    VARIANT_GEMV_SCALAR: "gemv_scalar", VARIANT_GEMM_TMA: "gemm_tma",
    VARIANT_GEMM_CPASYNC: "gemm_cpasync", VARIANT_GEMM_REG: "gemm_reg", VARIANT_GEMM_PACKED: "gemm_packed",
}
GEMV_MAX_M = 16

# the widened contraction (poot_contract)
DTYPE_F16 = 0
DTYPE_BF16 = 1
EP_ADD = 1
EP_MUL = 2
EP_SILU = 3
EP_GELU_TANH = 4
EP_GELU_ERF = 5
EPILOGUE_MAX_STEPS = 4
NOALLOC_SCRATCH_BYTES = 16 * 1024 * 1024  # POOT_NOALLOC_SCRATCH_BYTES
EP_CODES = {"add": EP_ADD, "mul": EP_MUL, "silu": EP_SILU, "gelu_tanh": EP_GELU_TANH, "gelu_erf": EP_GELU_ERF}



class Options(ctypes.Structure):
    """struct poot_linear_options (include/poot_linear.h)."""
    _fields_ = [("variant", ctypes.c_int), ("gemv_warps_per_row", ctypes.c_int),
                ("gemm_tile_n", ctypes.c_int), ("gemm_group_m", ctypes.c_int),
                ("gemm_k_chunk", ctypes.c_int), ("gemm_cluster", ctypes.c_int),
                ("gemm_split_k", ctypes.c_int)]


def options(variant: int = -1, gemv_warps_per_row: int = 0, gemm_tile_n: int = 0,
            gemm_group_m: int = 0, gemm_k_chunk: int = 0, gemm_cluster: int = 0,
            gemm_split_k: int = 0) -> Options:
    return Options(variant, gemv_warps_per_row, gemm_tile_n, gemm_group_m, gemm_k_chunk, gemm_cluster,
                   gemm_split_k)


class GemmPlan(ctypes.Structure):
    """struct poot_gemm_plan."""
    _fields_ = [(n, ctypes.c_int) for n in ("tile_n", "cluster", "split_k", "k_chunk", "tiles", "ctas")]


class EpilogueStep(ctypes.Structure):
    """struct poot_epilogue_step."""
    _fields_ = [("op", ctypes.c_int), ("operand", ctypes.c_void_p), ("ld", ctypes.c_int64)]


class ContractionSpec(ctypes.Structure):
    """struct poot_contraction_spec."""
    _fields_ = [("dtype", ctypes.c_int), ("out_f32", ctypes.c_int), ("num_steps", ctypes.c_int),
                ("steps", EpilogueStep * EPILOGUE_MAX_STEPS)]


# (name, restype, argtypes) of every exported symbol
_VP = ctypes.c_void_p
_I64 = ctypes.c_int64
EXPORTS = {
    "poot_linear_f16": (ctypes.c_int, [_VP, _VP, _VP, _VP, _I64, _I64, _I64, _VP]),
    "poot_linear_f16_ex": (ctypes.c_int, [_VP, _VP, _VP, _VP, _I64, _I64, _I64,
                                          ctypes.POINTER(Options), _VP]),
    "poot_linear_f16_variant": (ctypes.c_int, [_VP, _VP, _VP, _VP, _I64, _I64, _I64]),
    "poot_linear_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "poot_linear_last_cuda_error": (ctypes.c_char_p, []),
    "poot_linear_device_status": (ctypes.c_int, [_VP]),
    "poot_linear_version": (ctypes.c_int, []),
    "poot_contract": (ctypes.c_int, [_VP, _VP, _VP, _VP, _I64, _I64, _I64, ctypes.POINTER(ContractionSpec),
                                     ctypes.POINTER(Options), _VP]),
    "poot_contract_grouped": (ctypes.c_int, [_VP, _VP, _VP, _VP, _I64, _I64, _I64, _I64,
                                             ctypes.POINTER(ContractionSpec), ctypes.POINTER(Options), _VP]),
    "poot_linear_f16_splitk_noalloc": (ctypes.c_int, [_VP, _VP, _VP, _VP, _I64, _I64, _I64, ctypes.c_int, _VP]),
    "poot_linear_gemm_plan": (ctypes.c_int, [_I64, _I64, _I64, ctypes.c_int, ctypes.POINTER(GemmPlan)]),
    "poot_linear_tp_shard": (ctypes.c_int, [_I64, ctypes.c_int, ctypes.c_int, ctypes.POINTER(_I64),
                                            ctypes.POINTER(_I64)]),
    "poot_linear_gather_columns": (ctypes.c_int, [_VP, _VP, _I64, _I64, ctypes.c_int, _I64, _VP]),
    "poot_linear_f16_finish": (ctypes.c_int, [_VP, _VP, _VP, _I64, _I64, _VP]),
}

_lock = threading.Lock()
_lib = None


class PootLinearError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = f"{where}: {status_string(status)} (status {status})"
        if status == POOT_ERR_CUDA:
            msg += f" [{last_cuda_error()}]"
        super().__init__(msg)


def library_path() -> str:
    return _build.LIB


def load_library(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load (building first if needed) the CUDA library; raise if impossible."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if build_if_missing and not _build.up_to_date():
            _build.build()
        if not os.path.exists(path):
            raise RuntimeError(f"CUDA library missing: {path} (run python -m linear_fp16_gb300.build)")
        lib = ctypes.CDLL(path)
        for name, (res, args) in EXPORTS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


# ---- raw C entry points --------------------------------------------------
def poot_linear_f16(x: int, w: int, b: int, y: int, M: int, N: int, K: int, stream: int) -> int:
    return load_library().poot_linear_f16(x, w, b, y, M, N, K, stream)


def poot_linear_f16_ex(x: int, w: int, b: int, y: int, M: int, N: int, K: int, opts, stream: int) -> int:
    """opts: an Options instance or None (everything automatic)."""
    ref = ctypes.byref(opts) if opts is not None else None
    return load_library().poot_linear_f16_ex(x, w, b, y, M, N, K, ref, stream)


def poot_linear_f16_splitk_noalloc(x: int, w: int, b: int, y: int, M: int, N: int, K: int, split_k: int,
                                   stream: int) -> int:
    """Split-K with its partial sums in the library's fixed device array (no allocation)."""
    return load_library().poot_linear_f16_splitk_noalloc(x, w, b, y, M, N, K, split_k, stream)


def poot_linear_gemm_plan(M: int, N: int, K: int, sm_count: int = 152):
    """(status, plan dict) of the GEMM's automatic tile plan (host only)."""
    p = GemmPlan()
    rc = load_library().poot_linear_gemm_plan(M, N, K, sm_count, ctypes.byref(p))
    return rc, {n: getattr(p, n) for n, _ in GemmPlan._fields_}


def poot_linear_tp_shard(extent: int, world: int, rank: int):
    """(status, begin, end) of rank's shard of an axis of `extent` elements (host only)."""
    b, e = ctypes.c_int64(0), ctypes.c_int64(0)
    rc = load_library().poot_linear_tp_shard(extent, world, rank, ctypes.byref(b), ctypes.byref(e))
    return rc, b.value, e.value


def poot_linear_gather_columns(slots: int, y: int, M: int, N: int, world: int, slot_elems: int,
                               stream: int) -> int:
    """y [M,N] from the column shards in `world` slots of slot_elems elements."""
    return load_library().poot_linear_gather_columns(slots, y, M, N, world, slot_elems, stream)


def poot_linear_f16_finish(S: int, b: int, y: int, M: int, N: int, stream: int) -> int:
    """y = RN16(RN16(S) + b) for an FP32 sum S [M,N]."""
    return load_library().poot_linear_f16_finish(S, b, y, M, N, stream)


def poot_linear_f16_variant(x: int, w: int, b: int, y: int, M: int, N: int, K: int) -> int:
    return load_library().poot_linear_f16_variant(x, w, b, y, M, N, K)


def poot_linear_status_string(status: int) -> str:
    return load_library().poot_linear_status_string(status).decode()


def poot_linear_last_cuda_error() -> str:
    return load_library().poot_linear_last_cuda_error().decode()


def poot_linear_device_status(stream: int) -> int:
    return load_library().poot_linear_device_status(stream)


def poot_linear_version() -> int:
    return load_library().poot_linear_version()


def poot_contract(x: int, w: int, b: int, y: int, M: int, N: int, K: int, spec, opts, stream: int) -> int:
    """spec: a ContractionSpec; opts: an Options instance or None; b may be 0 (no bias)."""
    ref = ctypes.byref(opts) if opts is not None else None
    return load_library().poot_contract(x, w, b or None, y, M, N, K, ctypes.byref(spec), ref, stream)


def poot_contract_grouped(x: int, w: int, b: int, y: int, G: int, M: int, N: int, K: int, spec, opts,
                          stream: int) -> int:
    """G contractions: x [G,M,K], w [G*N,K], b [G*N] (or 0), y [G,M,N]."""
    ref = ctypes.byref(opts) if opts is not None else None
    return load_library().poot_contract_grouped(x, w, b or None, y, G, M, N, K, ctypes.byref(spec), ref, stream)


status_string = poot_linear_status_string
last_cuda_error = poot_linear_last_cuda_error


# ---- tensor-level call ---------------------------------------------------
def _check(t, name, ndim):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != torch.float16:
        raise TypeError(f"{name} must be float16, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def linear(x, w, b, out=None, *, variant: int = VARIANT_AUTO, gemv_warps_per_row: int = 0,
           gemm_tile_n: int = 0, gemm_group_m: int = 0, gemm_k_chunk: int = 0,
           gemm_cluster: int = 0, gemm_split_k: int = 0, stream=None):
    """y = FP16(x . W^T) + b with x [M,K], w [N,K], b [N] fp16 CUDA tensors.

    Runs on ``stream`` (default: the current torch stream of x's device) and
    returns y [M,N] (``out`` if given).  Raises PootLinearError on a status
    other than POOT_OK.
    """
    import torch
    _check(x, "x", 2)
    _check(w, "w", 2)
    _check(b, "b", 1)
    M, K = x.shape
    N, K2 = w.shape
    if K2 != K or b.shape[0] != N:
        raise ValueError(f"shape mismatch: x {tuple(x.shape)}, w {tuple(w.shape)}, b {tuple(b.shape)}")
    dev = x.device
    if w.device != dev or b.device != dev:
        raise ValueError("x, w and b must be on the same device")
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=dev)
    else:
        _check(out, "out", 2)
        if tuple(out.shape) != (M, N) or out.device != dev:
            raise ValueError("out must be [M, N] on x's device")
    with torch.cuda.device(dev):
        s = torch.cuda.current_stream(dev) if stream is None else stream
        rc = poot_linear_f16_ex(x.data_ptr(), w.data_ptr(), b.data_ptr(), out.data_ptr(), M, N, K,
                                options(variant, gemv_warps_per_row, gemm_tile_n, gemm_group_m,
                                        gemm_k_chunk, gemm_cluster, gemm_split_k),
                                s.cuda_stream)
    if rc != POOT_OK:
        raise PootLinearError(rc, "poot_linear_f16")
    return out


poot_linear = linear  # the tensor-level call under its C name's stem


def variant_for(x, w, b, y) -> int:
    """The variant the library would choose for these tensors."""
    M, K = x.shape
    N = w.shape[0]
    return poot_linear_f16_variant(x.data_ptr(), w.data_ptr(), b.data_ptr(), y.data_ptr(), M, N, K)


# ---- tensor-level widened contraction ------------------------------------
def contract(x, w, b=None, out=None, *, out_f32: bool = False, steps=(), gemm_tile_n: int = 0,
             gemm_group_m: int = 0, gemm_k_chunk: int = 0, gemm_cluster: int = 0, gemm_split_k: int = 0,
             variant: int = VARIANT_AUTO, stream=None):
    """The widened contraction (include/poot_linear.h, poot_contract).

    x [M,K], w [N,K] and b [N] (or None) are float16 or bfloat16 CUDA
    tensors of one dtype (the head dtype).  A 3-D x [G,M,K] with w [G*N,K]
    and b [G*N] runs the grouped form (poot_contract_grouped); y is then
    [G,M,N] and step operands [G,M,N].  ``steps``: a sequence of
    "silu", "gelu_tanh", "gelu_erf" or ("add" | "mul", r) with r an [M,N]
    tensor (row pitch from its stride) of the head dtype.  Returns y [M,N]:
    float32 with ``out_f32`` (no steps then), else the head dtype.
    M <= 16 (per group) runs on the GEMV kernels, larger M on the GEMM;
    ``variant`` may force VARIANT_GEMV or a GEMM variant, and the gemm_*
    knobs tune the GEMM (``gemm_split_k``: see include/poot_linear.h).
    """
    import torch
    dt = x.dtype
    if dt not in (torch.float16, torch.bfloat16):
        raise TypeError(f"x must be float16 or bfloat16, got {dt}")
    for name, t in (("x", x), ("w", w)) + ((("b", b),) if b is not None else ()):
        if not isinstance(t, torch.Tensor) or t.dtype != dt or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor of x's dtype")
    grouped = x.dim() == 3
    if x.dim() not in (2, 3) or w.dim() != 2 or x.shape[-1] != w.shape[1]:
        raise ValueError(f"x [M,K] or [G,M,K] and w [N,K] or [G*N,K] expected, got {tuple(x.shape)} "
                         f"{tuple(w.shape)}")
    G = x.shape[0] if grouped else 1
    M, K = x.shape[-2], x.shape[-1]
    if w.shape[0] % G != 0:
        raise ValueError(f"w must hold G = {G} blocks of N rows, got {tuple(w.shape)}")
    N = w.shape[0] // G
    if b is not None and tuple(b.shape) != (G * N,):
        raise ValueError(f"b must be [{'G*' if grouped else ''}N], got {tuple(b.shape)}")
    steps = list(steps)
    if len(steps) > EPILOGUE_MAX_STEPS:
        raise ValueError(f"at most {EPILOGUE_MAX_STEPS} epilogue steps")
    spec = ContractionSpec()
    spec.dtype = DTYPE_BF16 if dt == torch.bfloat16 else DTYPE_F16
    spec.out_f32 = int(bool(out_f32))
    spec.num_steps = len(steps)
    for i, st in enumerate(steps):
        name, operand = (st, None) if isinstance(st, str) else st
        if name not in EP_CODES:
            raise ValueError(f"unknown epilogue step {name!r}")
        spec.steps[i].op = EP_CODES[name]
        if name in ("add", "mul"):
            r = operand
            if (not isinstance(r, torch.Tensor) or r.dtype != dt or not r.is_cuda or r.dim() != x.dim()
                    or tuple(r.shape) != tuple(x.shape[:-1]) + (N,) or r.stride(-1) != 1
                    or (grouped and r.stride(0) != M * r.stride(1))):
                raise ValueError(f"step {name}: a CUDA tensor of x's dtype shaped like y, unit column "
                                 "stride (groups stacked by rows)")
            spec.steps[i].operand = r.data_ptr()
            spec.steps[i].ld = r.stride(-2)
    ydt = torch.float32 if out_f32 else dt
    yshape = tuple(x.shape[:-1]) + (N,)
    if out is None:
        out = torch.empty(yshape, dtype=ydt, device=x.device)
    elif out.dtype != ydt or tuple(out.shape) != yshape or not out.is_contiguous():
        raise ValueError(f"out must be a contiguous {yshape} {ydt} tensor")
    opts = options(variant, 0, gemm_tile_n, gemm_group_m, gemm_k_chunk, gemm_cluster, gemm_split_k)
    bp = b.data_ptr() if b is not None else 0
    with torch.cuda.device(x.device):
        s = torch.cuda.current_stream(x.device) if stream is None else stream
        if grouped:
            rc = poot_contract_grouped(x.data_ptr(), w.data_ptr(), bp, out.data_ptr(), G, M, N, K, spec, opts,
                                       s.cuda_stream)
        else:
            rc = poot_contract(x.data_ptr(), w.data_ptr(), bp, out.data_ptr(), M, N, K, spec, opts, s.cuda_stream)
    if rc != POOT_OK:
        raise PootLinearError(rc, "poot_contract_grouped" if grouped else "poot_contract")
    return out
