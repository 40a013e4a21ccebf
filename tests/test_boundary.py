"""The C-ABI boundary on the CPU: exports, argument checks, variant choice.

No test here needs a GPU: argument errors are detected before any CUDA
call, and the variant choice is pure host logic.
"""
import os
import re

import pytest

import linear_fp16_gb300 as L
from linear_fp16_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "poot_linear.h")

# fake, far-apart, 256-byte-aligned "device addresses" (never dereferenced)
X, W, B, Y = 0x1000_0000_0, 0x2000_0000_0, 0x3000_0000_0, 0x4000_0000_0


def declared_functions():
    src = open(HEADER).read()
    return re.findall(r"POOT_API\s+[\w\s\*]+?\b(poot_\w+)\s*\(", src)


def test_library_builds_and_loads():
    lib = L.load_library()
    assert os.path.exists(L.library_path())
    assert L.poot_linear_version() == 100
    assert lib is L.load_library()


def test_every_declared_symbol_is_exported_and_bound():
    names = declared_functions()
    assert len(names) == 14, names
    lib = L.load_library()
    for n in names:
        assert hasattr(lib, n), n
        assert n in binding.EXPORTS, n
    assert set(binding.EXPORTS) == set(names)


def test_status_strings():
    for code in range(6):
        s = L.poot_linear_status_string(code)
        assert s and s != "unknown status"
    assert L.poot_linear_status_string(99) == "unknown status"
    assert L.poot_linear_last_cuda_error() == "cudaSuccess"


@pytest.mark.parametrize("M,N,K,want", [
    (1, 4096, 4096, L.VARIANT_GEMV),
    (8, 4096, 4096, L.VARIANT_GEMV),
    (16, 4096, 4096, L.VARIANT_GEMV),
    (17, 4096, 4096, L.VARIANT_GEMM_TMA),
    (1024, 1024, 768, L.VARIANT_GEMM_TMA),
    (2047, 1000, 770, L.VARIANT_GEMM_PACKED),
    (100, 100, 771, L.VARIANT_GEMM_PACKED),
    (3, 10, 771, L.VARIANT_GEMV_SCALAR),
    (3, 10, 0, L.VARIANT_BIAS_ONLY),
    (0, 10, 5, L.VARIANT_NONE),
    (10, 0, 5, L.VARIANT_NONE),
])
def test_variant_choice(M, N, K, want):
    assert L.poot_linear_f16_variant(X, W, B, Y, M, N, K) == want


def test_variant_choice_follows_alignment():
    # 16-byte alignment of x and W selects TMA in place; anything else the
    # packed copies (the copy producers only when forced)
    assert L.poot_linear_f16_variant(X + 4, W, B, Y, 100, 64, 64) == L.VARIANT_GEMM_PACKED
    assert L.poot_linear_f16_variant(X, W + 2, B, Y, 100, 64, 64) == L.VARIANT_GEMM_PACKED
    assert L.poot_linear_f16_variant(X + 8, W, B, Y, 4, 64, 64) == L.VARIANT_GEMV_SCALAR
    # y alignment does not change the load variant (it only picks the store path)
    assert L.poot_linear_f16_variant(X, W, B, Y + 2, 100, 64, 64) == L.VARIANT_GEMM_TMA


@pytest.mark.parametrize("args,code", [
    ((X, W, B, Y, -1, 4, 4), L.POOT_ERR_INVALID_ARG),
    ((X, W, B, Y, 4, -1, 4), L.POOT_ERR_INVALID_ARG),
    ((X, W, B, Y, 4, 4, -1), L.POOT_ERR_INVALID_ARG),
    ((X, W, B, Y, 1 << 31, 4, 4), L.POOT_ERR_INVALID_ARG),
    ((X, W, B, 0, 4, 4, 4), L.POOT_ERR_INVALID_ARG),
    ((X, W, 0, Y, 4, 4, 4), L.POOT_ERR_INVALID_ARG),
    ((0, W, B, Y, 4, 4, 4), L.POOT_ERR_INVALID_ARG),
    ((X, 0, B, Y, 4, 4, 4), L.POOT_ERR_INVALID_ARG),
    ((X + 1, W, B, Y, 4, 4, 4), L.POOT_ERR_MISALIGNED),
    ((X, W + 1, B, Y, 4, 4, 4), L.POOT_ERR_MISALIGNED),
    ((X, W, B + 1, Y, 4, 4, 4), L.POOT_ERR_MISALIGNED),
    ((X, W, B, Y + 1, 4, 4, 4), L.POOT_ERR_MISALIGNED),
    ((X, W, B, X + 8, 4, 4, 4), L.POOT_ERR_INVALID_ARG),     # y overlaps x
    ((X, W, B, W - 16, 4, 4, 4), L.POOT_ERR_INVALID_ARG),    # y runs into W
    ((X, W, B, B, 4, 4, 4), L.POOT_ERR_INVALID_ARG),         # y is b
])
def test_argument_errors_before_any_cuda_call(args, code):
    assert L.poot_linear_f16(*args, 0) == code
    assert L.poot_linear_f16_variant(*args) == -code
    assert L.poot_linear_f16_ex(*args, L.options(), 0) == code
    assert L.poot_linear_f16_ex(*args, None, 0) == code


def test_empty_problems_need_no_pointers_and_no_device():
    assert L.poot_linear_f16(0, 0, 0, 0, 0, 5, 5, 0) == L.POOT_OK
    assert L.poot_linear_f16(0, 0, 0, 0, 5, 0, 5, 0) == L.POOT_OK


def test_k_zero_needs_no_x_or_w():
    assert L.poot_linear_f16_variant(0, 0, B, Y, 3, 4, 0) == L.VARIANT_BIAS_ONLY


@pytest.mark.parametrize("variant,M,K,xoff", [
    (L.VARIANT_GEMV, 17, 64, 0),          # M too large for the GEMV
    (L.VARIANT_GEMV, 4, 66, 0),           # K % 8 != 0
    (L.VARIANT_GEMM_TMA, 100, 64, 4),     # x not 16-byte aligned
    (L.VARIANT_GEMM_CPASYNC, 100, 65, 0), # odd K
    (L.VARIANT_BIAS_ONLY, 100, 64, 0),    # K != 0
    (L.VARIANT_NONE, 100, 64, 0),         # not empty
    (8, 100, 64, 0),                      # unknown
    (-2, 100, 64, 0),                     # unknown
])
def test_inapplicable_forced_variant_is_rejected(variant, M, K, xoff):
    assert L.poot_linear_f16_ex(X + xoff, W, B, Y, M, 64, K, L.options(variant), 0) == L.POOT_ERR_INVALID_ARG


@pytest.mark.parametrize("wpr", [3, 5, 16, -1])
def test_bad_gemv_warps_per_row(wpr):
    assert L.poot_linear_f16_ex(X, W, B, Y, 4, 64, 64, L.options(gemv_warps_per_row=wpr), 0) == \
        L.POOT_ERR_INVALID_ARG


@pytest.mark.parametrize("tile_n", [32, 48, 100, 288, -64])
def test_bad_gemm_tile_width(tile_n):
    assert L.poot_linear_f16_ex(X, W, B, Y, 400, 64, 64, L.options(gemm_tile_n=tile_n), 0) == \
        L.POOT_ERR_INVALID_ARG


@pytest.mark.parametrize("chunk", [-64, 32, 100])
def test_bad_gemm_k_chunk(chunk):
    assert L.poot_linear_f16_ex(X, W, B, Y, 400, 64, 64, L.options(gemm_k_chunk=chunk), 0) == \
        L.POOT_ERR_INVALID_ARG


@pytest.mark.parametrize("cluster", [-1, 3, 4, 8])
def test_bad_gemm_cluster(cluster):
    assert L.poot_linear_f16_ex(X, W, B, Y, 400, 64, 64, L.options(gemm_cluster=cluster), 0) == \
        L.POOT_ERR_INVALID_ARG


@pytest.mark.parametrize("split", [-1, 17])
def test_bad_gemm_split_k(split):
    assert L.poot_linear_f16_ex(X, W, B, Y, 400, 64, 2048, L.options(gemm_split_k=split), 0) == \
        L.POOT_ERR_INVALID_ARG
    assert L.poot_contract(X, W, B, Y, 400, 64, 2048, _spec(), L.options(gemm_split_k=split), 0) == \
        L.POOT_ERR_INVALID_ARG


def test_split_k_refused_with_groups():
    assert L.poot_contract_grouped(X, W, B, Y, 2, 400, 64, 2048, _spec(), L.options(gemm_split_k=2), 0) == \
        L.POOT_ERR_INVALID_ARG


def test_cluster_needs_the_tma_variant():
    assert L.poot_linear_f16_ex(X, W, B, Y, 400, 64, 64,
                                L.options(L.VARIANT_GEMM_CPASYNC, gemm_cluster=2), 0) == L.POOT_ERR_INVALID_ARG


def test_bad_gemm_group():
    assert L.poot_linear_f16_ex(X, W, B, Y, 400, 64, 64, L.options(gemm_group_m=-1), 0) == \
        L.POOT_ERR_INVALID_ARG


def test_no_device_is_a_cuda_error_not_a_crash():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert L.poot_linear_f16(X, W, B, Y, 4, 64, 64, 0) == L.POOT_ERR_CUDA
    assert L.poot_linear_last_cuda_error() != "cudaSuccess"


def test_tensor_call_checks_types():
    import torch
    x = torch.zeros(2, 3, dtype=torch.float16)
    with pytest.raises(ValueError):
        L.linear(x, x, torch.zeros(2, dtype=torch.float16))  # CPU tensors are refused
    with pytest.raises(TypeError):
        L.linear(x.float(), x, torch.zeros(2, dtype=torch.float16))


# ---- the widened contraction (poot_contract) ------------------------------------
R = 0x5000_0000_0  # fake epilogue operand


def _spec(dtype=L.DTYPE_F16, out_f32=0, steps=()):
    sp = L.ContractionSpec()
    sp.dtype, sp.out_f32, sp.num_steps = dtype, out_f32, len(steps)
    for i, (op, ptr, ld) in enumerate(steps):
        sp.steps[i].op, sp.steps[i].operand, sp.steps[i].ld = op, ptr, ld
    return sp


@pytest.mark.parametrize("spec,args,code", [
    (_spec(dtype=2), (X, W, B, Y, 4, 4, 4), L.POOT_ERR_INVALID_ARG),
    (_spec(out_f32=2), (X, W, B, Y, 4, 4, 4), L.POOT_ERR_INVALID_ARG),
    (_spec(out_f32=1, steps=[(L.EP_SILU, 0, 0)]), (X, W, B, Y, 4, 4, 4), L.POOT_ERR_INVALID_ARG),
    (_spec(steps=[(9, 0, 0)]), (X, W, B, Y, 4, 4, 4), L.POOT_ERR_INVALID_ARG),
    (_spec(steps=[(L.EP_ADD, 0, 0)]), (X, W, B, Y, 4, 4, 4), L.POOT_ERR_INVALID_ARG),   # no operand
    (_spec(steps=[(L.EP_MUL, R, 3)]), (X, W, B, Y, 4, 4, 4), L.POOT_ERR_INVALID_ARG),   # ld < N
    (_spec(steps=[(L.EP_MUL, R + 1, 0)]), (X, W, B, Y, 4, 4, 4), L.POOT_ERR_MISALIGNED),
    (_spec(steps=[(L.EP_ADD, Y + 8, 0)]), (X, W, B, Y, 4, 4, 4), L.POOT_ERR_INVALID_ARG),  # overlaps y
    (_spec(), (X, W, B, Y, 4, 4, 0), L.POOT_ERR_INVALID_ARG),                          # K == 0
    (_spec(), (0, W, B, Y, 4, 4, 4), L.POOT_ERR_INVALID_ARG),
    (_spec(), (X, W, B, Y + 1, 4, 4, 4), L.POOT_ERR_MISALIGNED),
    (_spec(out_f32=1), (X, W, B, Y + 2, 4, 4, 4), L.POOT_ERR_MISALIGNED),             # float32 y
    (_spec(), (X, W, B + 1, Y, 4, 4, 4), L.POOT_ERR_MISALIGNED),
    (_spec(), (X, W, B, X + 8, 4, 4, 4), L.POOT_ERR_INVALID_ARG),                     # y overlaps x
])
def test_contract_argument_errors_before_any_cuda_call(spec, args, code):
    assert L.poot_contract(*args, spec, None, 0) == code


def test_contract_rejects_clusters_of_four_and_inapplicable_gemv_variants():
    assert L.poot_contract(X, W, B, Y, 400, 64, 64, _spec(), L.options(gemm_cluster=4), 0) == L.POOT_ERR_INVALID_ARG
    # the scalar GEMV never serves the contraction; the vector GEMV only for
    # M <= 16 with 16-byte aligned x and W and K % 8 == 0
    assert L.poot_contract(X, W, B, Y, 4, 64, 64, _spec(), L.options(L.VARIANT_GEMV_SCALAR), 0) == \
        L.POOT_ERR_INVALID_ARG
    assert L.poot_contract(X, W, B, Y, 17, 64, 64, _spec(), L.options(L.VARIANT_GEMV), 0) == L.POOT_ERR_INVALID_ARG
    assert L.poot_contract(X, W, B, Y, 4, 64, 66, _spec(), L.options(L.VARIANT_GEMV), 0) == L.POOT_ERR_INVALID_ARG
    assert L.poot_contract(X + 2, W, B, Y, 4, 64, 64, _spec(), L.options(L.VARIANT_GEMV), 0) == \
        L.POOT_ERR_INVALID_ARG


def test_contract_null_spec_and_empty_problems():
    lib = L.load_library()
    assert lib.poot_contract(X, W, B, Y, 4, 4, 4, None, None, 0) == L.POOT_ERR_INVALID_ARG
    assert L.poot_contract(0, 0, 0, 0, 0, 5, 5, _spec(), None, 0) == L.POOT_OK


def test_contract_bias_is_optional():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    # passes every check and reaches the device query, which fails without a GPU
    assert L.poot_contract(X, W, 0, Y, 4, 64, 64, _spec(), None, 0) == L.POOT_ERR_CUDA


def test_grouped_argument_errors():
    sp = _spec()
    assert L.poot_contract_grouped(X, W, B, Y, 0, 4, 4, 4, sp, None, 0) == L.POOT_ERR_INVALID_ARG
    assert L.poot_contract_grouped(X, W, B, Y, 1 << 20, 1 << 12, 4, 4, sp, None, 0) == L.POOT_ERR_INVALID_ARG
    # y of 3 groups runs into W when the groups are counted
    assert L.poot_contract_grouped(X, W, B, W - 3 * 4 * 4 * 2 + 2, 3, 4, 4, 4, sp, None, 0) == \
        L.POOT_ERR_INVALID_ARG
    assert L.poot_contract_grouped(0, 0, 0, 0, 3, 0, 4, 4, sp, None, 0) == L.POOT_OK


def _header_constants():
    """Every `NAME = value` enumerator and `#define NAME value` of the header."""
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    vals = {m.group(1): int(m.group(2)) for m in re.finditer(r"\b(POOT_[A-Z0-9_]+)\s*=\s*(-?\d+)", src)}
    for m in re.finditer(r"#define\s+(POOT_[A-Z0-9_]+)\s+\(?(-?\d+)\)?\s*$", src, flags=re.M):
        vals[m.group(1)] = int(m.group(2))
    return vals


def test_binding_constants_match_the_header():
    vals = _header_constants()
    mirrors = {name: name[len("POOT_"):] for name in vals}
    mirrors.update({n: n for n in vals if n.startswith("POOT_OK") or n.startswith("POOT_ERR_")})
    checked = 0
    for cname, pyname in mirrors.items():
        if hasattr(binding, pyname):
            assert getattr(binding, pyname) == vals[cname], (cname, pyname)
            checked += 1
    # every status, variant, dtype and step code, and the two size constants
    for cname in vals:
        if cname.startswith(("POOT_ERR_", "POOT_VARIANT_", "POOT_DTYPE_", "POOT_EP_")) or cname == "POOT_OK":
            assert hasattr(binding, mirrors[cname]), cname
    assert binding.GEMV_MAX_M == vals["POOT_GEMV_MAX_M"]
    assert binding.EPILOGUE_MAX_STEPS == vals["POOT_EPILOGUE_MAX_STEPS"]
    assert checked == len(vals)  # every enumerator and size constant has its mirror
