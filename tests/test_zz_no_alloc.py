"""poot_linear_f16_splitk_noalloc: split-K whose partial sums live in the
library's fixed device array.

Its results must be the bits poot_linear_f16_ex gives with the same GEMM
variant and split factor, and must match the CPU oracle under the
contract's rule (bit-exact on small integers, else the 2-ulp rule with the
FP32-accumulation interval).  Two calls in a row (the second reusing the
array the first wrote) are each compared with that entry point and with the
oracle; argument and size errors are checked before any CUDA call.  The
file name keeps it last in collection; it also passes on its own.
"""
import re
from pathlib import Path

import numpy as np
import pytest
import torch

import linear_fp16_gb300 as L
from linear_fp16_gb300 import synth
from tests.parity import check_rows

ROOT = Path(__file__).resolve().parents[1]
X, W, B, Y = 0x1000_0000_0, 0x2000_0000_0, 0x3000_0000_0, 0x4000_0000_0   # never dereferenced
DEV = "cuda:0"


def test_scratch_size_matches_the_header():
    src = (ROOT / "include" / "poot_linear.h").read_text()
    m = re.search(r"#define\s+POOT_NOALLOC_SCRATCH_BYTES\s+\((\d+) \* (\d+) \* (\d+)\)", src)
    assert m is not None
    assert int(m.group(1)) * int(m.group(2)) * int(m.group(3)) == L.NOALLOC_SCRATCH_BYTES


@pytest.mark.parametrize("M,N,K,split_k", [
    (64, 256, 4096, 1),     # below 2
    (64, 256, 4096, 17),    # above 16
    (64, 256, 1000, 3),     # does not divide the 16 K blocks
    (64, 256, 0, 2),        # K == 0
    (1024, 4096, 4096, 2),  # 32 MiB of partial sums
    (256, 4104, 4096, 4),   # one row of 8 columns beyond the array
])
def test_argument_and_size_errors_before_any_cuda_call(M, N, K, split_k):
    assert L.poot_linear_f16_splitk_noalloc(X, W, B, Y, M, N, K, split_k, 0) == L.POOT_ERR_INVALID_ARG


def test_empty_output_is_a_no_op():
    assert L.poot_linear_f16_splitk_noalloc(0, 0, 0, 0, 0, 64, 4096, 2, 0) == L.POOT_OK


def _bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy()


def _run_both(x, w, b, split_k, variant):
    M, K = x.shape
    N = w.shape[0]
    y_na = torch.full((M, N), float("nan"), dtype=torch.float16, device=DEV)
    y_ex = torch.full((M, N), float("nan"), dtype=torch.float16, device=DEV)
    s = torch.cuda.current_stream().cuda_stream
    rc = L.poot_linear_f16_splitk_noalloc(x.data_ptr(), w.data_ptr(), b.data_ptr(), y_na.data_ptr(), M, N, K,
                                          split_k, s)
    assert rc == L.POOT_OK, L.poot_linear_status_string(rc)
    rc = L.poot_linear_f16_ex(x.data_ptr(), w.data_ptr(), b.data_ptr(), y_ex.data_ptr(), M, N, K,
                              L.options(variant, gemm_split_k=split_k), s)
    assert rc == L.POOT_OK, L.poot_linear_status_string(rc)
    return y_na, y_ex


@pytest.mark.gpu
def test_two_calls_in_a_row_match_the_workspace_entry_point():
    cases = [((128, 1024, 4096), 4, "normal", 11), ((64, 2048, 8192), 8, "smallint", 12)]
    outs = []
    for (M, N, K), S, dist, seed in cases:
        xh, wh, bh = synth.make_inputs(M, N, K, dist, seed)
        x, w, b = xh.to(DEV), wh.to(DEV), bh.to(DEV)
        outs.append((_run_both(x, w, b, S, L.VARIANT_GEMM_TMA), (xh, wh, bh), dist == "smallint"))
    torch.cuda.synchronize()
    assert L.poot_linear_device_status(0) == L.POOT_OK
    for (y_na, y_ex), (xh, wh, bh), exact in outs:
        assert not torch.isnan(y_na).any()
        assert np.array_equal(_bits(y_na), _bits(y_ex))
        u16 = lambda t: _bits(t).view(np.uint16)
        ok, rep = check_rows(u16(y_na), u16(xh), u16(wh), u16(bh), exact=exact)
        assert ok, rep


@pytest.mark.gpu
def test_the_array_filled_exactly_and_small_m_on_the_gemm():
    # S * M * N * 4 == the array's size; then M = 8 (on the GEMM, not the GEMV)
    for (M, N, K), S in (((256, 4096, 2048), 4), ((8, 1000, 4096), 16)):
        x, w, b = (t.to(DEV) for t in synth.make_inputs(M, N, K, "normal", 13 + M))
        y_na, y_ex = _run_both(x, w, b, S, L.VARIANT_GEMM_TMA)
        torch.cuda.synchronize()
        assert np.array_equal(_bits(y_na), _bits(y_ex))
    assert L.poot_linear_device_status(0) == L.POOT_OK


@pytest.mark.gpu
def test_ragged_k_takes_the_copy_producers():
    # K = 1002: no TMA for x and W; even K with 4-byte aligned rows -> cp.async
    x, w, b = (t.to(DEV) for t in synth.make_inputs(200, 300, 1002, "smallint", 14))
    y_na, y_ex = _run_both(x, w, b, 2, L.VARIANT_GEMM_CPASYNC)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(y_na), _bits(y_ex))
    assert L.poot_linear_device_status(0) == L.POOT_OK


@pytest.mark.gpu
def test_refused_size_leaves_y_alone():
    x = torch.zeros(256, 2048, dtype=torch.float16, device=DEV)
    w = torch.zeros(4104, 2048, dtype=torch.float16, device=DEV)
    b = torch.zeros(4104, dtype=torch.float16, device=DEV)
    y = torch.full((256, 4104), 7.0, dtype=torch.float16, device=DEV)
    rc = L.poot_linear_f16_splitk_noalloc(x.data_ptr(), w.data_ptr(), b.data_ptr(), y.data_ptr(), 256, 4104, 2048,
                                          4, 0)
    assert rc == L.POOT_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert bool((y == 7.0).all())
