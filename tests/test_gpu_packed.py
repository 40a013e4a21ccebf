"""GEMM_PACKED: x and W copied into 16-byte-pitched rows, then the TMA GEMM.

The copy keeps every element's bits and the tensor maps bound K, so the
rules are those of the TMA path: bit-exact on small-integer inputs, the
2-ulp rule (FP32-interval fallback) otherwise.  Covers every source
alignment class (row starts 2, 4, 8 or 16-byte aligned; odd K), the
automatic choice, CTA pairs, split-K, the widened and grouped contractions,
a large ragged shape on sampled rows, and stream capture.
"""
import numpy as np
import pytest
import torch

import linear_fp16_gb300 as L
from linear_fp16_gb300 import synth
from tests.test_gpu_contract import _check_f32, _check_head, _inputs, _operand
from tests.test_gpu_parity import _bits, _check, _sample_rows

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _offset_copy(t, off):
    """t copied to the device starting `off` elements into a fresh buffer."""
    buf = torch.zeros(t.numel() + off + 8, dtype=t.dtype, device=DEV)
    v = buf[off:off + t.numel()].view(t.shape)
    v.copy_(t.to(DEV))
    return v


def _run(x, w, b, off_x=0, off_w=0, **kw):
    xd, wd, bd = _offset_copy(x, off_x), _offset_copy(w, off_w), b.to(DEV)
    y = torch.full((x.shape[0], w.shape[0]), float("nan"), dtype=torch.float16, device=DEV)
    v = L.variant_for(xd, wd, bd, y)
    L.linear(xd, wd, bd, y, **kw)
    torch.cuda.synchronize()
    assert L.poot_linear_device_status(0) == L.POOT_OK
    return _bits(y), v


@pytest.mark.parametrize("K", [770, 771, 776, 5, 64])
@pytest.mark.parametrize("off_x,off_w", [(0, 0), (1, 0), (2, 3), (3, 1), (4, 2)])
def test_alignment_classes_exact(K, off_x, off_w):
    x, w, b = synth.make_inputs(300, 200, K, "smallint", 700 + K + 10 * off_x + off_w)
    y, v = _run(x, w, b, off_x, off_w)
    tma_in_place = K % 8 == 0 and off_x % 8 == 0 and off_w % 8 == 0
    assert v == (L.VARIANT_GEMM_TMA if tma_in_place else L.VARIANT_GEMM_PACKED)
    _check(x, w, b, y, exact_ints=True)
    # forced, whatever the alignment
    yp, _ = _run(x, w, b, off_x, off_w, variant=L.VARIANT_GEMM_PACKED)
    assert np.array_equal(yp, y)


def test_ragged_workload_packed_exact_and_normal():
    x, w, b = synth.workload_inputs("ragged_exact")
    y, v = _run(x, w, b)
    assert v == L.VARIANT_GEMM_PACKED
    _check(x, w, b, y, exact_ints=True)
    xn, wn, bn = synth.make_inputs(2047, 1000, 770, "normal", 710)
    _check(xn, wn, bn, _run(xn, wn, bn)[0])


@pytest.mark.parametrize("pair", [1, 2])
@pytest.mark.parametrize("tile_n", [0, 64, 256])
def test_packed_with_pairs_and_tile_widths(pair, tile_n):
    x, w, b = synth.make_inputs(600, 520, 1002, "smallint", 720 + pair + tile_n)
    y, _ = _run(x, w, b, 1, 0, gemm_cluster=pair, gemm_tile_n=tile_n)
    _check(x, w, b, y, exact_ints=True)


@pytest.mark.parametrize("S", [2, 4])
def test_packed_with_split_k(S):
    # K = 4094: 64 K blocks, the last one ragged; forced and automatic split
    x, w, b = synth.make_inputs(128, 1024, 4094, "smallint", 730 + S)
    y, v = _run(x, w, b, gemm_split_k=S)
    assert v == L.VARIANT_GEMM_PACKED
    _check(x, w, b, y, exact_ints=True)
    ya, _ = _run(x, w, b)
    _check(x, w, b, ya, exact_ints=True)


def test_large_ragged_sampled_rows():
    x, w, b = synth.make_inputs(4096, 4096, 4094, "normal", 740)
    y, v = _run(x, w, b, 0, 1)
    assert v == L.VARIANT_GEMM_PACKED
    rows = _sample_rows(4096, 24, 741)
    _check(x, w, b, y, rows=rows)
    assert not np.isnan(y.view(np.float16)).any()


@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_widened_contraction_packed(dt):
    M, N, K = 300, 264, 1001
    x, w, b = _inputs(M, N, K, "smallint", 750, dt)
    r = _operand(M, N, "smallint", 751, dt)
    steps = ["silu", ("mul", r)]
    xd, wd = _offset_copy(x, 1), w.to(DEV)
    y = L.contract(xd, wd, b.to(DEV), steps=[steps[0], ("mul", r.to(DEV))])
    torch.cuda.synchronize()
    _check_head(x, w, b, steps, y.cpu(), dt, exact_sums=True)
    y32 = L.contract(xd, wd, None, out_f32=True, variant=L.VARIANT_GEMM_PACKED)
    torch.cuda.synchronize()
    _check_f32(x, w, None, y32.cpu(), dt, exact_sums=True)
    assert L.poot_linear_device_status(0) == L.POOT_OK


def test_grouped_contraction_packed():
    G, M, N, K = 3, 130, 72, 515
    x = torch.randint(-4, 5, (G, M, K), generator=torch.Generator().manual_seed(760)).half()
    w = torch.randint(-4, 5, (G * N, K), generator=torch.Generator().manual_seed(761)).half()
    b = torch.randint(-4, 5, (G * N,), generator=torch.Generator().manual_seed(762)).half()
    y = L.contract(x.to(DEV), w.to(DEV), b.to(DEV))
    torch.cuda.synchronize()
    for g in range(G):
        _check_head(x[g], w[g * N:(g + 1) * N], b[g * N:(g + 1) * N], [], y[g].cpu(), "f16", exact_sums=True)


def test_stream_capture_packed():
    x, w, b = synth.make_inputs(300, 520, 1002, "smallint", 770)
    xd, wd, bd = _offset_copy(x, 1), w.to(DEV), b.to(DEV)
    y = torch.full((300, 520), float("nan"), dtype=torch.float16, device=DEV)
    L.linear(xd, wd, bd, y)
    torch.cuda.synchronize()
    eager = _bits(y)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        L.linear(xd, wd, bd, y)
    for _ in range(2):
        y.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(_bits(y), eager)
    _check(x, w, b, eager, exact_ints=True)
