"""The widened contraction for M <= 16 on the GEMV kernels, on a GPU.

Same rules as the GEMM forms (bit-exact head, bias and ADD / MUL on exact
sums, activations within a few ulps, the hull otherwise, the FP32 bound for
FP32 output).  On exact sums the GEMV result must also equal the GEMM's bit
for bit.  Covers both GEMV kernels (warp per row for M <= 2, tensor-core
tiles for 3 <= M <= 16, 8 or 16 warps), both head dtypes, every form.
"""
import numpy as np
import pytest
import torch

import linear_fp16_gb300 as L
from tests.test_gpu_contract import _check_f32, _check_head, _gpu, _inputs, _operand

pytestmark = pytest.mark.gpu
MS = [1, 2, 3, 8, 9, 16]
FORMS = {
    "bias": [],
    "silu_mul": ["silu", ("mul", None)],
    "add_gelu": [("add", None), "gelu_tanh"],
    "gelu_erf": ["gelu_erf"],
}


def _steps(form, M, N, dist, seed, dt):
    out = []
    for i, st in enumerate(FORMS[form]):
        out.append(st if isinstance(st, str) else (st[0], _operand(M, N, dist, seed + i, dt)))
    return out


@pytest.mark.parametrize("dt", ["f16", "bf16"])
@pytest.mark.parametrize("M", MS)
@pytest.mark.parametrize("form", sorted(FORMS))
def test_gemv_forms_exact(dt, M, form):
    N, K = 520, 1024
    x, w, b = _inputs(M, N, K, "smallint", 1200 + M, dt)
    steps = _steps(form, M, N, "smallint", 1300 + M, dt)
    y = _gpu(x, w, b, steps=steps)
    _check_head(x, w, b, steps, y, dt, exact_sums=True)
    y_gemm = _gpu(x, w, b, steps=steps, variant=L.VARIANT_GEMM_TMA)
    assert torch.equal(y.view(torch.int16), y_gemm.view(torch.int16))
    y_forced = _gpu(x, w, b, steps=steps, variant=L.VARIANT_GEMV)
    assert torch.equal(y.view(torch.int16), y_forced.view(torch.int16))


@pytest.mark.parametrize("dt", ["f16", "bf16"])
@pytest.mark.parametrize("M", [1, 5, 16])
def test_gemv_no_bias_and_f32_output(dt, M):
    N, K = 4104, 2048   # enough 16-row tiles for the 8-warp tensor-core GEMV
    x, w, b = _inputs(M, N, K, "smallint", 1400 + M, dt)
    _check_head(x, w, None, [], _gpu(x, w, None), dt, exact_sums=True)
    _check_f32(x, w, b, _gpu(x, w, b, out_f32=True), dt, exact_sums=True)
    _check_f32(x, w, None, _gpu(x, w, None, out_f32=True), dt, exact_sums=True)


@pytest.mark.parametrize("dt", ["f16", "bf16"])
@pytest.mark.parametrize("M", [1, 8])
def test_gemv_normal_inputs(dt, M):
    N, K = 4096, 4096
    x, w, b = _inputs(M, N, K, "normal", 1500 + M, dt)
    r = _operand(M, N, "normal", 1501, dt)
    steps = ["silu", ("mul", r)]
    _check_head(x, w, b, steps, _gpu(x, w, b, steps=steps), dt, exact_sums=False)
    _check_f32(x, w, b, _gpu(x, w, b, out_f32=True), dt, exact_sums=False)


def test_gemv_variant_refused_where_it_does_not_apply():
    x, w, b = _inputs(17, 64, 64, "smallint", 1600, "f16")
    with pytest.raises(L.PootLinearError):
        _gpu(x, w, b, variant=L.VARIANT_GEMV)   # M > 16
    x, w, b = _inputs(4, 64, 66, "smallint", 1601, "f16")
    with pytest.raises(L.PootLinearError):
        _gpu(x, w, b, variant=L.VARIANT_GEMV)   # K % 8 != 0


@pytest.mark.parametrize("dt", ["f16", "bf16"])
@pytest.mark.parametrize("G,M", [(3, 1), (4, 2), (2, 8), (5, 16)])
def test_grouped_gemv_exact(dt, G, M):
    # small M per group (one token per expert and the like) on the GEMV,
    # against the grouped GEMM bit for bit and the oracle per group
    N, K = 264, 512
    tdt = torch.bfloat16 if dt == "bf16" else torch.float16
    gen = torch.Generator().manual_seed(1700 + G * 31 + M)
    x = torch.randint(-4, 5, (G, M, K), generator=gen).to(tdt)
    w = torch.randint(-4, 5, (G * N, K), generator=gen).to(tdt)
    b = torch.randint(-4, 5, (G * N,), generator=gen).to(tdt)
    r = torch.randint(-4, 5, (G, M, N), generator=gen).to(tdt)
    dev = "cuda:0"
    steps = ["silu", ("mul", r.to(dev))]
    y = L.contract(x.to(dev), w.to(dev), b.to(dev), steps=steps)
    y_gemm = L.contract(x.to(dev), w.to(dev), b.to(dev), steps=steps, variant=L.VARIANT_GEMM_TMA)
    torch.cuda.synchronize()
    assert L.poot_linear_device_status(0) == L.POOT_OK
    assert torch.equal(y.view(torch.int16), y_gemm.view(torch.int16))
    for g in range(G):
        _check_head(x[g], w[g * N:(g + 1) * N], b[g * N:(g + 1) * N], ["silu", ("mul", r[g])], y[g].cpu(), dt,
                    exact_sums=True)
