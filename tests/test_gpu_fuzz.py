"""Seeded random sweep over shapes, pointer offsets and options, on a GPU.

Every case draws small-integer inputs, so all FP32 partial sums are exact and
the result must equal the oracle's bit for bit whatever kernel, tile plan,
split or packing the library picks.  The draws cover M from 1 (GEMV) to a few
hundred (GEMM, CTA pairs), ragged N and K, x / W / y offsets that break 16-,
8- and 4-byte alignment, forced variants, tile widths, split factors and the
widened forms (bfloat16 head, no bias, FP32 output, ADD / MUL / activation
steps).
"""
import numpy as np
import pytest
import torch

import linear_fp16_gb300 as L
import oracle
from linear_fp16_gb300 import synth
from tests.test_gpu_contract import _check_f32, _check_head
from tests.test_gpu_parity import _bits

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
CASES = 160


def _on_device(t, off):
    """t copied into a fresh device buffer starting `off` elements in."""
    buf = torch.zeros(t.numel() + off + 8, dtype=t.dtype, device=DEV)
    v = buf[off:off + t.numel()].view(t.shape)
    v.copy_(t.to(DEV))
    return v


def _draw(rng):
    M = int(rng.choice([1, 2, 3, 5, 8, 13, 16, 17, 64, 127, 128, 129, 200, 256, 300, 513]))
    N = int(rng.integers(1, 600))
    K = int(rng.choice([int(rng.integers(1, 200)), int(rng.integers(200, 3000)), 64 * int(rng.integers(1, 40))]))
    offs = [int(rng.choice([0, 0, 0, 1, 2, 4])) for _ in range(3)]
    return M, N, K, offs


@pytest.mark.parametrize("case", range(CASES))
def test_random_linear_exact(case):
    rng = np.random.default_rng(7000 + case)
    M, N, K, (ox, ow, oy) = _draw(rng)
    x, w, b = synth.make_inputs(M, N, K, "smallint", 7100 + case)
    xd, wd, bd = _on_device(x, ox), _on_device(w, ow), b.to(DEV)
    ybuf = torch.full((M * N + oy + 8,), float("nan"), dtype=torch.float16, device=DEV)
    yd = ybuf[oy:oy + M * N].view(M, N)
    kw = {}
    r = rng.random()
    if M > L.GEMV_MAX_M and r < 0.3:
        kw["gemm_tile_n"] = int(rng.choice([64, 96, 128, 160, 192, 224, 256]))
    elif M > L.GEMV_MAX_M and r < 0.5:
        nkb = -(-K // 64)
        divs = [s for s in (2, 3, 4, 8) if nkb % s == 0]
        if divs:
            kw["gemm_split_k"] = int(rng.choice(divs))
    elif r < 0.6:
        kw["variant"] = L.VARIANT_GEMM_PACKED
    L.linear(xd, wd, bd, yd, **kw)
    torch.cuda.synchronize()
    assert L.poot_linear_device_status(0) == L.POOT_OK
    yr = oracle.linear_f16(_bits(x), _bits(w), _bits(b))
    got = _bits(yd)
    assert np.array_equal(got, yr), f"M={M} N={N} K={K} offs={(ox, ow, oy)} {kw}: {(got != yr).sum()} differ"
    # nothing written outside y
    assert torch.isnan(ybuf[:oy]).all() and torch.isnan(ybuf[oy + M * N:]).all()


STEP_CHOICES = [[], ["silu"], [("add", None)], [("mul", None)], ["silu", ("mul", None)], [("add", None), "gelu_erf"]]


@pytest.mark.parametrize("case", range(CASES // 2))
def test_random_contraction_exact(case):
    rng = np.random.default_rng(8000 + case)
    M, N, K, (ox, ow, _) = _draw(rng)
    dt = "bf16" if rng.random() < 0.5 else "f16"
    tdt = torch.bfloat16 if dt == "bf16" else torch.float16
    g = torch.Generator().manual_seed(8100 + case)
    x = torch.randint(-4, 5, (M, K), generator=g).to(tdt)
    w = torch.randint(-4, 5, (N, K), generator=g).to(tdt)
    b = torch.randint(-4, 5, (N,), generator=g).to(tdt) if rng.random() < 0.7 else None
    xd, wd = _on_device(x, ox), _on_device(w, ow)
    bd = b.to(DEV) if b is not None else None
    if rng.random() < 0.25:
        y = L.contract(xd, wd, bd, out_f32=True)
        torch.cuda.synchronize()
        _check_f32(x, w, b, y.cpu(), dt, exact_sums=True)
        return
    steps = STEP_CHOICES[int(rng.integers(0, len(STEP_CHOICES)))]
    host_steps, dev_steps = [], []
    for st in steps:
        if isinstance(st, str):
            host_steps.append(st)
            dev_steps.append(st)
        else:
            r = torch.randint(-4, 5, (M, N), generator=g).to(tdt)
            host_steps.append((st[0], r))
            dev_steps.append((st[0], r.to(DEV)))
    y = L.contract(xd, wd, bd, steps=dev_steps)
    torch.cuda.synchronize()
    assert L.poot_linear_device_status(0) == L.POOT_OK
    _check_head(x, w, b, host_steps, y.cpu(), dt, exact_sums=True)


@pytest.mark.parametrize("case", range(CASES // 2))
def test_random_linear_normal(case):
    # normal inputs: the 2-ulp rule of the contract, each output beyond it
    # inside the FP32-accumulation interval (tests.parity)
    from tests.parity import compare, intervals
    rng = np.random.default_rng(9000 + case)
    M, N, K, (ox, ow, oy) = _draw(rng)
    x, w, b = synth.make_inputs(M, N, K, "normal", 9100 + case)
    xd, wd, bd = _on_device(x, ox), _on_device(w, ow), b.to(DEV)
    ybuf = torch.full((M * N + oy + 8,), float("nan"), dtype=torch.float16, device=DEV)
    yd = ybuf[oy:oy + M * N].view(M, N)
    L.linear(xd, wd, bd, yd)
    torch.cuda.synchronize()
    assert L.poot_linear_device_status(0) == L.POOT_OK
    got = _bits(yd)
    yr, pr = oracle.linear_f16(_bits(x), _bits(w), _bits(b), want_proj=True)
    interval, wide = intervals(x.numpy(), w.numpy(), b.numpy())
    # every output beyond 2 ulps must lie inside the FP32-accumulation
    # interval; a case of a few ten thousand outputs may hold a handful
    # (the large-workload tests keep the 1e-5 fraction)
    ok, rep = compare(got, yr, pr, exact=False, interval=interval, max_outside=max(1e-5, 4.0 / got.size),
                      wide_interval=wide)
    print(rep)
    assert ok, rep
