"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Every configured workload, every kernel variant, the golden fixtures, a
sweep of ragged tiny shapes and the edge cases (K = 0, empty outputs, guard
bands around y, unaligned pointers).  Large workloads are checked on sampled
rows (every column of those rows, including all tile boundaries in N).
"""
import numpy as np
import pytest
import torch

import linear_fp16_gb300 as L
import oracle
from linear_fp16_gb300 import synth
from tests import exact
from tests.parity import compare, intervals

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
GEMM_VARIANTS = [L.VARIANT_GEMM_TMA, L.VARIANT_GEMM_CPASYNC, L.VARIANT_GEMM_REG, L.VARIANT_GEMM_PACKED]
GEMV_VARIANTS = [L.VARIANT_GEMV, L.VARIANT_GEMV_SCALAR]


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _gpu(x, w, b, variant=L.VARIANT_AUTO, wpr=0, tile_n=0, group_m=0, k_chunk=0, pair=0):
    xd, wd, bd = x.to(DEV), w.to(DEV), b.to(DEV)
    y = torch.full((x.shape[0], w.shape[0]), float("nan"), dtype=torch.float16, device=DEV)
    L.linear(xd, wd, bd, y, variant=variant, gemv_warps_per_row=wpr, gemm_tile_n=tile_n,
             gemm_group_m=group_m, gemm_k_chunk=k_chunk, gemm_cluster=pair)
    torch.cuda.synchronize()
    assert L.poot_linear_device_status(0) == L.POOT_OK
    return _bits(y)


# Outputs beyond 2 FP16 ulps of the oracle may be at most this fraction of
# those compared (each must also lie inside the interval of round-to-nearest
# FP32 accumulations in any order).
# Legal IEEE FP32 reorderings reach about 1.5e-6 on the MLP workload; the
# kernels are deterministic, so the count does not vary between runs.
MAX_BEYOND = 1e-5


def _check(x, w, b, y_bits, exact_ints=False, rows=None):
    xs = x if rows is None else x[rows]
    yr, pr = oracle.linear_f16(_bits(xs), _bits(w), _bits(b), want_proj=True)
    yg = y_bits if rows is None else y_bits[rows]
    interval = wide = None
    if not exact_ints:
        interval, wide = intervals(xs.numpy(), w.numpy(), b.numpy())
    ok, rep = compare(yg, yr, pr, exact=exact_ints, interval=interval, max_outside=MAX_BEYOND, wide_interval=wide)
    assert ok, rep
    print(rep)
    return rep


def _applicable(variant, M, K):
    if variant in GEMV_VARIANTS:
        return M <= L.GEMV_MAX_M and (variant == L.VARIANT_GEMV_SCALAR or K % 8 == 0)
    if variant == L.VARIANT_GEMM_TMA:
        return K % 8 == 0
    if variant == L.VARIANT_GEMM_CPASYNC:
        return K % 2 == 0
    return True


# ---- golden fixtures through every variant -----------------------------------
@pytest.mark.parametrize("name", ["round_before_bias.txt", "fp32_accumulation.txt",
                                  "no_product_rounding.txt", "overflow_boundary.txt",
                                  "subnormal_rounding.txt"])
@pytest.mark.parametrize("variant", GEMM_VARIANTS + GEMV_VARIANTS)
def test_golden_on_gpu(name, variant):
    x, w, b, y = exact.parse_golden(name)
    xt, wt, bt = (torch.from_numpy(a.copy()) for a in (x, w, b))
    if not _applicable(variant, xt.shape[0], xt.shape[1]):
        pytest.skip("variant not applicable to this shape")
    got = _gpu(xt, wt, bt, variant).view(np.float16).astype(np.float64)
    assert exact.same_values(got, y), (got, y)


# ---- configured workloads ----------------------------------------------------
def test_toy_full():
    x, w, b = synth.workload_inputs("toy")
    assert L.poot_linear_f16_variant(*(t.to(DEV).data_ptr() for t in (x, w, b)), 1 << 40,
                                     1024, 1024, 768) == L.VARIANT_GEMM_TMA
    _check(x, w, b, _gpu(x, w, b))


def test_ragged_exact_full_is_bit_exact():
    x, w, b = synth.workload_inputs("ragged_exact")
    _check(x, w, b, _gpu(x, w, b), exact_ints=True)


@pytest.mark.parametrize("variant", GEMM_VARIANTS)
def test_ragged_exact_every_gemm_variant_where_legal(variant):
    x, w, b = synth.workload_inputs("ragged_exact")
    if not _applicable(variant, 2047, 770):
        pytest.skip("K % 8 != 0: no TMA")
    _check(x, w, b, _gpu(x, w, b, variant), exact_ints=True)


@pytest.mark.parametrize("name", ["gemv_m1", "gemv_m8"])
def test_gemv_full(name):
    x, w, b = synth.workload_inputs(name)
    _check(x, w, b, _gpu(x, w, b))


@pytest.mark.parametrize("name", ["gemv_m1", "gemv_m8"])
@pytest.mark.parametrize("wpr", [1, 2, 4, 8])
def test_gemv_warps_per_row(name, wpr):
    x, w, b = synth.workload_inputs(name)
    _check(x, w, b, _gpu(x, w, b, L.VARIANT_GEMV, wpr))


def _sample_rows(M, n_random, seed):
    fixed = {0, 1, 127, 128, 129, 255, 256, M // 2, M - 129, M - 128, M - 2, M - 1}
    rng = np.random.default_rng(seed)
    rnd = set(int(r) for r in rng.choice(M, size=n_random, replace=False))
    return sorted(r for r in fixed | rnd if 0 <= r < M)


@pytest.mark.parametrize("name", ["prefill", "mlp_up"])
def test_large_sampled_rows(name):
    x, w, b = synth.workload_inputs(name)
    y = _gpu(x, w, b)
    rows = _sample_rows(x.shape[0], 24, 7)
    _check(x, w, b, y, rows=rows)
    # rows not sampled must still be written (y was prefilled with NaN)
    assert not np.isnan(y.view(np.float16)).any()


# ---- ragged tiny sweep ---------------------------------------------------------
SWEEP = [(M, N, K) for M in (1, 2, 7, 16, 17, 127, 129, 255) for N in (1, 8, 13, 129, 257)
         for K in (1, 7, 8, 9, 16, 63, 64, 65, 136)]


@pytest.mark.parametrize("variant", GEMM_VARIANTS + GEMV_VARIANTS)
def test_tiny_sweep_smallint_exact(variant):
    rng_seed = 100 + variant
    n = 0
    for (M, N, K) in SWEEP:
        if not _applicable(variant, M, K):
            continue
        x, w, b = synth.make_inputs(M, N, K, "smallint", rng_seed + M * 7 + N * 3 + K)
        _check(x, w, b, _gpu(x, w, b, variant), exact_ints=True)
        n += 1
    assert n > 0


@pytest.mark.parametrize("variant", [L.VARIANT_AUTO] + GEMM_VARIANTS)
def test_tiny_sweep_normal(variant):
    for (M, N, K) in SWEEP[::3]:
        if variant != L.VARIANT_AUTO and not _applicable(variant, M, K):
            continue
        x, w, b = synth.make_inputs(M, N, K, "normal", 500 + M + N + K)
        _check(x, w, b, _gpu(x, w, b, variant))


def test_many_tiles_long_k():
    # several M and N tiles, K spanning many K blocks and a tail
    x, w, b = synth.make_inputs(300, 600, 1000, "normal", 77)
    _check(x, w, b, _gpu(x, w, b, L.VARIANT_GEMM_TMA if 1000 % 8 == 0 else L.VARIANT_AUTO))
    x, w, b = synth.make_inputs(300, 600, 1002, "smallint", 78)
    for v in (L.VARIANT_GEMM_CPASYNC, L.VARIANT_GEMM_REG):
        _check(x, w, b, _gpu(x, w, b, v), exact_ints=True)


@pytest.mark.parametrize("tile_n", [64, 96, 128, 160, 192, 224, 256])
@pytest.mark.parametrize("variant", GEMM_VARIANTS)
def test_every_tile_width(tile_n, variant):
    # ragged N against each tile width; K spans several K blocks and a tail
    M, N, K = 300, 700, 200 if variant not in (L.VARIANT_GEMM_REG, L.VARIANT_GEMM_PACKED) else 203
    x, w, b = synth.make_inputs(M, N, K, "smallint", 60 + tile_n)
    if not _applicable(variant, M, K):
        pytest.skip("variant not applicable")
    _check(x, w, b, _gpu(x, w, b, variant, tile_n=tile_n), exact_ints=True)


@pytest.mark.parametrize("group_m", [1, 2, 3, 8, 64])
def test_tile_order_groups(group_m):
    x, w, b = synth.make_inputs(1100, 900, 96, "smallint", 70 + group_m)
    _check(x, w, b, _gpu(x, w, b, tile_n=128, group_m=group_m), exact_ints=True)


@pytest.mark.parametrize("k_chunk", [64, 128, 192, 256, 1024])
@pytest.mark.parametrize("variant", GEMM_VARIANTS)
def test_k_chunk_promotion(k_chunk, variant):
    # K = 1000 (1002 for odd-pitch copies): chunk boundaries inside and at
    # the end of the K range, a partial last chunk, and a single chunk
    K = 1000 if variant not in (L.VARIANT_GEMM_REG, L.VARIANT_GEMM_PACKED) else 1002
    x, w, b = synth.make_inputs(260, 300, K, "smallint", 80 + k_chunk)
    _check(x, w, b, _gpu(x, w, b, variant, k_chunk=k_chunk), exact_ints=True)
    xn, wn, bn = synth.make_inputs(260, 300, K, "normal", 81 + k_chunk)
    _check(xn, wn, bn, _gpu(xn, wn, bn, variant, k_chunk=k_chunk))


# ---- CTA pairs (2-SM MMA) ------------------------------------------------------
@pytest.mark.parametrize("M,N,K", [(256, 256, 64), (512, 512, 256), (300, 520, 136), (1000, 700, 1000),
                                   (129, 64, 64), (2047, 1000, 776)])
@pytest.mark.parametrize("pair", [1, 2])
def test_cta_pair_exact(M, N, K, pair):
    x, w, b = synth.make_inputs(M, N, K, "smallint", 40 + M % 97 + N % 13 + K)
    _check(x, w, b, _gpu(x, w, b, L.VARIANT_GEMM_TMA, pair=pair), exact_ints=True)


@pytest.mark.parametrize("tile_n", [64, 128, 192, 224, 256])
def test_cta_pair_tile_widths(tile_n):
    x, w, b = synth.make_inputs(700, 900, 200, "smallint", 50 + tile_n)
    _check(x, w, b, _gpu(x, w, b, L.VARIANT_GEMM_TMA, tile_n=tile_n, pair=2), exact_ints=True)


@pytest.mark.parametrize("k_chunk", [64, 256, 4096])
def test_cta_pair_chunks_normal(k_chunk):
    x, w, b = synth.make_inputs(600, 800, 1000, "normal", 55 + k_chunk)
    _check(x, w, b, _gpu(x, w, b, L.VARIANT_GEMM_TMA, k_chunk=k_chunk, pair=2))


def test_cta_pair_many_tiles_per_pair():
    # more tiles than pairs: the persistent loop and both chunk buffers;
    # N = 2560 / 128 = 20 tile columns, 2600 a ragged 21st
    for N in (2560, 2600):
        x, w, b = synth.make_inputs(4096, N, 128, "smallint", 57 + N)
        _check(x, w, b, _gpu(x, w, b, L.VARIANT_GEMM_TMA, tile_n=128, pair=2), exact_ints=True)


# Paired stages (two K blocks per MMA batch, released together, a chunk's
# last pair released through the chunk-complete barrier) run when every chunk
# holds an even number of at least `stages` K blocks; otherwise one stage at a
# time.  Each case below runs more tiles than CTAs (or pairs), so chunk
# counting continues across tiles.  K blocks of 64: 832 -> 13 (odd: one stage
# at a time); 1152 -> 18 = 16 + a 2-block tail (too short: one at a time);
# 1536 -> 24 = 16 + 8 (paired, with a tail chunk); 1536 with 384-element
# chunks -> 4 chunks of 6 (paired at 6 stages, one at a time at 8); 1536 with
# 192-element chunks -> chunks of 3 (odd: one at a time); 768 -> one chunk.
@pytest.mark.parametrize("K,k_chunk", [(832, 0), (1152, 0), (1536, 0), (1536, 384), (1536, 192), (768, 0)])
@pytest.mark.parametrize("pair", [1, 2])
def test_stage_pairing_boundaries(K, k_chunk, pair):
    x, w, b = synth.make_inputs(520, 2048, K, "smallint", 90 + K + k_chunk)
    _check(x, w, b, _gpu(x, w, b, L.VARIANT_GEMM_TMA, tile_n=64, k_chunk=k_chunk, pair=pair), exact_ints=True)
    xn, wn, bn = synth.make_inputs(520, 2048, K, "normal", 91 + K + k_chunk)
    _check(xn, wn, bn, _gpu(xn, wn, bn, L.VARIANT_GEMM_TMA, tile_n=256, k_chunk=k_chunk, pair=pair))


def test_more_tiles_than_sms():
    # forces the persistent loop to take several tiles per CTA and both
    # TMEM accumulators
    x, w, b = synth.make_inputs(2048, 5120, 128, "smallint", 79)
    _check(x, w, b, _gpu(x, w, b), exact_ints=True)


# ---- edge cases ------------------------------------------------------------------
def test_k_zero_is_bias():
    b = torch.tensor([1.5, -2.0, -0.0, 65504.0], dtype=torch.float16)
    x = torch.zeros((3, 0), dtype=torch.float16)
    w = torch.zeros((4, 0), dtype=torch.float16)
    y = _gpu(x, w, b)
    want = np.broadcast_to(_bits(b), (3, 4)).copy()
    want[:, 2] = 0  # +0 + -0 = +0
    assert np.array_equal(y, want)


def test_empty_outputs_launch_nothing():
    x = torch.zeros((0, 5), dtype=torch.float16, device=DEV)
    w = torch.zeros((4, 5), dtype=torch.float16, device=DEV)
    b = torch.zeros((4,), dtype=torch.float16, device=DEV)
    y = L.linear(x, w, b)
    assert y.shape == (0, 4)


@pytest.mark.parametrize("M,N,K", [(1, 64, 64), (200, 136, 72), (33, 1001, 40)])
def test_guard_bands_untouched(M, N, K):
    # y lives inside a larger buffer whose margins hold a sentinel
    x, w, b = synth.make_inputs(M, N, K, "smallint", 90 + M)
    pad = 4096
    buf = torch.full((pad + M * N + pad,), 12345.0, dtype=torch.float16, device=DEV)
    y = buf[pad:pad + M * N].view(M, N)
    L.linear(x.to(DEV), w.to(DEV), b.to(DEV), y)
    torch.cuda.synchronize()
    assert torch.all(buf[:pad] == 12345.0) and torch.all(buf[pad + M * N:] == 12345.0)
    _check(x, w, b, _bits(y), exact_ints=True)


@pytest.mark.parametrize("M", [5, 300])
def test_unaligned_pointers_take_the_ragged_paths(M):
    N, K = 72, 64
    x, w, b = synth.make_inputs(M, N, K, "smallint", 91 + M)
    xs = torch.zeros(M * K + 1, dtype=torch.float16, device=DEV)
    ws = torch.zeros(N * K + 3, dtype=torch.float16, device=DEV)
    xd = xs[1:].view(M, K)
    wd = ws[3:].view(N, K)
    xd.copy_(x)
    wd.copy_(w)
    y = torch.empty((M, N), dtype=torch.float16, device=DEV)
    v = L.variant_for(xd, wd, b, y)
    assert v in (L.VARIANT_GEMV_SCALAR, L.VARIANT_GEMM_PACKED)
    L.linear(xd, wd, b.to(DEV), y)
    torch.cuda.synchronize()
    _check(x, w, b, _bits(y), exact_ints=True)


def test_odd_n_uses_plain_stores():
    x, w, b = synth.make_inputs(257, 1003, 128, "normal", 92)
    _check(x, w, b, _gpu(x, w, b))


def test_nonfinite_inputs_propagate():
    x, w, b = synth.make_inputs(130, 16, 16, "smallint", 93)
    x[3, 5] = float("inf")
    x[7, 2] = float("nan")
    y = _gpu(x, w, b).view(np.float16)
    assert np.isnan(y[7]).all()
    row3 = y[3]
    wcol = w[:, 5].float().numpy()
    for n in range(16):
        if wcol[n] > 0:
            assert np.isposinf(row3[n])
        elif wcol[n] < 0:
            assert np.isneginf(row3[n])
        else:
            assert np.isnan(row3[n])  # inf * 0


def test_repeated_calls_are_deterministic():
    x, w, b = synth.make_inputs(512, 512, 512, "normal", 94)
    y1 = _gpu(x, w, b)
    y2 = _gpu(x, w, b)
    assert np.array_equal(y1, y2)


def test_runs_on_a_side_stream():
    x, w, b = synth.make_inputs(256, 256, 256, "smallint", 95)
    s = torch.cuda.Stream()
    xd, wd, bd = x.to(DEV), w.to(DEV), b.to(DEV)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        y = L.linear(xd, wd, bd)
    s.synchronize()
    _check(x, w, b, _bits(y), exact_ints=True)
