"""Split-K (the K range cut into S ranges, FP32 partial sums added in range
order by a second kernel that applies the epilogue), on a GPU.

Any FP32 summation order is legal for the sum of products, so the rules are
those of the unsplit path: bit-exact on small-integer inputs, the 2-ulp rule
(with the FP32-interval fallback) otherwise; the widened forms use the same
checks as their unsplit tests.  Covers forced split factors (including one K
block per range and a ragged last block), the automatic split on shapes with
few output tiles, CTA pairs, every GEMM variant, the widened epilogues, the
workspace's growth and sharing per stream, and stream capture.
"""
import numpy as np
import pytest
import torch

import linear_fp16_gb300 as L
from linear_fp16_gb300 import synth
from tests.test_gpu_contract import _check_f32, _check_head, _inputs, _operand
from tests.test_gpu_parity import _bits, _check

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)
GEMM_VARIANTS = [L.VARIANT_GEMM_TMA, L.VARIANT_GEMM_CPASYNC, L.VARIANT_GEMM_REG]


def _lin(x, w, b, **kw):
    xd, wd, bd = x.to(DEV), w.to(DEV), b.to(DEV)
    y = torch.full((x.shape[0], w.shape[0]), float("nan"), dtype=torch.float16, device=DEV)
    L.linear(xd, wd, bd, y, **kw)
    torch.cuda.synchronize()
    assert L.poot_linear_device_status(0) == L.POOT_OK
    return _bits(y)


def _con(x, w, b, steps=(), out_f32=False, **kw):
    bd = b.to(DEV) if b is not None else None
    dsteps = [s if isinstance(s, str) else (s[0], s[1].to(DEV)) for s in steps]
    y = L.contract(x.to(DEV), w.to(DEV), bd, out_f32=out_f32, steps=dsteps, **kw)
    torch.cuda.synchronize()
    assert L.poot_linear_device_status(0) == L.POOT_OK
    return y.cpu()


# ---- the plain path -----------------------------------------------------------
@pytest.mark.parametrize("S", [2, 4, 8, 16])
@pytest.mark.parametrize("variant", GEMM_VARIANTS)
def test_forced_split_exact(S, variant):
    # K = 1000 / 1002: 16 K blocks, the last one ragged; S = 16 leaves one
    # block per range
    K = 1000 if variant != L.VARIANT_GEMM_REG else 1002
    x, w, b = synth.make_inputs(200, 300, K, "smallint", 900 + S + variant)
    _check(x, w, b, _lin(x, w, b, variant=variant, gemm_split_k=S), exact_ints=True)


@pytest.mark.parametrize("S", [2, 8])
def test_forced_split_normal(S):
    x, w, b = synth.make_inputs(260, 520, 2048, "normal", 910 + S)
    _check(x, w, b, _lin(x, w, b, gemm_split_k=S))


@pytest.mark.parametrize("S", [2, 4])
def test_forced_split_with_cta_pairs(S):
    x, w, b = synth.make_inputs(512, 512, 1024, "smallint", 920 + S)
    _check(x, w, b, _lin(x, w, b, gemm_cluster=2, gemm_split_k=S), exact_ints=True)
    xn, wn, bn = synth.make_inputs(600, 520, 1024, "normal", 921 + S)
    _check(xn, wn, bn, _lin(xn, wn, bn, gemm_cluster=2, gemm_split_k=S))


@pytest.mark.parametrize("k_chunk", [64, 256])
def test_split_with_chunked_promotion(k_chunk):
    x, w, b = synth.make_inputs(130, 200, 2048, "smallint", 930 + k_chunk)
    _check(x, w, b, _lin(x, w, b, gemm_split_k=4, gemm_k_chunk=k_chunk), exact_ints=True)


@pytest.mark.parametrize("M,N,K", [(128, 1024, 8192), (256, 2048, 4096), (64, 512, 16384), (100, 700, 3000)])
def test_automatic_split_shapes(M, N, K):
    # few output tiles and a long K: the automatic plan splits these
    x, w, b = synth.make_inputs(M, N, K, "smallint", 940 + M)
    _check(x, w, b, _lin(x, w, b), exact_ints=True)
    xn, wn, bn = synth.make_inputs(M, N, K, "normal", 941 + M)
    _check(xn, wn, bn, _lin(xn, wn, bn))


def test_no_split_and_split_agree_on_exact_sums():
    x, w, b = synth.make_inputs(128, 1024, 8192, "smallint", 950)
    y1 = _lin(x, w, b, gemm_split_k=1)
    for S in (2, 4, 8, 16):
        assert np.array_equal(y1, _lin(x, w, b, gemm_split_k=S))


def test_split_is_deterministic():
    x, w, b = synth.make_inputs(128, 1024, 8192, "normal", 951)
    y = _lin(x, w, b, gemm_split_k=8)
    for _ in range(3):
        assert np.array_equal(y, _lin(x, w, b, gemm_split_k=8))


def test_split_that_does_not_divide_the_k_blocks_is_refused():
    xd = torch.zeros(64, 1000, dtype=torch.float16, device=DEV)   # 16 K blocks
    wd = torch.zeros(128, 1000, dtype=torch.float16, device=DEV)
    bd = torch.zeros(128, dtype=torch.float16, device=DEV)
    yd = torch.zeros(64, 128, dtype=torch.float16, device=DEV)
    for S in (3, 5, 6):
        rc = L.poot_linear_f16_ex(xd.data_ptr(), wd.data_ptr(), bd.data_ptr(), yd.data_ptr(), 64, 128, 1000,
                                  L.options(L.VARIANT_GEMM_TMA, gemm_split_k=S), 0)
        assert rc == L.POOT_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert torch.count_nonzero(yd) == 0


# ---- the widened contraction ----------------------------------------------------
@pytest.mark.parametrize("dt", ["f16", "bf16"])
@pytest.mark.parametrize("S", [2, 8])
def test_widened_head_bias_and_steps(dt, S):
    M, N, K = 150, 260, 2048
    x, w, b = _inputs(M, N, K, "smallint", 960 + S, dt)
    _check_head(x, w, b, [], _con(x, w, b, gemm_split_k=S), dt, exact_sums=True)
    _check_head(x, w, None, [], _con(x, w, None, gemm_split_k=S), dt, exact_sums=True)
    r = _operand(M, N, "smallint", 961 + S, dt)
    steps = ["silu", ("mul", r)]
    _check_head(x, w, b, steps, _con(x, w, b, steps, gemm_split_k=S), dt, exact_sums=True)
    xn, wn, bn = _inputs(M, N, K, "normal", 962 + S, dt)
    rn = _operand(M, N, "normal", 963 + S, dt)
    steps = [("add", rn), "gelu_tanh"]
    _check_head(xn, wn, bn, steps, _con(xn, wn, bn, steps, gemm_split_k=S), dt, exact_sums=False)


@pytest.mark.parametrize("dt", ["f16", "bf16"])
@pytest.mark.parametrize("with_bias", [True, False])
def test_widened_f32_output(dt, with_bias):
    M, N, K = 130, 258, 1024
    x, w, b = _inputs(M, N, K, "smallint", 970, dt)
    b = b if with_bias else None
    _check_f32(x, w, b, _con(x, w, b, out_f32=True, gemm_split_k=4), dt, exact_sums=True)
    xn, wn, bn = _inputs(M, N, K, "normal", 971, dt)
    bn = bn if with_bias else None
    _check_f32(xn, wn, bn, _con(xn, wn, bn, out_f32=True, gemm_split_k=4), dt, exact_sums=False)


def test_widened_automatic_split():
    M, N, K = 128, 1024, 8192
    x, w, b = _inputs(M, N, K, "smallint", 975, "bf16")
    r = _operand(M, N, "smallint", 976, "bf16")
    steps = ["silu", ("mul", r)]
    _check_head(x, w, b, steps, _con(x, w, b, steps), "bf16", exact_sums=True)


def test_grouped_contraction_refuses_a_split():
    x = torch.zeros(2, 64, 1024, dtype=torch.float16, device=DEV)
    w = torch.zeros(256, 1024, dtype=torch.float16, device=DEV)
    with pytest.raises(L.PootLinearError):
        L.contract(x, w, gemm_split_k=2)


# ---- workspace ------------------------------------------------------------------
def test_workspace_grows_and_stays_correct():
    # a small split, a larger one (the workspace grows), the small one again
    shapes = [(64, 256, 2048), (256, 2048, 4096), (64, 256, 2048)]
    for i, (M, N, K) in enumerate(shapes):
        x, w, b = synth.make_inputs(M, N, K, "smallint", 980 + i)
        _check(x, w, b, _lin(x, w, b, gemm_split_k=8), exact_ints=True)


def test_two_streams_in_flight():
    # each stream has its own workspace: calls queued on both at once
    ins = [synth.make_inputs(128, 1024, 4096, "smallint", 985 + i) for i in range(2)]
    dev = [tuple(t.to(DEV) for t in xwb) for xwb in ins]
    ys = [torch.empty(128, 1024, dtype=torch.float16, device=DEV) for _ in range(2)]
    streams = [torch.cuda.Stream(DEV) for _ in range(2)]
    torch.cuda.synchronize()
    for rep in range(4):
        for i in range(2):
            with torch.cuda.stream(streams[i]):
                L.linear(*dev[i], ys[i], gemm_split_k=8)
    torch.cuda.synchronize()
    assert L.poot_linear_device_status(0) == L.POOT_OK
    for i in range(2):
        _check(*ins[i], _bits(ys[i]), exact_ints=True)


def test_stream_capture_uses_a_graph_owned_workspace():
    x, w, b = synth.make_inputs(128, 1024, 8192, "smallint", 990)
    xd, wd, bd = x.to(DEV), w.to(DEV), b.to(DEV)
    y = torch.full((128, 1024), float("nan"), dtype=torch.float16, device=DEV)
    L.linear(xd, wd, bd, y, gemm_split_k=8)   # an eager call first (its own workspace)
    torch.cuda.synchronize()
    eager = _bits(y)
    y.fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        L.linear(xd, wd, bd, y, gemm_split_k=8)
    for _ in range(2):
        y.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(_bits(y), eager)
    assert L.poot_linear_device_status(0) == L.POOT_OK
    _check(x, w, b, eager, exact_ints=True)


# ---- long K and concurrent host threads -----------------------------------------
@pytest.mark.parametrize("M,N", [(200, 300), (1, 520), (8, 264)])
def test_k_65536_exact(M, N):
    # |S| <= 65536 * 16 < 2^24: every FP32 partial sum is exact, so the result
    # is bit-exact whatever the split and chunking (GEMM with automatic
    # split for M = 200; the GEMVs for M = 1 and 8)
    x, w, b = synth.make_inputs(M, N, 65536, "smallint", 996 + M)
    _check(x, w, b, _lin(x, w, b), exact_ints=True)


def test_two_host_threads_on_their_own_streams():
    import threading
    ins = [synth.make_inputs(128, 1024, 8192, "smallint", 997 + i) for i in range(2)]
    dev = [tuple(t.to(DEV) for t in xwb) for xwb in ins]
    ys = [torch.empty(128, 1024, dtype=torch.float16, device=DEV) for _ in range(2)]
    torch.cuda.synchronize()
    errors = []

    def work(i):
        try:
            s = torch.cuda.Stream(DEV)
            with torch.cuda.stream(s):
                for _ in range(5):
                    L.linear(*dev[i], ys[i])   # automatic split-K: the stream's own workspace
            s.synchronize()
        except Exception as e:  # pragma: no cover - reported below
            errors.append(e)

    th = [threading.Thread(target=work, args=(i,)) for i in range(2)]
    for t in th:
        t.start()
    for t in th:
        t.join()
    assert not errors, errors
    assert L.poot_linear_device_status(0) == L.POOT_OK
    for i in range(2):
        _check(*ins[i], _bits(ys[i]), exact_ints=True)


def test_per_thread_default_stream_handle_from_two_threads():
    # cudaStreamPerThread (handle 2) names a different stream in each thread:
    # each thread gets its own workspace
    import threading
    PER_THREAD = 2
    ins = [synth.make_inputs(128, 1024, 8192, "smallint", 1990 + i) for i in range(2)]
    dev = [tuple(t.to(DEV) for t in xwb) for xwb in ins]
    ys = [torch.empty(128, 1024, dtype=torch.float16, device=DEV) for _ in range(2)]
    torch.cuda.synchronize()
    rcs = [None, None]

    def work(i):
        x, w, b = dev[i]
        for _ in range(5):
            rc = L.poot_linear_f16(x.data_ptr(), w.data_ptr(), b.data_ptr(), ys[i].data_ptr(), 128, 1024, 8192,
                                   PER_THREAD)
            if rc != L.POOT_OK:
                break
        rcs[i] = rc

    th = [threading.Thread(target=work, args=(i,)) for i in range(2)]
    for t in th:
        t.start()
    for t in th:
        t.join()
    torch.cuda.synchronize()
    assert rcs == [L.POOT_OK, L.POOT_OK]
    assert L.poot_linear_device_status(0) == L.POOT_OK
    for i in range(2):
        _check(*ins[i], _bits(ys[i]), exact_ints=True)
