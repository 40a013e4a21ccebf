"""Parity of the widened contraction (poot_contract) with the oracle, on a GPU.

Rules (the readings of the source pages on the widened contraction):
* small-integer inputs make every sum exact, so the head value is the
  oracle's; bias, ADD and MUL steps are then bit-exact, and activation steps
  may differ only where FP32 expf / erff and the oracle's binary64 exp / erf
  round to different head values (rare, a few ulps);
* otherwise the head value is within the base contract's 2-ulp rule, and y
  must lie within the oracle's epilogue applied to its head value +-2 ulps
  (the hull), widened by 2 ulps for those exp / erf roundings;
* FP32 output: the sum error bound gamma_K sum|x w| with u = 2^-24 (any
  round-to-nearest FP32 order), plus one FP32 rounding of the bias add.
"""
import numpy as np
import pytest
import torch

import linear_fp16_gb300 as L
import oracle
from linear_fp16_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)
TDT = {"f16": torch.float16, "bf16": torch.bfloat16}
MAX_OUTSIDE_HULL = 1e-4    # outputs allowed outside the hull (each inside the interval image)
MAX_ACT_INEXACT = 2e-3     # activation outputs allowed to differ at all (exact-sum inputs)


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _val(bits, dt) -> np.ndarray:
    bits = np.asarray(bits, dtype=np.uint16)
    if dt == "f16":
        return bits.view(np.float16).astype(np.float64)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _ulp(v, dt) -> np.ndarray:
    """Spacing of the head format at |v| (its minimum below the normal range)."""
    p, emin = (11, -14) if dt == "f16" else (8, -126)
    a = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, emin)
    return np.where(np.isfinite(a), np.exp2(e - (p - 1)), np.inf)


def _neighbour(bits, j):
    """Head-format value j steps away (monotone integer key of the bits)."""
    b = np.asarray(bits, dtype=np.int64)
    key = np.where(b & 0x8000, -(b & 0x7FFF), b) + j
    return np.where(key < 0, (-key) | 0x8000, key).astype(np.uint16)


def _inputs(M, N, K, dist, seed, dt):
    x, w, b = synth.make_inputs(M, N, K, dist, seed)   # float16 draws
    if dt == "bf16":
        x, w, b = (t.float().to(torch.bfloat16) for t in (x, w, b))
    return x, w, b


def _operand(M, N, dist, seed, dt, lo=-4, hi=5):
    g = torch.Generator().manual_seed(seed)
    if dist == "smallint":
        r = torch.randint(lo, hi, (M, N), generator=g).float()
    else:
        r = torch.randn((M, N), generator=g)
    return r.to(TDT[dt])


def _gpu(x, w, b, steps=(), out_f32=False, **kw):
    xd, wd = x.to(DEV), w.to(DEV)
    bd = b.to(DEV) if b is not None else None
    dsteps = [s if isinstance(s, str) else (s[0], s[1].to(DEV)) for s in steps]
    y = L.contract(xd, wd, bd, out_f32=out_f32, steps=dsteps, **kw)
    torch.cuda.synchronize()
    assert L.poot_linear_device_status(0) == L.POOT_OK
    return y.cpu()


def _ref_steps(steps, rows=None):
    out = []
    for s in steps:
        if isinstance(s, str):
            out.append(s)
        else:
            r = s[1] if rows is None else s[1][rows]
            out.append((s[0], _bits(r)))
    return out


def _check_head(x, w, b, steps, y, dt, exact_sums, rows=None):
    xs = x if rows is None else x[rows]
    st = _ref_steps(steps, rows)
    bb = _bits(b) if b is not None else None
    yr, pr = oracle.contraction(_bits(xs), _bits(w), bb, dtype=dt, steps=st, want_proj=True)
    yg = _bits(y if rows is None else y[rows])
    has_act = any(isinstance(s, str) for s in steps)
    gv, rv = _val(yg, dt), _val(yr, dt)
    same = (yg == yr) | (np.isnan(gv) & np.isnan(rv)) | ((gv == 0) & (rv == 0))
    if exact_sums and not has_act:
        assert same.all(), f"{(~same).sum()} of {same.size} differ"
        return
    if exact_sums:
        close = same | (np.abs(gv - rv) <= 4 * _ulp(rv, dt))
        assert close.all(), f"{(~close).sum()} beyond 4 ulps"
        assert (~same).mean() <= MAX_ACT_INEXACT, f"{(~same).sum()} of {same.size} inexact"
        return
    # the hull of the oracle's epilogue over head values within 2 ulps of its own
    hull = [oracle.epilogue(_neighbour(pr, j), bb, dtype=dt, steps=st) for j in range(-2, 3)]
    hv = np.stack([_val(h, dt) for h in hull])
    lo, hi = np.nanmin(hv, axis=0), np.nanmax(hv, axis=0)
    inside = same | ((gv >= lo - 2 * _ulp(lo, dt)) & (gv <= hi + 2 * _ulp(hi, dt)))
    # outside the hull: a cancelling sum whose head value moved more than 2
    # ulps; legal if y is the epilogue of some head value that an FP32 sum of
    # the same products can round to (Higham's bound, u = 2^-24)
    outl = np.argwhere(~inside)
    for m, n in outl:
        assert _in_interval_image(xs, w, b, st, m, n, gv[m, n], dt), \
            f"y[{m},{n}] = {gv[m, n]} is no epilogue of a legal FP32 sum"
    assert len(outl) <= max(1, int(MAX_OUTSIDE_HULL * inside.size)), f"{len(outl)} of {inside.size} outside the hull"
    print(f"bit-identical {same.mean():.5f}, outside hull (inside the interval image) {len(outl)}")


def _in_interval_image(xs, w, b, st, m, n, yv, dt):
    xv = xs[m].double() if dt == "f16" else xs[m].float().double()
    wv = w[n].double() if dt == "f16" else w[n].float().double()
    S = float((xv * wv).sum())
    A = float((xv * wv).abs().sum())
    K = xv.numel()
    u = 2.0 ** -24
    E = K * u / (1 - K * u) * A
    conv = oracle.f64_to_f16_rn if dt == "f16" else oracle.f64_to_bf16_rn
    k_lo, k_hi = (_key(conv([S - E])[0]), _key(conv([S + E])[0]))
    keys = np.arange(k_lo, k_hi + 1)[:1 << 16]
    t = np.where(keys < 0, (-keys) | 0x8000, keys).astype(np.uint16).reshape(1, -1)
    bb = None if b is None else np.full(t.shape[1], _bits(b)[n], dtype=np.uint16)
    st1 = [s if isinstance(s, str) else (s[0], np.full(t.shape, s[1][m, n], dtype=np.uint16)) for s in st]
    img = _val(oracle.epilogue(t, bb, dtype=dt, steps=st1), dt)
    lo, hi = np.nanmin(img), np.nanmax(img)
    return lo - 2 * _ulp(lo, dt) <= yv <= hi + 2 * _ulp(hi, dt)


def _key(bits):
    b = int(bits)
    return -(b & 0x7FFF) if b & 0x8000 else b


def _check_f32(x, w, b, y, dt, exact_sums):
    xs = x.double() if dt == "f16" else x.float().double()
    ws = w.double() if dt == "f16" else w.float().double()
    yg = y.double().numpy()
    if exact_sums:
        yr = oracle.contraction(_bits(x), _bits(w), _bits(b) if b is not None else None, dtype=dt, out_f32=True)
        assert np.array_equal(yg, yr.astype(np.float64))
        return
    S = (xs @ ws.T).numpy()
    A = (xs.abs() @ ws.abs().T).numpy()
    K = x.shape[1]
    u = 2.0 ** -24
    bound = K * u / (1 - K * u) * A
    if b is not None:
        S = S + b.double().numpy() if dt == "f16" else S + b.float().double().numpy()
        bound = bound + np.abs(S) * 2.0 ** -24
    err = np.abs(yg - S)
    print(f"FP32 output: largest error / bound {float((err / (bound + 1e-30)).max()):.4f}")
    assert np.all(err <= bound + 1e-30)


# ---- head dtype, bias, no steps ---------------------------------------------------
@pytest.mark.parametrize("dt", ["f16", "bf16"])
@pytest.mark.parametrize("M,N,K", [(300, 520, 256), (2047, 1000, 770), (5, 264, 200), (129, 72, 75)])
def test_head_and_bias_exact(dt, M, N, K):
    x, w, b = _inputs(M, N, K, "smallint", 300 + M + K, dt)
    _check_head(x, w, b, [], _gpu(x, w, b), dt, exact_sums=True)


@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_no_bias(dt):
    x, w, _ = _inputs(600, 520, 512, "smallint", 310, dt)
    _check_head(x, w, None, [], _gpu(x, w, None), dt, exact_sums=True)
    xn, wn, _ = _inputs(600, 520, 512, "normal", 311, dt)
    _check_head(xn, wn, None, [], _gpu(xn, wn, None), dt, exact_sums=False)


def test_f16_head_equals_the_plain_path_on_exact_sums():
    x, w, b = _inputs(700, 900, 320, "smallint", 312, "f16")
    yp = L.linear(x.to(DEV), w.to(DEV), b.to(DEV)).cpu()
    assert torch.equal(_gpu(x, w, b).view(torch.int16), yp.view(torch.int16))


@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_normal_inputs_with_bias(dt):
    x, w, b = _inputs(520, 700, 1024, "normal", 313, dt)
    _check_head(x, w, b, [], _gpu(x, w, b), dt, exact_sums=False)


# ---- FP32 output ------------------------------------------------------------------
@pytest.mark.parametrize("dt", ["f16", "bf16"])
@pytest.mark.parametrize("with_bias", [True, False])
@pytest.mark.parametrize("M,N,K", [(600, 520, 512), (130, 70, 74), (7, 66, 96)])
def test_f32_output(dt, with_bias, M, N, K):
    x, w, b = _inputs(M, N, K, "smallint", 320 + N, dt)
    b = b if with_bias else None
    y = _gpu(x, w, b, out_f32=True)
    assert y.dtype == torch.float32
    _check_f32(x, w, b, y, dt, exact_sums=True)
    xn, wn, bn = _inputs(M, N, K, "normal", 321 + N, dt)
    bn = bn if with_bias else None
    _check_f32(xn, wn, bn, _gpu(xn, wn, bn, out_f32=True), dt, exact_sums=False)


# ---- epilogue steps ---------------------------------------------------------------
STEP_SETS = {
    "add": lambda r: [("add", r)],
    "mul": lambda r: [("mul", r)],
    "silu": lambda r: ["silu"],
    "gelu_tanh": lambda r: ["gelu_tanh"],
    "gelu_erf": lambda r: ["gelu_erf"],
    "swiglu": lambda r: ["silu", ("mul", r)],
    "residual_gelu": lambda r: ["gelu_erf", ("add", r)],
    "four": lambda r: [("mul", r), "gelu_tanh", ("add", r), "silu"],
}


@pytest.mark.parametrize("dt", ["f16", "bf16"])
@pytest.mark.parametrize("name", sorted(STEP_SETS))
def test_steps_on_exact_sums(dt, name):
    M, N, K = 520, 700, 256
    x, w, b = _inputs(M, N, K, "smallint", 330, dt)
    # small sums keep the activations in their interesting range
    x, w = x / 4, w / 4
    r = _operand(M, N, "smallint", 331, dt)
    steps = STEP_SETS[name](r)
    _check_head(x, w, b, steps, _gpu(x, w, b, steps=steps), dt, exact_sums=True)


@pytest.mark.parametrize("dt", ["f16", "bf16"])
@pytest.mark.parametrize("name", ["swiglu", "residual_gelu", "gelu_tanh", "four"])
def test_steps_on_normal_inputs(dt, name):
    M, N, K = 600, 520, 1024
    x, w, b = _inputs(M, N, K, "normal", 340, dt)
    r = _operand(M, N, "normal", 341, dt)
    steps = STEP_SETS[name](r)
    _check_head(x, w, b, steps, _gpu(x, w, b, steps=steps), dt, exact_sums=False)


@pytest.mark.parametrize("pair", [1, 2])
@pytest.mark.parametrize("tile_n", [64, 128, 256])
def test_steps_across_tiles_and_pairs(pair, tile_n):
    M, N, K = 1000, 900, 512
    x, w, b = _inputs(M, N, K, "smallint", 350 + tile_n, "f16")
    x, w = x / 4, w / 4
    r = _operand(M, N, "smallint", 351, "f16")
    steps = ["silu", ("mul", r), ("add", r)]
    y = _gpu(x, w, b, steps=steps, gemm_cluster=pair, gemm_tile_n=tile_n)
    _check_head(x, w, b, steps, y, "f16", exact_sums=True)


def test_strided_and_unaligned_operands():
    # an operand that is a column slice of a wider tensor (ld > N, so no
    # 16-byte vector loads), and one that starts 2 bytes off 16-byte alignment
    M, N, K = 300, 264, 128
    x, w, b = _inputs(M, N, K, "smallint", 360, "f16")
    wide = _operand(M, N + 24, "smallint", 361, "f16")
    r1 = wide[:, 8:8 + N]
    flat = _operand(1, M * N + 1, "smallint", 362, "f16")
    r2 = flat[0, 1:].view(M, N)
    steps = [("add", r1), ("mul", r2)]
    xd, wd, bd = x.to(DEV), w.to(DEV), b.to(DEV)
    wide_d, flat_d = wide.to(DEV), flat.to(DEV)
    y = L.contract(xd, wd, bd, steps=[("add", wide_d[:, 8:8 + N]), ("mul", flat_d[0, 1:].view(M, N))]).cpu()
    torch.cuda.synchronize()
    _check_head(x, w, b, [("add", r1.contiguous()), ("mul", r2.contiguous())], y, "f16", exact_sums=True)


@pytest.mark.parametrize("pair,tile_n", [(1, 64), (1, 128), (2, 224), (2, 256)])
@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_staged_operand_boxes(pair, tile_n, dt):
    # The first ADD / MUL step's operand, 16-byte aligned with ld % 8 == 0, is
    # staged through shared memory box by box (cp.async); here ld = N + 4 with
    # N % 8 == 4, so the last 16-byte chunk of each row is half inside the
    # operand (a partial copy, zero-filled), M leaves a ragged last tile, and
    # the tile widths give one to four boxes per epilogue warp.  A second
    # operand step reads its operand directly.
    M, N, K = 333, 1004, 256
    x, w, b = _inputs(M, N, K, "smallint", 400 + tile_n, dt)
    x, w = x / 4, w / 4
    wide = _operand(M, N + 4, "smallint", 401, dt)
    r1 = wide[:, :N]
    r2 = _operand(M, N, "smallint", 402, dt)
    xd, wd, bd = x.to(DEV), w.to(DEV), b.to(DEV)
    wide_d, r2_d = wide.to(DEV), r2.to(DEV)
    assert wide_d[:, :N].stride(0) % 8 == 0 and wide_d.data_ptr() % 16 == 0
    for steps_d, steps_h in (
            ([("add", wide_d[:, :N]), "silu", ("mul", r2_d)], [("add", r1.contiguous()), "silu", ("mul", r2)]),
            (["gelu_tanh", ("mul", wide_d[:, :N])], ["gelu_tanh", ("mul", r1.contiguous())])):
        y = L.contract(xd, wd, bd, steps=steps_d, gemm_cluster=pair, gemm_tile_n=tile_n).cpu()
        torch.cuda.synchronize()
        assert L.poot_linear_device_status(0) == L.POOT_OK
        _check_head(x, w, b, steps_h, y, dt, exact_sums=True)


@pytest.mark.parametrize("M,N,K", [(1, 4096, 512), (8, 1000, 770), (16, 72, 33)])
def test_small_m_on_the_gemv_and_the_gemm(M, N, K):
    # K % 8 == 0: the GEMV with the per-element epilogue; else (and when the
    # GEMM is forced) the tcgen05 GEMM with M rows of its 128-row tile
    x, w, b = _inputs(M, N, K, "smallint", 370 + K, "f16")
    r = _operand(M, N, "smallint", 371, "f16")
    steps = [("mul", r), "silu"]
    _check_head(x, w, b, steps, _gpu(x, w, b, steps=steps), "f16", exact_sums=True)
    _check_head(x, w, b, steps, _gpu(x, w, b, steps=steps, variant=L.VARIANT_GEMM_PACKED), "f16",
                exact_sums=True)


def test_large_swiglu_sampled_rows():
    # MLP up-projection shape with the SwiGLU gate epilogue: every column of
    # 96 sampled rows (tile boundaries included) against the oracle
    M, N, K = 8192, 14336, 4096
    x, w, b = _inputs(M, N, K, "normal", 1005, "f16")
    up = _operand(M, N, "normal", 380, "f16")
    steps = ["silu", ("mul", up)]
    y = _gpu(x, w, b, steps=steps)
    g = np.random.default_rng(381)
    rows = np.unique(np.concatenate([[0, 127, 128, 255, 256, M - 1], g.integers(0, M, 90)]))
    _check_head(x, w, b, steps, y, "f16", exact_sums=False, rows=torch.from_numpy(rows))


def test_contract_is_deterministic():
    x, w, b = _inputs(700, 600, 512, "normal", 390, "bf16")
    r = _operand(700, 600, "normal", 391, "bf16")
    a = _gpu(x, w, b, steps=["gelu_erf", ("mul", r)])
    c = _gpu(x, w, b, steps=["gelu_erf", ("mul", r)])
    assert torch.equal(a.view(torch.int16), c.view(torch.int16))


# ---- grouped contraction ----------------------------------------------------------
def _grouped_inputs(G, M, N, K, dist, seed, dt):
    x, w, b = _inputs(G * M, G * N, K, dist, seed, dt)
    return x.reshape(G, M, K), w, b


@pytest.mark.parametrize("dt", ["f16", "bf16"])
@pytest.mark.parametrize("G,M,N,K,pair", [
    (4, 300, 264, 256, 0),      # M not a multiple of 128 or 256: tiles overhang their group
    (3, 129, 72, 200, 1),       # single CTAs, ragged N
    (8, 64, 520, 512, 0),       # many small groups
    (2, 1000, 900, 770, 0),     # K % 8 != 0: the copy producers
    (5, 256, 256, 128, 2),      # CTA pairs, groups of exactly one pair tile
])
def test_grouped_exact(dt, G, M, N, K, pair):
    x, w, b = _grouped_inputs(G, M, N, K, "smallint", 400 + G + M, dt)
    x = x / 4
    r = _operand(G * M, N, "smallint", 401, dt).reshape(G, M, N)
    steps = [("mul", r), ("add", r)]
    y = _gpu(x, w, b, steps=steps, gemm_cluster=pair)
    assert tuple(y.shape) == (G, M, N)
    want = oracle.contraction_grouped(_bits(x.reshape(G, M, K)), _bits(w), _bits(b), dtype=dt,
                                      steps=[(s[0], _bits(s[1])) for s in steps])
    assert np.array_equal(_bits(y), want)


@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_grouped_activation_and_f32(dt):
    G, M, N, K = 3, 200, 300, 512
    x, w, b = _grouped_inputs(G, M, N, K, "normal", 410, dt)
    steps = ["gelu_erf"]
    y = _gpu(x, w, b, steps=steps)
    for g in range(G):
        _check_head(x[g], w[g * N:(g + 1) * N], b[g * N:(g + 1) * N], steps, y[g], dt, exact_sums=False)
    yf = _gpu(x, w, None, out_f32=True)
    for g in range(G):
        _check_f32(x[g], w[g * N:(g + 1) * N], None, yf[g], dt, exact_sums=False)


def test_grouped_with_one_group_equals_the_plain_form():
    x, w, b = _inputs(700, 520, 320, "normal", 420, "f16")
    a = _gpu(x, w, b, steps=["silu"])
    g1 = _gpu(x.reshape(1, 700, 320), w, b, steps=["silu"])
    assert torch.equal(a.view(torch.int16), g1[0].view(torch.int16))


def test_grouped_leaves_other_groups_rows_alone():
    # every group's y block is written exactly; a guard row after the last
    # group (part of the same allocation) is never touched
    G, M, N, K = 3, 131, 264, 128
    x, w, b = _grouped_inputs(G, M, N, K, "smallint", 430, "f16")
    xd, wd, bd = x.to(DEV), w.to(DEV), b.to(DEV)
    buf = torch.full((G * M + 1, N), 12345.0, dtype=torch.float16, device=DEV)
    y = buf[:G * M].view(G, M, N)
    L.contract(xd, wd, bd, out=y)
    torch.cuda.synchronize()
    assert torch.all(buf[G * M] == 12345.0)
    want = oracle.contraction_grouped(_bits(x), _bits(w), _bits(b))
    assert np.array_equal(_bits(y), want)


@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_f32_output_store_paths(dt):
    # N % 4 == 0 and a 16-byte aligned y: TMA stores of 32 x 16 FP32 boxes,
    # clipped at a ragged M; the same y 4 bytes off its alignment: direct stores
    M, N, K = 301, 264, 192
    x, w, b = _inputs(M, N, K, "smallint", 330, dt)
    y_tma = _gpu(x, w, b, out_f32=True)
    _check_f32(x, w, b, y_tma, dt, exact_sums=True)
    buf = torch.full((M * N + 1,), float("nan"), dtype=torch.float32, device=DEV)
    y_off = buf[1:].view(M, N)
    L.contract(x.to(DEV), w.to(DEV), b.to(DEV), out=y_off, out_f32=True)
    torch.cuda.synchronize()
    assert L.poot_linear_device_status(0) == L.POOT_OK
    assert torch.equal(y_off.cpu(), y_tma)
