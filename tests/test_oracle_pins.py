"""Pins for the CPU oracle: each test ties it to something other than itself.

* torch's CPU float8 casts (an independent library routine) for the byte-level
  encoder and decoder, exhaustively over every bf16 value and every byte;
* the numbers printed on the fp8_parity page (smoke steps 1-4), read from
  tests/golden/fp8_parity_constants.json;
* closed forms (power-of-two scales, one-hot GEMM rows) and exact rational
  brute force for the GEMM;
* structural invariants (column tiles are row tiles of the transpose, a tile
  of a one-tile matrix is the per-tensor case).

A plausible slip in the oracle -- a wrong bias or mantissa width, truncation
instead of ties-to-even, a lost sign, a transposed scale index, a dropped
scale factor, the current tensor leaking into its own delayed scale -- fails
at least one test here.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                   "fp8_parity_constants.json")))
FMT = {oracle.E4M3: torch.float8_e4m3fn, oracle.E5M2: torch.float8_e5m2}
BOTH = [oracle.E4M3, oracle.E5M2]


def torch_cast_bytes(v: np.ndarray, fmt: int) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32))
    return t.to(FMT[fmt]).view(torch.uint8).numpy()


# ---------------------------------------------------------------- formats

def test_constants_match_page():
    assert oracle.fmax(oracle.E4M3) == GOLD["E4M3_MAX"]["value"]
    assert oracle.fmax(oracle.E5M2) == GOLD["E5M2_MAX"]["value"]
    # torch's own finfo agrees with the page (smoke step 1's first asserts)
    assert torch.finfo(torch.float8_e4m3fn).max == GOLD["E4M3_MAX"]["value"]
    assert torch.finfo(torch.float8_e5m2).max == GOLD["E5M2_MAX"]["value"]


@pytest.mark.parametrize("fmt", BOTH)
def test_decode_all_bytes_vs_torch(fmt):
    ours = oracle.decode_table(fmt)
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(FMT[fmt]).to(
        torch.float64).numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])


def test_fixed_codes():
    e, f = oracle.E4M3, oracle.E5M2
    s1 = GOLD["smoke1"]
    assert oracle.encode_scalar(448.0, e) == 0x7E
    assert oracle.encode_scalar(57344.0, f) == 0x7B
    assert oracle.encode_scalar(s1["E4M3"]["smallest_normal"], e) == 0x08
    assert oracle.encode_scalar(s1["E5M2"]["smallest_normal"], f) == 0x04
    assert oracle.encode_scalar(2.0 ** -9, e) == 0x01      # smallest subnormal
    assert oracle.encode_scalar(2.0 ** -16, f) == 0x01
    assert oracle.encode_scalar(-0.0, e) == 0x80
    assert oracle.encode_scalar(1.0, e) == 0x38
    assert oracle.encode_scalar(1.0, f) == 0x3C
    assert oracle.encode_scalar(-2.0, e) == 0xC0


@pytest.mark.parametrize("fmt", BOTH)
def test_encode_every_bf16_vs_torch(fmt):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    v = oracle.widen(bits)
    assert np.array_equal(oracle.encode(v, fmt), torch_cast_bytes(v, fmt))


@pytest.mark.parametrize("fmt", BOTH)
def test_encode_random_fp32_vs_torch(fmt):
    rng = np.random.default_rng(123)
    bits = rng.integers(0, 2 ** 32, size=1 << 20, dtype=np.uint64).astype(np.uint32)
    v = bits.view(np.float32)
    # and values concentrated in the FP8 range, where rounding matters
    w = (rng.standard_normal(1 << 20) * 64).astype(np.float32)
    for arr in (v, w):
        assert np.array_equal(oracle.encode(arr, fmt), torch_cast_bytes(arr, fmt))


@pytest.mark.parametrize("fmt", BOTH)
def test_encode_midpoints_vs_torch(fmt):
    """Ties and near-ties between every pair of adjacent FP8 values, including
    the overflow midpoint above the largest finite value."""
    table = oracle.decode_table(fmt)
    fin = np.unique(table[np.isfinite(table) & (table >= 0)])
    step_top = fin[-1] - fin[-2]
    fin = np.append(fin, fin[-1] + step_top)        # next grid point past fmax
    mids = ((fin[1:] + fin[:-1]) / 2).astype(np.float32)
    assert np.array_equal(mids.astype(np.float64), (fin[1:] + fin[:-1]) / 2)  # exact
    cands = np.concatenate([mids, np.nextafter(mids, np.float32(np.inf)),
                            np.nextafter(mids, np.float32(0))])
    cands = np.concatenate([cands, -cands]).astype(np.float32)
    assert np.array_equal(oracle.encode(cands, fmt), torch_cast_bytes(cands, fmt))


@pytest.mark.parametrize("fmt", BOTH)
def test_encode_saturating(fmt):
    """Saturating mode equals torch's cast of the value clamped to +-fmax."""
    rng = np.random.default_rng(7)
    fm = oracle.fmax(fmt)
    v = np.concatenate([(rng.standard_normal(200000) * fm * 1.5),
                        [np.inf, -np.inf, 1e30, -1e30, 464.0, 465.0, 61440.0, -61440.0]]
                       ).astype(np.float32)
    ref = torch_cast_bytes(np.clip(v, -fm, fm), fmt)
    assert np.array_equal(oracle.encode(v, fmt, saturate=True), ref)
    nan = np.array([np.nan, -np.nan], dtype=np.float32)
    assert list(oracle.encode(nan, fmt, saturate=True)) == [0x7F, 0xFF]


# --------------------------------------------------------- amax and scale

def test_amax_brute_force():
    rng = np.random.default_rng(0)
    for n in (1, 7, 128, 1000):
        x = (rng.standard_normal(n) * 10).astype(np.float32)
        assert oracle.amax(x) == np.max(np.abs(x))
    x = np.array([-0.0, 0.0], np.float32)
    assert oracle.amax(x) == 0.0
    x = np.array([1.0, np.nan, -5.0], np.float32)
    assert np.isnan(oracle.amax(x))
    x = np.array([1.0, -np.inf], np.float32)
    assert oracle.amax(x) == np.inf
    bf = np.array([0xC2C8, 0x4120], np.uint16)   # -100.0, 10.0 as bf16
    assert oracle.amax(bf) == 100.0


def test_scale_closed_form_power_of_two():
    """amax = fmax * 2^k gives s = 2^k exactly, and x / 2^k is exact, so the
    cast is the plain cast of x * 2^-k (torch)."""
    rng = np.random.default_rng(3)
    for fmt in BOTH:
        for k in (-20, -3, 0, 5):
            s = oracle.scale_from_amax(oracle.fmax(fmt) * 2.0 ** k, fmt)
            assert s == np.float32(2.0 ** k)
            x = (rng.standard_normal(4096) * oracle.fmax(fmt) * 2.0 ** k / 4).astype(np.float32)
            assert np.array_equal(oracle.cast(x, s, fmt),
                                  torch_cast_bytes(x * np.float32(2.0 ** -k), fmt))


def test_scale_floor():
    assert oracle.scale_from_amax(0.0, oracle.E4M3) == np.float32(GOLD["scale_floor"]["value"])
    assert oracle.scale_from_amax(1e-20, oracle.E5M2) == np.float32(1e-12)
    assert np.isnan(oracle.scale_from_amax(np.nan, oracle.E4M3))


def test_scale_is_fp32_division():
    rng = np.random.default_rng(5)
    a = np.abs(rng.standard_normal(1000).astype(np.float32)) * 100
    for fmt in BOTH:
        got = np.array([oracle.scale_from_amax(v, fmt) for v in a], np.float32)
        ref = (torch.from_numpy(a) / oracle.fmax(fmt)).clamp_min(1e-12).numpy()
        assert np.array_equal(got, ref)


@pytest.mark.parametrize("fmt", BOTH)
def test_cast_is_division_near_fp8_midpoints(fmt):
    """The cast divides (x / scale in fp32, then one rounding into the
    format); multiplying by a rounded reciprocal is not the definition.
    Inputs a few ulps around midpoint * s, for every midpoint between
    neighbouring FP8 magnitudes, put the quotient next to a rounding boundary
    of the format, where the two differ in a few percent of the cases: the
    bytes must equal torch's fp32 division followed by its cast."""
    rng = np.random.default_rng(17)
    table = oracle.decode_table(fmt)
    mags = np.unique(np.abs(table[np.isfinite(table)]))
    mids = (mags[1:] + mags[:-1]) / 2
    for s in (rng.uniform(0.5, 2, 24) * 2.0 ** rng.integers(-30, 10, 24)).astype(np.float32):
        x0 = (mids * np.float64(s)).astype(np.float32).view(np.int32)
        x = np.concatenate([x0 + k for k in range(-3, 4)]).view(np.float32)
        ref = (torch.from_numpy(x) / torch.tensor(s)).to(FMT[fmt]).view(torch.uint8).numpy()
        assert np.array_equal(oracle.cast(x, s, fmt), ref)


# ------------------------------------------------------ page smoke steps

def _torch_gen(seed):
    g = torch.Generator()
    g.manual_seed(seed)
    return g


@pytest.mark.parametrize("fmt,key", [(oracle.E4M3, "E4M3"), (oracle.E5M2, "E5M2")])
def test_smoke1_roundtrip_bound(fmt, key):
    s1 = GOLD["smoke1"]
    x = (torch.randn(s1["n"], generator=_torch_gen(0)) * s1["x_std"]).numpy()
    y, s = oracle.scaled_roundtrip(x, fmt)
    normal = np.abs(x / s) >= s1[key]["smallest_normal"]
    rel = (np.abs(y - x) / np.abs(x))[normal]
    assert rel.max() <= s1[key]["rel_bound"]
    # tighter: round-to-nearest is within half a grid step of x / s
    grid = np.unique(np.abs(oracle.decode_table(fmt)[np.isfinite(oracle.decode_table(fmt))]))
    v = np.abs(x / s).astype(np.float64)
    idx = np.searchsorted(grid, v)
    lo = grid[np.clip(idx - 1, 0, grid.size - 1)]
    hi = grid[np.clip(idx, 0, grid.size - 1)]
    half = (hi - lo) / 2
    err = np.abs(np.abs(y / s) - v)
    assert np.all(err <= half * (1 + 1e-6) + 1e-30)


def test_smoke2_unscaled_cast_does_not_survive():
    s2 = GOLD["smoke2"]
    big = np.array(s2["values"], np.float32)
    q = oracle.cast(big, 1.0, oracle.E4M3)
    plain = oracle.decode(q, oracle.E4M3)
    with np.errstate(invalid="ignore"):
        rel = np.abs(plain - big) / np.abs(big)
        assert not np.any(rel < s2["min_rel_err"])
    assert list(q) == [0x7F, 0xFF, 0x7F]      # NaN, -NaN, NaN


def test_smoke3_delayed_misses_spike_current_holds_it():
    s3 = GOLD["smoke3"]
    g = _torch_gen(0)
    hist = [torch.randn(s3["n"], generator=g).abs().max().item() for _ in range(s3["history_len"])]
    act = torch.randn(s3["n"], generator=g).numpy()
    act[s3["spike_index"]] = s3["spike"]
    fmt = oracle.E4M3
    q_d, _, s_d, new_hist, nxt = oracle.quantize_delayed(act[None, :], fmt, hist, 0)
    y_d = oracle.dequantize(q_d, fmt, s_d)[0]
    y_c, s_c = oracle.scaled_roundtrip(act[None, :], fmt)
    y_c = y_c[0]
    with np.errstate(invalid="ignore"):
        assert not (abs(y_d[s3["spike_index"]] - s3["spike"]) < s3["delayed_min_err"])
    assert abs(y_c[s3["spike_index"]] - s3["spike"]) <= s3["current_max_err"]
    # the delayed scale used only the history; the spike's amax was recorded after
    assert s_d == np.float32(np.float32(max(hist)) / np.float32(448.0))
    assert new_hist[0] == s3["spike"] and nxt == 1
    # current scaling maps the spike onto the largest code exactly
    q_c, _, _ = oracle.quantize_tensor(act[None, :], fmt)
    assert q_c[0, s3["spike_index"]] == 0x7E


def test_smoke4_tiles_beat_tensor_on_outlier_row():
    s4 = GOLD["smoke4"]
    a = (torch.randn(*s4["shape"], generator=_torch_gen(0)) * s4["std"]).numpy()
    a[s4["outlier_row"]] *= s4["outlier_factor"]
    fmt = oracle.E4M3
    y_tensor, _ = oracle.scaled_roundtrip(a, fmt)
    q, sc = oracle.quantize_tile_rows(a, fmt)
    y_tile = np.stack([oracle.dequantize(q[r], fmt, sc[0, r]) for r in range(a.shape[0])])
    err_tensor = np.mean((y_tensor - a)[1:] ** 2)
    err_tile = np.mean((y_tile - a)[1:] ** 2)
    assert err_tile < err_tensor


# ------------------------------------------------ tile / block / transpose

def _page_roundtrip_torch(x: torch.Tensor, dtype, fmax):
    """The fp8_parity page's scaled_roundtrip run on torch CPU ops (a library
    implementation of the same definition), returning the fp8 bytes and the
    scale."""
    scale = (x.abs().max() / fmax).clamp_min(1e-12)
    return (x / scale).to(dtype).view(torch.uint8), scale


@pytest.mark.parametrize("fmt", BOTH)
@pytest.mark.parametrize("shape", [(3, 128), (5, 300), (130, 64)])
def test_tile_rows_vs_torch_per_tile(fmt, shape):
    rng = np.random.default_rng(11)
    x = (rng.standard_normal(shape) * rng.choice([1e-3, 1, 100], size=(shape[0], 1))
         ).astype(np.float32)
    x[0, :] = 0.0                       # an all-zero row: scale floor, zero codes
    q, sc = oracle.quantize_tile_rows(x, fmt)
    rows, cols = shape
    for r in range(rows):
        for kb in range((cols + 127) // 128):
            c0, c1 = kb * 128, min(cols, kb * 128 + 128)
            qb, s = _page_roundtrip_torch(torch.from_numpy(x[r, c0:c1]), FMT[fmt],
                                          oracle.fmax(fmt))
            assert sc[kb, r] == s.item()
            assert np.array_equal(q[r, c0:c1], qb.numpy())


@pytest.mark.parametrize("fmt", BOTH)
def test_tile_cols_is_rows_of_transpose(fmt):
    rng = np.random.default_rng(12)
    x = (rng.standard_normal((200, 48)) * 3).astype(np.float32)
    x[7, 3] = 900.0
    qt, sc = oracle.quantize_tile_cols(x, fmt)
    q2, sc2 = oracle.quantize_tile_rows(np.ascontiguousarray(x.T), fmt)
    assert np.array_equal(qt, q2) and np.array_equal(sc, sc2)


@pytest.mark.parametrize("fmt", BOTH)
def test_block_is_tensor_per_block(fmt):
    rng = np.random.default_rng(13)
    x = (rng.standard_normal((300, 260)) * 2).astype(np.float32)
    x[200:, 130:] *= 1000
    q, qt, sc = oracle.quantize_block(x, fmt, want_qt=True)
    assert np.array_equal(qt, q.T)
    for rb in range(3):
        for cb in range(3):
            blk = x[rb * 128:(rb + 1) * 128, cb * 128:(cb + 1) * 128]
            qb, s = _page_roundtrip_torch(torch.from_numpy(np.ascontiguousarray(blk)),
                                          FMT[fmt], oracle.fmax(fmt))
            assert sc[rb, cb] == s.item()
            assert np.array_equal(q[rb * 128:(rb + 1) * 128, cb * 128:(cb + 1) * 128],
                                  qb.numpy().reshape(blk.shape))


@pytest.mark.parametrize("fmt", BOTH)
def test_tensor_matches_page_and_transpose(fmt):
    rng = np.random.default_rng(14)
    x = (rng.standard_normal((77, 96)) * 5).astype(np.float32)
    q, qt, s = oracle.quantize_tensor(x, fmt, want_qt=True)
    qb, sb = _page_roundtrip_torch(torch.from_numpy(x), FMT[fmt], oracle.fmax(fmt))
    assert s == sb.item()
    assert np.array_equal(q, qb.numpy().reshape(x.shape))
    assert np.array_equal(qt, q.T)


def test_bf16_input_widening():
    rng = np.random.default_rng(15)
    f = rng.standard_normal((64, 128)).astype(np.float32)
    bits = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    wid = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    assert np.array_equal(oracle.widen(bits), wid)
    q1, s1 = oracle.quantize_tile_rows(bits, oracle.E4M3)
    q2, s2 = oracle.quantize_tile_rows(wid, oracle.E4M3)
    assert np.array_equal(q1, q2) and np.array_equal(s1, s2)


# ----------------------------------------------------------------- delayed

def test_delayed_ring_bookkeeping():
    """Feed constant tensors with known amax through 40 delayed calls and
    check each call's scale against a brute-force window of the amaxes seen
    before it."""
    fmt = oracle.E5M2
    L = 16
    hist = np.zeros(L, np.float32)
    nxt = 0
    seen = []
    rng = np.random.default_rng(16)
    for step in range(40):
        a = np.float32(rng.uniform(0.1, 50))
        x = np.full((2, 16), a, np.float32)
        x[1, 5] = -a
        _, _, s, hist, nxt = oracle.quantize_delayed(x, fmt, hist, nxt)
        window = (seen[-L:] + [0.0] * L)[:L] if seen else [0.0]
        expect = max(np.float32(max(window)) / np.float32(57344.0), np.float32(1e-12))
        assert s == np.float32(expect), step
        seen.append(float(a))
        assert nxt == (step + 1) % L


# -------------------------------------------------------------------- GEMM

def _rand_codes(rng, shape, fmt):
    """Random finite FP8 bytes."""
    table = oracle.decode_table(fmt)
    finite = np.nonzero(np.isfinite(table))[0].astype(np.uint8)
    return rng.choice(finite, size=shape)


def _expand_scales(op_rows, K, scaling, scales, transposed_block=False):
    """Dense [rows, K] matrix of per-element scales, built by np.repeat."""
    if scaling == oracle.SCALE_TENSOR:
        return np.full((op_rows, K), scales, np.float64)
    if scaling == oracle.SCALE_TILE:           # scales [kb][row]
        return np.repeat(scales.T.astype(np.float64), 128, axis=1)[:, :K]
    sc = scales.T if transposed_block else scales   # [rb][kb]
    return np.repeat(np.repeat(sc.astype(np.float64), 128, axis=0), 128, axis=1)[:op_rows, :K]


def test_gemm_exact_rational_tiny():
    rng = np.random.default_rng(20)
    M, N, K = 5, 4, 40
    for fa, fb in [(oracle.E4M3, oracle.E4M3), (oracle.E5M2, oracle.E4M3)]:
        A = _rand_codes(rng, (M, K), fa)
        B = _rand_codes(rng, (N, K), fb)
        sa, sb = np.float32(0.37), np.float32(1e-3)
        y, ab = oracle.gemm_rows(oracle.GemmOperand.tensor(A, fa, sa),
                                 oracle.GemmOperand.tensor(B, fb, sb))
        ta, tb = oracle.decode_table(fa), oracle.decode_table(fb)
        for m in range(M):
            for n in range(N):
                exact = sum(Fraction(ta[A[m, k]]) * Fraction(float(sa)) *
                            Fraction(tb[B[n, k]]) * Fraction(float(sb)) for k in range(K))
                aexact = sum(abs(Fraction(ta[A[m, k]]) * Fraction(float(sa)) *
                                 Fraction(tb[B[n, k]]) * Fraction(float(sb))) for k in range(K))
                assert abs(Fraction(y[m, n]) - exact) <= Fraction(1, 2 ** 50) * aexact
                assert abs(Fraction(ab[m, n]) - aexact) <= Fraction(1, 2 ** 50) * aexact


@pytest.mark.parametrize("kind", ["tensor", "tile_block", "tile_tile", "block_t"])
def test_gemm_vs_numpy_dense(kind):
    rng = np.random.default_rng(21)
    M, N, K = 150, 140, 300
    fa, fb = oracle.E4M3, oracle.E5M2
    A = _rand_codes(rng, (M, K), fa)
    B = _rand_codes(rng, (N, K), fb)
    nkb = (K + 127) // 128
    if kind == "tensor":
        opA = oracle.GemmOperand.tensor(A, fa, 0.5)
        opB = oracle.GemmOperand.tensor(B, fb, 3.0)
        SA = _expand_scales(M, K, oracle.SCALE_TENSOR, 0.5)
        SB = _expand_scales(N, K, oracle.SCALE_TENSOR, 3.0)
    elif kind in ("tile_block", "block_t"):
        sa = rng.uniform(0.1, 2, size=(nkb, M)).astype(np.float32)
        sb = rng.uniform(0.1, 2, size=((N + 127) // 128, nkb)).astype(np.float32)
        opA = oracle.GemmOperand.tile(A, fa, sa)
        SA = _expand_scales(M, K, oracle.SCALE_TILE, sa)
        if kind == "tile_block":
            opB = oracle.GemmOperand.block(B, fb, sb)
            SB = _expand_scales(N, K, oracle.SCALE_BLOCK, sb)
        else:
            sbt = np.ascontiguousarray(sb.T)                  # [kb][nb]
            opB = oracle.GemmOperand.block(B, fb, sbt, transposed=True)
            SB = _expand_scales(N, K, oracle.SCALE_BLOCK, sbt, transposed_block=True)
    else:
        sa = rng.uniform(0.1, 2, size=(nkb, M)).astype(np.float32)
        sb = rng.uniform(0.1, 2, size=(nkb, N)).astype(np.float32)
        opA = oracle.GemmOperand.tile(A, fa, sa)
        opB = oracle.GemmOperand.tile(B, fb, sb)
        SA = _expand_scales(M, K, oracle.SCALE_TILE, sa)
        SB = _expand_scales(N, K, oracle.SCALE_TILE, sb)
    Ad = oracle.decode_table(fa)[A] * SA
    Bd = oracle.decode_table(fb)[B] * SB
    ref = Ad @ Bd.T
    y, ab = oracle.gemm_rows(opA, opB)
    assert np.all(np.abs(y - ref) <= 1e-13 * ab + 1e-300)
    assert np.allclose(ab, np.abs(Ad) @ np.abs(Bd).T, rtol=1e-13)
    # the point interface computes the same numbers
    ms = rng.integers(0, M, 50)
    ns = rng.integers(0, N, 50)
    yp, abp = oracle.gemm_points(opA, opB, ms, ns)
    assert np.array_equal(yp, y[ms, ns]) and np.array_equal(abp, ab[ms, ns])


def test_gemm_one_hot_closed_form():
    """B row n has one nonzero code at column n: C[m, n] = A_deq[m, n] * B_deq[n, n]."""
    rng = np.random.default_rng(22)
    M, N, K = 9, 6, 16
    A = _rand_codes(rng, (M, K), oracle.E4M3)
    B = np.zeros((N, K), np.uint8)
    for n in range(N):
        B[n, n] = 0x38 + n          # 1.0, 1.125, ... in E4M3
    y, _ = oracle.gemm_rows(oracle.GemmOperand.tensor(A, oracle.E4M3, 2.0),
                            oracle.GemmOperand.tensor(B, oracle.E4M3, 0.25))
    ta = oracle.decode_table(oracle.E4M3)
    for m in range(M):
        for n in range(N):
            assert y[m, n] == ta[A[m, n]] * 2.0 * ta[0x38 + n] * 0.25


def test_gemm_transpose_symmetry():
    rng = np.random.default_rng(23)
    A = _rand_codes(rng, (20, 256), oracle.E4M3)
    B = _rand_codes(rng, (12, 256), oracle.E5M2)
    sa = rng.uniform(0.5, 1.5, size=(2, 20)).astype(np.float32)
    sb = rng.uniform(0.5, 1.5, size=(2, 12)).astype(np.float32)
    y1, _ = oracle.gemm_rows(oracle.GemmOperand.tile(A, oracle.E4M3, sa),
                             oracle.GemmOperand.tile(B, oracle.E5M2, sb))
    y2, _ = oracle.gemm_rows(oracle.GemmOperand.tile(B, oracle.E5M2, sb),
                             oracle.GemmOperand.tile(A, oracle.E4M3, sa))
    assert np.allclose(y1, y2.T, rtol=1e-14, atol=0)


def test_bf16_ulp_vs_torch_spacing():
    """The bf16 output allowance of the GEMM bound is one bf16 spacing at the
    reference value: the gap from a bf16 number to the next one up, taken
    from torch's bf16 bit patterns, over normal magnitudes of both signs."""
    rng = np.random.default_rng(24)
    v = (rng.standard_normal(5000) * 2.0 ** rng.integers(-100, 100, 5000)).astype(np.float32)
    t = torch.from_numpy(v).to(torch.bfloat16)
    a = t.abs()
    up = (a.view(torch.int16) + 1).view(torch.bfloat16)
    spacing = (up.double() - a.double()).numpy()
    assert np.array_equal(oracle.bf16_ulp(t.double().numpy()), spacing)
    # and rounding any value to bf16 moves it by at most half of that spacing
    assert np.all(np.abs(t.double().numpy() - v.astype(np.float64))
                  <= oracle.bf16_ulp(v.astype(np.float64)) / 2)


def test_fp8matmul_roles_vs_page_torch():
    """Fprop / Dgrad / Wgrad on the tiny linear match the page's FP8Matmul
    (forward xq @ wq.T, backward gq @ wq and gq.T @ xq, fp32 on dequantised
    operands, run here with torch CPU ops) within fp32 rounding."""
    import workloads
    x, w, g = workloads.tiny_linear()
    E4, E5 = torch.float8_e4m3fn, torch.float8_e5m2

    def rt(t, dt, fm):
        s = (t.abs().max() / fm).clamp_min(1e-12)
        return (t / s).to(dt).float() * s

    xq, wq, gq = rt(x, E4, 448.0), rt(w, E4, 448.0), rt(g, E5, 57344.0)
    ref = {"fprop": xq @ wq.T, "dgrad": gq @ wq, "wgrad": gq.T @ xq}

    qx, qxt, sx = oracle.quantize_tensor(x.numpy(), oracle.E4M3, want_qt=True)
    qw, qwt, sw = oracle.quantize_tensor(w.numpy(), oracle.E4M3, want_qt=True)
    qg, qgt, sg = oracle.quantize_tensor(g.numpy(), oracle.E5M2, want_qt=True)
    T = oracle.GemmOperand.tensor
    got = {
        "fprop": oracle.gemm_rows(T(qx, oracle.E4M3, sx), T(qw, oracle.E4M3, sw)),
        "dgrad": oracle.gemm_rows(T(qg, oracle.E5M2, sg), T(qwt, oracle.E4M3, sw)),
        "wgrad": oracle.gemm_rows(T(qgt, oracle.E5M2, sg), T(qxt, oracle.E4M3, sx)),
    }
    for role in ref:
        y, ab = got[role]
        r = ref[role].double().numpy()
        assert y.shape == r.shape
        assert np.all(np.abs(y - r) <= 1e-6 * ab + 1e-12), role


# ---------------------------------------------------------------- row-wise

@pytest.mark.parametrize("fmt", BOTH)
def test_rowwise_is_page_roundtrip_per_row_and_column(fmt):
    """Row-wise scaling applies the page's scaled_roundtrip to each whole row
    (and to each whole column for the transposed copy)."""
    rng = np.random.default_rng(30)
    x = (rng.standard_normal((40, 352)) * rng.choice([1e-2, 1, 50], size=(40, 1))).astype(np.float32)
    x[3, :] = 0.0
    q, qs, qt, qts = oracle.quantize_rowwise(x, fmt, rows=True, cols=True)
    for r in range(x.shape[0]):
        qb, sb = _page_roundtrip_torch(torch.from_numpy(x[r].copy()), FMT[fmt], oracle.fmax(fmt))
        assert qs[r] == sb.item() and np.array_equal(q[r], qb.numpy())
    for c in range(x.shape[1]):
        qb, sb = _page_roundtrip_torch(torch.from_numpy(x[:, c].copy()), FMT[fmt],
                                       oracle.fmax(fmt))
        assert qts[c] == sb.item() and np.array_equal(qt[c], qb.numpy())


def test_rowwise_equals_tiles_when_a_row_is_one_tile():
    rng = np.random.default_rng(31)
    x = (rng.standard_normal((64, 128)) * 3).astype(np.float32)
    q, qs, _, _ = oracle.quantize_rowwise(x, oracle.E4M3)
    q2, s2 = oracle.quantize_tile_rows(x, oracle.E4M3)
    assert np.array_equal(q, q2) and np.array_equal(qs, s2[0])


def test_gemm_row_scales_vs_numpy():
    rng = np.random.default_rng(32)
    M, N, K = 70, 90, 260
    A = _rand_codes(rng, (M, K), oracle.E4M3)
    B = _rand_codes(rng, (N, K), oracle.E5M2)
    sa = rng.uniform(0.1, 2, M).astype(np.float32)
    sb = rng.uniform(0.1, 2, N).astype(np.float32)
    y, ab = oracle.gemm_rows(oracle.GemmOperand.row(A, oracle.E4M3, sa),
                             oracle.GemmOperand.row(B, oracle.E5M2, sb))
    ref = (oracle.decode_table(oracle.E4M3)[A] * sa[:, None].astype(np.float64)) @ \
          (oracle.decode_table(oracle.E5M2)[B] * sb[:, None].astype(np.float64)).T
    assert np.all(np.abs(y - ref) <= 1e-13 * ab + 1e-300)


# ------------------------------------------------------------------ MXFP8
# The pages name MXFP8 (the SpikingJelly precision page's fp8_recipe list, the
# blog repost's Blackwell baseline) but give no encoding; the oracle follows
# the OCP Microscaling Formats v1.0 specification.  These pins tie it to
# torch's E8M0 and FP8 casts, to exact rational arithmetic and to a
# brute-force search, not to its own code.

EMAX_ELEM = {oracle.E4M3: 8, oracle.E5M2: 15}   # 448 = 1.75 * 2^8, 57344 = 1.75 * 2^15


def test_e8m0_decode_all_codes_vs_torch():
    ours = oracle.e8m0_decode(np.arange(256, dtype=np.uint8))
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(
        torch.float8_e8m0fnu).to(torch.float64).numpy()
    assert np.isnan(ours[255]) and np.isnan(ref[255])
    assert np.array_equal(ours[:255], ref[:255])


@pytest.mark.parametrize("fmt", BOTH)
def test_emax_elem_from_the_page_constants(fmt):
    """emax_elem is the binade of the page's largest value: fmax / 2^emax in [1, 2)."""
    fm = GOLD["E4M3_MAX" if fmt == oracle.E4M3 else "E5M2_MAX"]["value"]
    assert 1.0 <= fm / 2.0 ** EMAX_ELEM[fmt] < 2.0
    # an amax equal to fmax gets scale 1 (code 127): the block needs no scaling
    assert oracle.mx_scale_code(fm, fmt) == 127


@pytest.mark.parametrize("fmt", BOTH)
def test_mx_scale_bracket_in_exact_rationals(fmt):
    """X = 2^(code-127) puts the block max in [2^emax, 2^(emax+1)) * X (floor of
    log2 minus emax_elem), checked with Fractions, except where the E8M0 range
    clamps the exponent at -127."""
    rng = np.random.default_rng(30)
    mags = np.concatenate([
        2.0 ** rng.uniform(-149, 127.9, 4000),
        2.0 ** np.arange(-149, 128, dtype=np.float64),             # powers of two
        np.nextafter(np.float32(2.0) ** np.arange(-120, 127), np.float32(0)),  # just below
    ]).astype(np.float32)
    mags = mags[np.isfinite(mags) & (mags > 0)]
    lo, hi = Fraction(2) ** EMAX_ELEM[fmt], Fraction(2) ** (EMAX_ELEM[fmt] + 1)
    for a in mags:
        code = oracle.mx_scale_code(float(a), fmt)
        assert 0 <= code <= 254
        X = Fraction(2) ** (code - 127)
        r = Fraction(float(a)) / X
        if code == 0:
            assert r < hi          # clamped at the bottom of E8M0
        else:
            assert lo <= r < hi, (a, code)


def test_mx_scale_special_cases():
    for fmt in BOTH:
        assert oracle.mx_scale_code(0.0, fmt) == 0
        assert oracle.mx_scale_code(float("nan"), fmt) == 255
        assert oracle.mx_scale_code(float("inf"), fmt) == 255
        # amax = 448 * 2^k -> X = 2^k exactly (E4M3), 57344 * 2^k likewise for E5M2
        fm = oracle.fmax(fmt)
        for k in (-20, -3, 0, 5, 40):
            assert oracle.mx_scale_code(fm * 2.0 ** k, fmt) == 127 + k
        # a block max so small that floor(log2 amax) - emax_elem falls below E8M0's
        # -127 takes the clamped exponent -127 (code 0), as an all-zero block does
        for tiny in (2.0 ** -120, 2.0 ** -140, 2.0 ** -149):
            assert oracle.mx_scale_code(tiny, fmt) == 0


def _nearest_code_brute(v: Fraction, fmt: int) -> int:
    """The finite FP8 code nearest to v, ties to the even code (mantissa LSB
    0), magnitudes beyond the largest finite value clamped -- by search over
    every finite code."""
    table = oracle.decode_table(fmt)
    best = None
    for c in range(256):
        t = table[c]
        if not np.isfinite(t):
            continue
        d = abs(Fraction(t) - v)
        key = (d, c & 1)
        if best is None or key < best[0]:
            best = (key, c)
    c = best[1]
    # zero keeps the sign of the value (a negative value that rounds to zero is -0)
    if table[c] == 0:
        c = 0x80 if v < 0 else 0x00
    return c


@pytest.mark.parametrize("fmt", BOTH)
def test_mx_elements_are_the_nearest_value_brute_force(fmt):
    rng = np.random.default_rng(31)
    # three rows: moderate values with a wide spread, values that hit the
    # clamp (block max just below the next power of two), and tiny values
    x = np.empty((3, 64), np.float32)
    x[0] = rng.standard_normal(64) * 2.0 ** rng.integers(-6, 6, 64)
    x[1] = rng.uniform(-1, 1, 64)
    x[1, 5] = 1.999
    x[1, 40] = -1.99
    x[2] = rng.standard_normal(64) * 1e-30
    q, sc = oracle.quantize_mx_rows(x, fmt)
    for r in range(3):
        for j in range(2):
            X = Fraction(2) ** (int(sc[r, j]) - 127)
            for c in range(32 * j, 32 * j + 32):
                want = _nearest_code_brute(Fraction(float(x[r, c])) / X, fmt)
                assert q[r, c] == want, (r, c, x[r, c], q[r, c], want)


@pytest.mark.parametrize("fmt", BOTH)
def test_mx_elements_vs_torch_cast(fmt):
    """Bytes equal torch's CPU cast of clamp(V / X, +-fmax) (bf16 inputs)."""
    rng = np.random.default_rng(32)
    x = (torch.from_numpy(rng.standard_normal((64, 256)).astype(np.float32)) *
         torch.from_numpy(2.0 ** rng.integers(-10, 10, (64, 1)).astype(np.float32)))
    xb = x.to(torch.bfloat16)
    q, sc = oracle.quantize_mx_rows(xb.view(torch.int16).numpy().view(np.uint16), fmt)
    X = torch.from_numpy(np.ldexp(1.0, sc.astype(np.int64) - 127)).repeat_interleave(32, dim=1)
    fm = oracle.fmax(fmt)
    v = (xb.double() / X).clamp(-fm, fm).float()       # exact: X is a power of two
    ref = v.to(FMT[fmt]).view(torch.uint8).numpy()
    assert np.array_equal(q, ref)


@pytest.mark.parametrize("fmt", BOTH)
def test_mx_zero_nonfinite_and_ragged_blocks(fmt):
    x = np.zeros((2, 80), np.float32)
    x[0, :32] = -0.0                 # all-zero block with negative zeros
    x[0, 32:64] = np.linspace(-3, 3, 32)
    x[0, 50] = np.nan                # a NaN poisons its block only
    # ragged last block (16 elements) of values exact in both formats
    x[1, 64:80] = [0.125, 0.1875, 0.25, 0.375, 0.5, 0.75, 1, 1.5, 2, 3, 4, 6, 8, 12, 14, 16]
    q, sc = oracle.quantize_mx_rows(x, fmt)
    assert sc.shape == (2, 3)
    assert sc[0, 0] == 0 and np.all(q[0, :32] == 0x80)
    assert sc[0, 1] == 255 and np.all(q[0, 32:64] == 0x7F)
    assert sc[1, 0] == 0 and sc[1, 1] == 0
    assert sc[1, 2] == 127 + 4 - EMAX_ELEM[fmt]         # max 16 = 2^4
    d = oracle.decode_table(fmt)[q[1, 64:80]] * 2.0 ** (int(sc[1, 2]) - 127)
    assert np.array_equal(d, x[1, 64:80].astype(np.float64))


@pytest.mark.parametrize("fmt", BOTH)
def test_mx_cols_is_rows_of_transpose(fmt):
    rng = np.random.default_rng(33)
    x = (rng.standard_normal((96, 48)) * 3).astype(np.float32)
    qt, sct = oracle.quantize_mx_cols(x, fmt)
    q2, sc2 = oracle.quantize_mx_rows(np.ascontiguousarray(x.T), fmt)
    assert np.array_equal(qt, q2) and np.array_equal(sct, sc2)


@pytest.mark.parametrize("fmt,rel", [(oracle.E4M3, 2.0 ** -4), (oracle.E5M2, 2.0 ** -3)])
def test_mx_roundtrip_error_bound(fmt, rel):
    """Elements whose |V/X| is a normal at most fmax come back within half an
    ulp (the smoke step 1 bound); those between fmax and 2^(emax+1) clamp to
    fmax * X."""
    rng = np.random.default_rng(34)
    x = (rng.standard_normal((128, 128)) * 5).astype(np.float32)
    q, sc = oracle.quantize_mx_rows(x, fmt)
    X = np.repeat(np.ldexp(1.0, sc.astype(np.int64) - 127), 32, axis=1)
    d = oracle.decode_table(fmt)[q] * X
    r = np.abs(x.astype(np.float64)) / X
    fm = oracle.fmax(fmt)
    normal = (r >= 2.0 ** (1 - (7 if fmt == oracle.E4M3 else 15))) & (r <= fm)
    err = np.abs(d - x) / np.abs(x)
    assert np.all(err[normal] <= rel)
    over = r > fm
    assert np.all(np.abs(d[over]) == fm * X[over])


def test_gemm_mx_exact_rational_tiny():
    rng = np.random.default_rng(35)
    M, N, K = 4, 3, 80          # three 32-blocks, the last one partial
    for fa, fb in [(oracle.E4M3, oracle.E4M3), (oracle.E5M2, oracle.E4M3)]:
        A = _rand_codes(rng, (M, K), fa)
        B = _rand_codes(rng, (N, K), fb)
        sa = rng.integers(100, 150, (M, 3)).astype(np.uint8)
        sb = rng.integers(100, 150, (N, 3)).astype(np.uint8)
        y, ab = oracle.gemm_rows(oracle.GemmOperand.mx(A, fa, sa), oracle.GemmOperand.mx(B, fb, sb))
        ta, tb = oracle.decode_table(fa), oracle.decode_table(fb)
        for m in range(M):
            for n in range(N):
                terms = [Fraction(ta[A[m, k]]) * Fraction(2) ** (int(sa[m, k // 32]) - 127) *
                         Fraction(tb[B[n, k]]) * Fraction(2) ** (int(sb[n, k // 32]) - 127)
                         for k in range(K)]
                exact = sum(terms)
                aexact = sum(abs(t) for t in terms)
                assert abs(Fraction(y[m, n]) - exact) <= Fraction(1, 2 ** 50) * aexact
                assert abs(Fraction(ab[m, n]) - aexact) <= Fraction(1, 2 ** 50) * aexact


def test_gemm_mx_vs_numpy_dense():
    rng = np.random.default_rng(36)
    M, N, K = 70, 90, 256
    fa, fb = oracle.E5M2, oracle.E4M3
    A = _rand_codes(rng, (M, K), fa)
    B = _rand_codes(rng, (N, K), fb)
    sa = rng.integers(110, 140, (M, K // 32)).astype(np.uint8)
    sb = rng.integers(110, 140, (N, K // 32)).astype(np.uint8)
    Ad = oracle.decode_table(fa)[A] * np.repeat(np.ldexp(1.0, sa.astype(np.int64) - 127), 32, 1)
    Bd = oracle.decode_table(fb)[B] * np.repeat(np.ldexp(1.0, sb.astype(np.int64) - 127), 32, 1)
    y, ab = oracle.gemm_rows(oracle.GemmOperand.mx(A, fa, sa), oracle.GemmOperand.mx(B, fb, sb))
    assert np.all(np.abs(y - Ad @ Bd.T) <= 1e-13 * ab + 1e-300)
    assert np.allclose(ab, np.abs(Ad) @ np.abs(Bd).T, rtol=1e-13)
