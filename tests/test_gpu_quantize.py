"""GPU parity of steps a1-a3 (amax, scale, cast) against the CPU oracle.

Everything here is integer/byte work with a single correct answer: FP8 bytes
and fp32 scales must match the oracle bit for bit.  Inputs are the seeded
workloads plus edge cases: ragged tiles, empty tensors, all-zero tiles,
signed zeros, NaN/Inf, overflow under delayed scaling, every bf16 value.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.gpu_helpers import assert_bytes_equal, assert_f32_bits_equal, f32, to_oracle, u8

pytestmark = pytest.mark.gpu

FMTS = [0, 1]   # E4M3, E5M2 (same numbering in oracle and binding)


@pytest.fixture(scope="module")
def fq():
    import scaled_quantize_fp8_warp_gb300 as fq
    from scaled_quantize_fp8_warp_gb300 import build_lib
    build_lib.build()
    fq.load_library()
    assert fq.device_supported(), "this suite needs a compute capability 10.3 device"
    return fq


def _dev(x):
    return x.cuda()


# -------------------------------------------------------------------- amax

@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("n", [0, 1, 7, 8, 9, 1000, (1 << 20) + 3, 3 * (1 << 22) + 5])
def test_amax(fq, dtype, n):
    x = workloads.normal((n,), 3.0, 100 + n % 97, dtype=dtype)
    got = fq.fp8_amax(_dev(x)).item()
    ref = oracle.amax(to_oracle(x))
    assert np.float32(got).view(np.uint32) == np.float32(ref).view(np.uint32)


def test_amax_special(fq):
    x = torch.tensor([-0.0, 0.0, -3.5, 2.0], dtype=torch.float32)
    assert fq.fp8_amax(_dev(x)).item() == 3.5
    x = torch.tensor([1.0, float("-inf"), 2.0], dtype=torch.bfloat16)
    assert fq.fp8_amax(_dev(x)).item() == float("inf")
    x = torch.zeros(4099, dtype=torch.bfloat16)
    x[4097] = float("nan")
    assert np.isnan(fq.fp8_amax(_dev(x)).item())
    # the call overwrites, it does not accumulate into a stale value
    out = torch.full((1,), 1e30, device="cuda")
    fq.fp8_amax(_dev(torch.ones(64)), out=out)
    assert out.item() == 1.0


# ------------------------------------------------------- per-tensor current

@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("dtype,shape", [
    (torch.float32, (512, 32)), (torch.float32, (64, 32)), (torch.float32, (512, 64)),
    (torch.bfloat16, (300, 160)), (torch.bfloat16, (400, 272)), (torch.bfloat16, (16, 16)),
    (torch.bfloat16, (1, 4096)), (torch.bfloat16, (2049, 4112)),
])
def test_quantize_tensor(fq, fmt, dtype, shape):
    x = workloads.normal(shape, 2.0, 11, dtype=dtype)
    want_qt = shape[0] % 16 == 0
    xd = _dev(x)
    amax = fq.fp8_amax(xd)
    q, qt, s = fq.fp8_quantize_tensor(xd, fmt, amax, want_q=True, want_qt=want_qt)
    rq, rqt, rs = oracle.quantize_tensor(to_oracle(x), fmt, want_qt=want_qt)
    assert_f32_bits_equal(f32(s), np.array([rs], np.float32), "scale")
    assert_bytes_equal(u8(q), rq, "q")
    if want_qt:
        assert_bytes_equal(u8(qt), rqt, "q_t")


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("saturate", [False, True])
def test_every_bf16_value_many_scales(fq, fmt, saturate):
    """All 65536 bf16 bit patterns (NaN, Inf, subnormals, signed zeros) cast
    with 48 scales, including scales far below the data's amax (overflow,
    NaN/Inf codes, saturation) and far above it (underflow to signed zero).
    The cast uses the amax it is given, so any scale can be reached."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(512, 128)
    x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)
    xd = _dev(x)
    rng = np.random.default_rng(0)
    amaxes = np.concatenate([
        [448.0, 57344.0, 1.0, 3.0, 1e-30, 1e30, 0.0, 3.4e38],
        np.exp(rng.uniform(np.log(1e-20), np.log(1e20), 40)),
    ]).astype(np.float32)
    for a in amaxes:
        amax = torch.tensor([a], dtype=torch.float32, device="cuda")
        q, qt, s = fq.fp8_quantize_tensor(xd, fmt, amax, want_q=True, want_qt=True,
                                          saturate=saturate)
        rs = oracle.scale_from_amax(a, fmt)
        rq, rqt, _ = oracle.quantize_tensor(bits, fmt, s=rs, saturate=saturate, want_qt=True)
        assert_f32_bits_equal(f32(s), np.array([rs], np.float32), f"scale amax={a}")
        assert_bytes_equal(u8(q), rq, f"q amax={a}")
        assert_bytes_equal(u8(qt), rqt, f"q_t amax={a}")


@pytest.mark.parametrize("fmt", FMTS)
def test_random_fp32_bits_random_scales(fq, fmt):
    """Random fp32 bit patterns within the FP8 range of random scales: the
    division and rounding on inputs bf16 cannot express."""
    rng = np.random.default_rng(1)
    for trial in range(6):
        a = np.float32(np.exp(rng.uniform(np.log(1e-10), np.log(1e10))))
        s = oracle.scale_from_amax(a, fmt)
        mant = rng.integers(0, 1 << 23, size=(256, 512), dtype=np.uint64).astype(np.uint32)
        v = (mant | 0x3F800000).view(np.float32) * rng.choice([-1, 1], size=mant.shape)
        v = (v * np.float32(s) * np.exp2(rng.integers(-12, 9, size=mant.shape))).astype(np.float32)
        xd = torch.from_numpy(v).cuda()
        q, qt, _ = fq.fp8_quantize_tensor(xd, fmt, torch.tensor([a], device="cuda"),
                                          want_qt=True)
        rq, rqt, _ = oracle.quantize_tensor(v, fmt, s=s, want_qt=True)
        assert_bytes_equal(u8(q), rq, f"q trial {trial}")
        assert_bytes_equal(u8(qt), rqt, f"q_t trial {trial}")


def test_empty_tensor(fq):
    x = torch.empty((0, 32), dtype=torch.bfloat16, device="cuda")
    amax = fq.fp8_amax(x)
    assert amax.item() == 0.0
    q, qt, s = fq.fp8_quantize_tensor(x, 0, amax, want_qt=True)
    assert q.shape == (0, 32) and qt.shape == (32, 0)
    assert s.item() == np.float32(1e-12)


# ---------------------------------------------------------------- delayed

@pytest.mark.parametrize("fmt", FMTS)
def test_delayed_sequence(fq, fmt):
    """20 consecutive delayed calls: scale, bytes and the history ring match
    the oracle after every call; a spike of 40 overflows (NaN/Inf codes)."""
    hist0 = [float(oracle.amax(to_oracle(d))) for d in
             workloads.history_draws((4096,), std=1e-3)]
    h = fq.History(initial=hist0)
    ref_h, ref_next = np.array(hist0, np.float32), 0
    for step in range(20):
        x, _ = workloads.with_spikes((256, 512), 1e-3, 40.0, 1e5, 500 + step)
        if step == 7:
            x = x * 50      # a jump in magnitude the history has not seen
        q, qt, s = fq.fp8_quantize_delayed(_dev(x), fmt, h, want_qt=True)
        rq, rqt, rs, ref_h, ref_next = oracle.quantize_delayed(to_oracle(x), fmt, ref_h, ref_next,
                                                               want_qt=True)
        assert_f32_bits_equal(f32(s), np.array([rs], np.float32), f"scale step {step}")
        assert_bytes_equal(u8(q), rq, f"q step {step}")
        assert_bytes_equal(u8(qt), rqt, f"q_t step {step}")
        amax_ring, nxt, last = h.state()
        assert_f32_bits_equal(np.array(amax_ring, np.float32), ref_h, f"history step {step}")
        assert nxt == ref_next and np.float32(last) == rs
        assert h.scratch() == (0, 0)
        if step == 0:
            # the first call's scale comes from spike-free history: its 40.0
            # spikes cannot be represented (NaN for E4M3, Inf for E5M2)
            spike_codes = u8(q)[to_oracle(x) == np.uint16(0x4220)]
            assert spike_codes.size and np.all((spike_codes & 0x7F) == (0x7C if fmt else 0x7F))


def test_delayed_saturating(fq):
    h = fq.History(initial=[1e-3] * 16)
    x, _ = workloads.with_spikes((128, 256), 1e-3, 40.0, 1e4, 77)
    q, _, s = fq.fp8_quantize_delayed(_dev(x), 1, h, saturate=True)
    rq, _, rs, _, _ = oracle.quantize_delayed(to_oracle(x), 1, [1e-3] * 16, 0, saturate=True)
    assert_bytes_equal(u8(q), rq, "q")


# ------------------------------------------------------------------- tiles

TILE_SHAPES = [(128, 128), (200, 176), (16, 4096), (1000, 272), (256, 48), (130, 16)]


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("shape", TILE_SHAPES)
@pytest.mark.parametrize("which", ["rows", "cols", "both"])
def test_tile1x128(fq, fmt, dtype, shape, which):
    rows, cols = which in ("rows", "both"), which in ("cols", "both")
    if cols and shape[0] % 16:
        pytest.skip("column tiles need rows % 16 == 0")
    x, _ = workloads.with_outlier_rows(shape, 0.5, 0.05, 300.0, 21, dtype=dtype)
    x[: min(3, shape[0]), :].zero_()                   # all-zero tiles
    if shape[0] > 5:
        x[5, 0] = -0.0
    q, qs, qt, qts = fq.fp8_quantize_tile1x128(_dev(x), fmt, rows=rows, cols=cols)
    xo = to_oracle(x)
    if rows:
        rq, rs = oracle.quantize_tile_rows(xo, fmt)
        assert_f32_bits_equal(f32(qs), rs, "row tile scales")
        assert_bytes_equal(u8(q), rq, "row tile bytes")
    if cols:
        rqt, rts = oracle.quantize_tile_cols(xo, fmt)
        assert_f32_bits_equal(f32(qts), rts, "column tile scales")
        assert_bytes_equal(u8(qt), rqt, "column tile bytes")


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("shape", [(128, 128), (300, 272), (16, 16), (512, 4096), (4096, 1040)])
def test_block128(fq, fmt, shape):
    x = workloads.normal(shape, 0.02, 31)
    x[:, : min(128, shape[1])] *= 100
    want_qt = shape[0] % 16 == 0
    q, qt, sc = fq.fp8_quantize_block128x128(_dev(x), fmt, want_q=True, want_qt=want_qt)
    rq, rqt, rsc = oracle.quantize_block(to_oracle(x), fmt, want_qt=want_qt)
    assert_f32_bits_equal(f32(sc), rsc, "block scales")
    assert_bytes_equal(u8(q), rq, "q")
    if want_qt:
        assert_bytes_equal(u8(qt), rqt, "q_t")


# ------------------------------------------------- the 8192x4096 activation

@pytest.fixture(scope="module")
def activation():
    x, outlier_rows = workloads.quantize_activation()
    return x, outlier_rows


def test_activation_tiles_full_size(fq, activation):
    """Bandwidth workload at full size, E4M3, 1x128 tiles: every byte and
    scale, plus the MSE of the non-outlier rows (tiles below per-tensor)."""
    x, outlier_rows = activation
    xo = to_oracle(x)
    q, qs, _, _ = fq.fp8_quantize_tile1x128(_dev(x), 0, rows=True)
    rq, rs = oracle.quantize_tile_rows(xo, 0)
    assert_f32_bits_equal(f32(qs), rs, "tile scales")
    assert_bytes_equal(u8(q), rq, "tile bytes")
    amax = fq.fp8_amax(_dev(x))
    qt_, _, s = fq.fp8_quantize_tensor(_dev(x), 0, amax)
    tq, _, ts = oracle.quantize_tensor(xo, 0)
    assert_bytes_equal(u8(qt_), tq, "tensor bytes")
    keep = np.ones(x.shape[0], bool)
    keep[outlier_rows.numpy()] = False
    xf = oracle.widen(xo)
    table = oracle.decode_table(0).astype(np.float32)
    d_tile = table[u8(q)] * np.repeat(f32(qs).T, 128, axis=1)
    d_tensor = table[u8(qt_)] * f32(s)[0]
    mse_tile = np.mean((d_tile[keep] - xf[keep]) ** 2)
    mse_tensor = np.mean((d_tensor[keep] - xf[keep]) ** 2)
    assert mse_tile < mse_tensor


# --------------------------------------------------------------- row-wise

@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("shape", [(128, 128), (200, 176), (16, 4096), (1024, 272), (272, 48)])
@pytest.mark.parametrize("which", ["rows", "cols", "both"])
def test_rowwise(fq, fmt, dtype, shape, which):
    rows, cols = which in ("rows", "both"), which in ("cols", "both")
    if cols and shape[0] % 16:
        pytest.skip("column scales (transposed copy) need rows % 16 == 0")
    x, _ = workloads.with_outlier_rows(shape, 0.5, 0.05, 300.0, 41, dtype=dtype)
    x[: min(2, shape[0]), :].zero_()
    x[:, : min(16, shape[1])] *= 20
    q, qs, qt, qts = fq.fp8_quantize_rowwise(x.cuda(), fmt, rows=rows, cols=cols)
    rq, rqs, rqt, rqts = oracle.quantize_rowwise(to_oracle(x), fmt, rows=rows, cols=cols)
    if rows:
        assert_f32_bits_equal(f32(qs), rqs, "row scales")
        assert_bytes_equal(u8(q), rq, "row bytes")
    if cols:
        assert_f32_bits_equal(f32(qts), rqts, "column scales")
        assert_bytes_equal(u8(qt), rqt, "column bytes")


def test_rowwise_repeated_calls_reset_accumulators(fq):
    """The scale arrays double as amax accumulators: a second call with
    smaller data must not keep the first call's larger amaxes."""
    x = workloads.normal((256, 512), 10.0, 42).cuda()
    q, qs, qt, qts = fq.fp8_quantize_rowwise(x, 0, rows=True, cols=True)
    y = (x * 1e-3).contiguous()
    fq.fp8_quantize_rowwise(y, 0, rows=True, cols=True, q=q, q_scales=qs, q_t=qt, qt_scales=qts)
    rq, rqs, rqt, rqts = oracle.quantize_rowwise(to_oracle(y.cpu()), 0, rows=True, cols=True)
    assert_f32_bits_equal(f32(qs), rqs, "row scales")
    assert_f32_bits_equal(f32(qts), rqts, "column scales")
    assert_bytes_equal(u8(q), rq, "row bytes")
    assert_bytes_equal(u8(qt), rqt, "column bytes")


# ------------------------------------------- amax + cast in one call

@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("shape,which", [
    ((128, 128), "q"), ((200, 176), "q"), ((1024, 272), "both"), ((272, 48), "qt"),
    ((2048, 2048), "both"),        # 8 MiB of bf16: one cooperative launch (fp32: two kernels)
    ((8192, 4096), "both"),        # the activation, 64 MiB: two kernels
])
def test_quantize_tensor_current_matches_two_calls(fq, dtype, shape, which):
    """fp8_quantize_tensor_current equals fp8_amax + fp8_quantize_tensor bit
    for bit (amax, scale, q, q_t) and the oracle's per-tensor quantisation."""
    x, _ = workloads.with_outlier_rows(shape, 1.0, 0.02, 300.0, 44, dtype=dtype)
    xd = x.cuda()
    want_q, want_qt = which in ("q", "both"), which in ("qt", "both")
    q, qt, am, sc = fq.fp8_quantize_tensor_current(xd, 0, want_q=want_q, want_qt=want_qt)
    am2 = fq.fp8_amax(xd)
    q2, qt2, sc2 = fq.fp8_quantize_tensor(xd, 0, am2, want_q=want_q, want_qt=want_qt)
    assert fq.device_status() == 0
    assert_f32_bits_equal(f32(am), f32(am2), "amax")
    assert_f32_bits_equal(f32(sc), f32(sc2), "scale")
    if want_q:
        assert_bytes_equal(u8(q), u8(q2), "q")
    if want_qt:
        assert_bytes_equal(u8(qt), u8(qt2), "q_t")
    # against the oracle at every size, the cooperative one-launch case
    # (2048 x 2048 bf16, 8 MiB) and the 64 MiB activation included
    xo = to_oracle(x)
    assert_f32_bits_equal(f32(am), np.array([oracle.amax(xo)], np.float32), "oracle amax")
    rq, rqt, rs = oracle.quantize_tensor(xo, 0, want_q=want_q, want_qt=want_qt)
    assert_f32_bits_equal(f32(sc), np.array([rs], np.float32), "oracle scale")
    if want_q:
        assert_bytes_equal(u8(q), rq, "oracle q")
    if want_qt:
        assert_bytes_equal(u8(qt), rqt, "oracle q_t")


def test_quantize_tensor_current_special_values_and_repeats(fq):
    """NaN / Inf propagate as in the two-call path; repeated calls with the
    same outputs start from a zeroed amax."""
    x = workloads.normal((256, 512), 1.0, 45)
    for case in ("plain", "inf", "nan", "plain"):
        y = x.clone()
        if case == "inf":
            y[3, 7] = float("inf")
        if case == "nan":
            y[100, 200] = float("nan")
        yd = y.cuda()
        q, _, am, sc = fq.fp8_quantize_tensor_current(yd, 1)
        am2 = fq.fp8_amax(yd)
        q2, _, sc2 = fq.fp8_quantize_tensor(yd, 1, am2)
        assert fq.device_status() == 0
        assert_f32_bits_equal(f32(am), f32(am2), case + " amax")
        assert_f32_bits_equal(f32(sc), f32(sc2), case + " scale")
        assert_bytes_equal(u8(q), u8(q2), case + " q")


def test_quantize_tensor_current_empty(fq):
    x = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    q, _, am, sc = fq.fp8_quantize_tensor_current(x, 0)
    assert fq.device_status() == 0
    assert f32(am)[0] == 0.0
