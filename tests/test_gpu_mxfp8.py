"""GPU parity of the MXFP8 path (OCP MX v1.0: 1x32 blocks, E8M0 scales)
against the CPU oracle.

* fp8_quantize_mxfp8: element bytes and scale codes bit-exact against
  oracle.quantize_mx_rows / quantize_mx_cols, both orientations, bf16 and
  fp32 inputs, E4M3 and E5M2, ragged shapes, every bf16 value, zero / NaN /
  Inf blocks, negative zeros and fp32 subnormals.  The library's scales come
  in its 512-byte atom layout (include/fp8q.h); atoms_to_plain() below reads
  them back into the oracle's [rows, ceil(K/32)] layout by that formula.
* the MXFP8 GEMM (hardware block scaling): within the error bound of the
  oracle's double-accumulated GEMM on random codes and scales (operands built
  on the host, so the GEMM is checked on its own), exact where every partial
  sum is exact, and on sampled 64 x 64 output blocks of the transformer
  layer's full-size Fprop / Dgrad / Wgrad shapes, where the oracle quantises
  the same rows of the seeded inputs itself.
* fp8_linear_autocast with the MXFP8 recipe against the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.gpu_helpers import assert_bytes_equal, f32, to_oracle, u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fq():
    import scaled_quantize_fp8_warp_gb300 as fq
    from scaled_quantize_fp8_warp_gb300 import build_lib
    build_lib.build()
    fq.load_library()
    assert fq.device_supported()
    return fq


def cdiv(a, b):
    return (a + b - 1) // b


def atoms_to_plain(atoms, R: int, K: int) -> np.ndarray:
    """E8M0 atoms of an [R, K] operand -> [R, ceil(K/32)] codes.  Atom (rb, kb)
    starts at (rb * ceil(K/128) + kb) * 512; row 128 rb + r, block 4 kb + j sits
    at byte (r % 32) * 16 + (r // 32) * 4 + j.  Padding (rows >= R, blocks past
    K) must be code 0."""
    a = np.asarray(atoms, dtype=np.uint8)
    nrb, nkb = cdiv(R, 128), cdiv(K, 128)
    assert a.size == nrb * nkb * 512
    t = a.reshape(nrb, nkb, 32, 4, 4)            # rb, kb, r%32, r//32, j
    full = t.transpose(0, 3, 2, 1, 4).reshape(nrb * 128, nkb * 4)
    nb = cdiv(K, 32)
    assert not full[R:].any() and not full[:, nb:].any(), "padding scales are not 0"
    return np.ascontiguousarray(full[:R, :nb])


def plain_to_atoms(plain: np.ndarray, R: int, K: int) -> np.ndarray:
    nrb, nkb = cdiv(R, 128), cdiv(K, 128)
    full = np.zeros((nrb * 128, nkb * 4), np.uint8)
    full[:R, :plain.shape[1]] = plain
    t = full.reshape(nrb, 4, 32, nkb, 4).transpose(0, 3, 2, 1, 4)
    return np.ascontiguousarray(t.reshape(-1))


def test_atom_helpers_round_trip():
    rng = np.random.default_rng(0)
    for R, K in [(1, 32), (130, 80), (300, 512)]:
        p = rng.integers(0, 255, (R, cdiv(K, 32)), dtype=np.uint8)
        assert np.array_equal(atoms_to_plain(plain_to_atoms(p, R, K), R, K), p)


def check_quantize(fq, x: torch.Tensor, fmt: int, what: str, rows=True, cols=True):
    R, C = x.shape
    q, qs, qt, qts = fq.fp8_quantize_mxfp8(x.cuda(), fmt, rows=rows, cols=cols)
    assert fq.device_status() == 0
    xo = to_oracle(x)
    if rows:
        rq, rs = oracle.quantize_mx_rows(xo, fmt)
        assert_bytes_equal(atoms_to_plain(u8(qs), R, C), rs, what + " row scales")
        assert_bytes_equal(u8(q), rq, what + " q")
    if cols:
        rqt, rst = oracle.quantize_mx_cols(xo, fmt)
        assert_bytes_equal(atoms_to_plain(u8(qts), C, R), rst, what + " column scales")
        assert_bytes_equal(u8(qt), rqt, what + " q_t")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("shape", [(16, 32), (144, 96), (272, 208), (256, 384), (1040, 2064)])
def test_quantize_matches_oracle(fq, dtype, fmt, shape):
    R, C = shape
    g = torch.Generator().manual_seed(R * 7 + C + fmt)
    x = torch.randn(shape, generator=g) * torch.pow(
        2.0, torch.randint(-12, 12, (R, 1), generator=g).float())
    x[R // 3] *= 1e4                    # an outlier row
    check_quantize(fq, x.to(dtype), fmt, f"{dtype} fmt{fmt} {shape}")


@pytest.mark.parametrize("fmt", [0, 1])
def test_quantize_every_bf16_value(fq, fmt):
    """All 65536 bf16 patterns, shuffled into 32-element blocks of mixed
    magnitude (blocks holding a NaN or an Inf become NaN blocks)."""
    perm = np.random.default_rng(5).permutation(65536).astype(np.uint16)
    x = torch.from_numpy(perm.view(np.int16).copy()).view(torch.bfloat16).reshape(512, 128)
    check_quantize(fq, x, fmt, f"all bf16 fmt{fmt}")
    # the same values each paired with a finite block maximum, so that every
    # pattern is also cast under a range of ordinary scales
    bits = np.arange(65536, dtype=np.uint32)
    finite = bits[((bits >> 7) & 0xFF) != 0xFF].astype(np.uint16)
    vals = finite[: (finite.size // 31) * 31].reshape(-1, 31)
    exps = np.random.default_rng(6).integers(-130, 120, vals.shape[0])
    maxima = np.ldexp(np.float32(1.0), exps).astype(np.float32)   # powers of two: exact in bf16
    mx = (maxima.view(np.uint32) >> 16).astype(np.uint16)
    blocks = np.concatenate([mx[:, None], vals], axis=1)
    rows = blocks.shape[0] - blocks.shape[0] % 16
    xb = torch.from_numpy(blocks[:rows].view(np.int16).copy()).view(torch.bfloat16)
    check_quantize(fq, xb, fmt, f"bf16 under varied maxima fmt{fmt}")


@pytest.mark.parametrize("fmt", [0, 1])
def test_quantize_special_blocks(fq, fmt):
    x = torch.randn(64, 256) * 3.0
    x[0, :32] = 0.0                         # all-zero block
    x[1, :32] = -0.0                        # negative zeros
    x[2, 40] = float("nan")                 # NaN poisons its block only
    x[3, 100] = float("inf")
    x[4, 200] = -float("inf")
    x[5, :32] = torch.tensor(1e-40)         # fp32 subnormals (max subnormal -> code 0)
    x[6, 32:64] = 3.0e38                    # near the top of fp32
    x[7, 64:96] = torch.linspace(-1.999, 1.999, 32)   # maxima just below a power of two
    x[8, 96:128] = 448.0 * 2.0 ** -20       # exactly fmax * 2^k
    x[9] = 2.0 ** torch.arange(-120, 136, dtype=torch.float32).clamp(max=127)
    x[:, 250] = -1e-30                      # tiny negatives round to -0
    check_quantize(fq, x, fmt, f"special f32 fmt{fmt}")
    check_quantize(fq, x.to(torch.bfloat16), fmt, f"special bf16 fmt{fmt}")


def test_quantize_single_orientation(fq):
    x = workloads.normal((272, 160), 1.0, 41)
    check_quantize(fq, x, 0, "rows only", rows=True, cols=False)
    check_quantize(fq, x, 1, "cols only", rows=False, cols=True)


# ------------------------------------------------------------------ GEMM

def _rand_codes(rng, shape, fmt):
    table = oracle.decode_table(fmt)
    finite = np.nonzero(np.isfinite(table))[0].astype(np.uint8)
    return rng.choice(finite, size=shape)


def check_bound(got, y_ref, absum, out_bf16, what):
    tol = oracle.gemm_bound(y_ref, absum, out_bf16)
    err = np.abs(got.astype(np.float64) - y_ref)
    bad = np.nonzero(~(err <= tol))
    assert bad[0].size == 0, (f"{what}: {bad[0].size} outputs outside the bound; first at "
                              f"{tuple(b[0] for b in bad)}: got {got[tuple(b[0] for b in bad)]}"
                              f", ref {y_ref[tuple(b[0] for b in bad)]}")


def gemm_host_operands(fq, A, sa, B, sb, fa, fb):
    M, K = A.shape
    N = B.shape[0]
    opA = fq.GemmOperand.mx(torch.from_numpy(A).cuda(), fa,
                            torch.from_numpy(plain_to_atoms(sa, M, K)).cuda())
    opB = fq.GemmOperand.mx(torch.from_numpy(B).cuda(), fb,
                            torch.from_numpy(plain_to_atoms(sb, N, K)).cuda())
    return opA, opB


@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (300, 384, 224), (257, 272, 80),
                                   (64, 64, 32), (512, 512, 1024)])
@pytest.mark.parametrize("fa,fb", [(0, 0), (1, 0), (0, 1)])
@pytest.mark.parametrize("out", [torch.float32, torch.bfloat16])
def test_gemm_random_codes_and_scales(fq, M, N, K, fa, fb, out):
    rng = np.random.default_rng(M * 3 + N + K + fa * 7 + fb)
    A = _rand_codes(rng, (M, K), fa)
    B = _rand_codes(rng, (N, K), fb)
    sa = rng.integers(110, 140, (M, cdiv(K, 32))).astype(np.uint8)
    sb = rng.integers(110, 140, (N, cdiv(K, 32))).astype(np.uint8)
    opA, opB = gemm_host_operands(fq, A, sa, B, sb, fa, fb)
    y = fq.fp8_gemm(opA, opB, out_dtype=out)
    assert fq.device_status() == 0
    ref, ab = oracle.gemm_rows(oracle.GemmOperand.mx(A, fa, sa), oracle.GemmOperand.mx(B, fb, sb))
    check_bound(f32(y), ref, ab, out == torch.bfloat16, f"mx gemm {M}x{N}x{K} {fa}{fb}")


def test_gemm_exact_when_sums_are_exact(fq):
    """Small-integer codes with power-of-two scales 2^0..2^3: every product and
    partial sum is an integer below 2^24, so the result is exact."""
    rng = np.random.default_rng(11)
    M, N, K = 256, 256, 256
    ints = np.arange(-4, 5, dtype=np.float32)
    A = oracle.encode(rng.choice(ints, size=(M, K)), 0)
    B = oracle.encode(rng.choice(ints, size=(N, K)), 0)
    sa = rng.integers(127, 129, (M, K // 32)).astype(np.uint8)
    sb = rng.integers(127, 129, (N, K // 32)).astype(np.uint8)
    opA, opB = gemm_host_operands(fq, A, sa, B, sb, 0, 0)
    y = fq.fp8_gemm(opA, opB, out_dtype=torch.float32)
    assert fq.device_status() == 0
    ref, _ = oracle.gemm_rows(oracle.GemmOperand.mx(A, 0, sa), oracle.GemmOperand.mx(B, 0, sb))
    assert np.array_equal(f32(y).astype(np.float64), ref)


@pytest.mark.parametrize("M,N,K", [(128, 512, 512), (384, 768, 256), (256, 272, 128),
                                   (128, 128, 256)])
def test_gemm_scale_selects_each_block(fq, M, N, K):
    """A's and B's codes all 1.0, a different scale per row and 32-wide block:
    C[m, n] = 32 * sum_j 2^(sa[m, j] - 127) * 2^(sb[n, j] - 127), a closed
    form that pins which scale byte (and which tensor-memory column and lane)
    every K step uses.  Codes stay within 125..129, so every term is a
    multiple of 2^-3 and the sums are exact in fp32: the result must equal the
    closed form bit for bit.  (With terms spread over 2^25 the tensor cores'
    accumulator, which drops addends below the running sum's last place, can
    land 2.3e-6 low on such an all-positive sum.)  The shapes cover the
    one-SM kernel (N <= 128) and the CTA-pair kernel with an odd count of
    128-row tiles and a ragged last column tile."""
    A = np.full((M, K), 0x38, np.uint8)
    B = np.full((N, K), 0x38, np.uint8)
    rng = np.random.default_rng(12)
    sa = rng.integers(125, 130, (M, K // 32)).astype(np.uint8)
    sb = rng.integers(125, 130, (N, K // 32)).astype(np.uint8)
    opA, opB = gemm_host_operands(fq, A, sa, B, sb, 0, 0)
    y = f32(fq.fp8_gemm(opA, opB, out_dtype=torch.float32)).astype(np.float64)
    ea = np.ldexp(1.0, sa.astype(np.int64) - 127)
    eb = np.ldexp(1.0, sb.astype(np.int64) - 127)
    closed = 32.0 * ea @ eb.T
    assert np.array_equal(y, closed)


@pytest.mark.parametrize("layer", [1, 3])   # attention out (4096x4096), MLP down (K = 16384)
def test_layer_roles_sampled(fq, layer):
    """Full-size Fprop / Dgrad / Wgrad of a transformer linear with MXFP8 on
    x, w and grad_out (E4M3 / E4M3 / E5M2), as the layer runs them, checked
    on a 64 x 64 block of each output: the oracle quantises those 64 rows of
    each operand from the seeded inputs itself."""
    shape = workloads.LAYER[layer]
    x, w, g = workloads.layer_inputs(shape, layer)
    M, K, N = x.shape[0], shape.K, shape.N
    xd, wd, gd = x.cuda(), w.cuda(), g.cuda()
    qx, sx, qxt, sxt = fq.fp8_quantize_mxfp8(xd, 0, rows=True, cols=True)
    qw, sw, qwt, swt = fq.fp8_quantize_mxfp8(wd, 0, rows=True, cols=True)
    qg, sg, qgt, sgt = fq.fp8_quantize_mxfp8(gd, 1, rows=True, cols=True)
    Op = fq.GemmOperand.mx
    y = fq.fp8_gemm_fprop(Op(qx, 0, sx), Op(qw, 0, sw))
    dx = fq.fp8_gemm_dgrad(Op(qg, 1, sg), Op(qwt, 0, swt))
    dw = fq.fp8_gemm_wgrad(Op(qgt, 1, sgt), Op(qxt, 0, sxt))
    assert fq.device_status() == 0
    rng = np.random.default_rng(layer)
    xo, wo, go = to_oracle(x), to_oracle(w), to_oracle(g)

    def rows_of(src, idx, fmt):        # oracle: 1x32 blocks of the chosen rows
        return oracle.quantize_mx_rows(np.ascontiguousarray(src[idx]), fmt)

    def cols_of(src, idx, fmt):        # oracle: 32x1 blocks of the chosen columns
        return oracle.quantize_mx_cols(np.ascontiguousarray(src[:, idx]), fmt)

    cases = [
        ("fprop", y, lambda i: rows_of(xo, i, 0), lambda j: rows_of(wo, j, 0), M, N, 0, 0),
        ("dgrad", dx, lambda i: rows_of(go, i, 1), lambda j: cols_of(wo, j, 0), M, K, 1, 0),
        ("wgrad", dw, lambda i: cols_of(go, i, 1), lambda j: cols_of(xo, j, 0), N, K, 1, 0),
    ]
    for name, out, a_rows, b_rows, R, C, fa, fb in cases:
        mi = np.sort(rng.choice(R, 64, replace=False))
        ni = np.sort(rng.choice(C, 64, replace=False))
        qa, sa = a_rows(mi)
        qb, sb = b_rows(ni)
        ref, ab = oracle.gemm_rows(oracle.GemmOperand.mx(qa, fa, sa),
                                   oracle.GemmOperand.mx(qb, fb, sb))
        got = f32(out[torch.from_numpy(mi).cuda()][:, torch.from_numpy(ni).cuda()])
        check_bound(got, ref, ab, True, f"layer {layer} {name}")
    # the GPU's quantised bytes of the sampled rows agree with the oracle too
    qa, sa = rows_of(xo, np.arange(256), 0)
    assert_bytes_equal(u8(qx[:256]), qa, "x rows")
    assert_bytes_equal(atoms_to_plain(u8(sx), M, K)[:256], sa, "x row scales")


def test_linear_autocast_mxfp8(fq):
    M, N, K = 640, 384, 1024
    x = workloads.normal((M, K), 1.0, 51)
    w = workloads.normal((N, K), 0.02, 52)
    y = fq.fp8_linear_autocast(x.cuda(), w.cuda(), recipe=fq.RECIPE_MXFP8)
    assert fq.device_status() == 0
    qx, sx = oracle.quantize_mx_rows(to_oracle(x), 0)
    qw, sw = oracle.quantize_mx_rows(to_oracle(w), 0)
    ref, ab = oracle.gemm_rows(oracle.GemmOperand.mx(qx, 0, sx), oracle.GemmOperand.mx(qw, 0, sw))
    check_bound(f32(y), ref, ab, True, "autocast mxfp8")


def test_gemm_amax_mx(fq):
    rng = np.random.default_rng(13)
    M, N, K = 384, 512, 256
    A = _rand_codes(rng, (M, K), 0)
    B = _rand_codes(rng, (N, K), 0)
    sa = rng.integers(115, 130, (M, K // 32)).astype(np.uint8)
    sb = rng.integers(115, 130, (N, K // 32)).astype(np.uint8)
    opA, opB = gemm_host_operands(fq, A, sa, B, sb, 0, 0)
    y, am = fq.fp8_gemm_amax(opA, opB)
    assert fq.device_status() == 0
    assert np.float32(am.item()) == oracle.amax(to_oracle(y))
