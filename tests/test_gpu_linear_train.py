"""fp8_linear_train and fp8_linear_train_host: one linear layer's Fprop,
Dgrad and Wgrad with x, w and grad_out quantized on the fly ("fp8_parity.py",
FP8Matmul forward and backward), against the CPU oracle for every recipe.

The oracle quantizes the same seeded inputs itself (E4M3 x and w, E5M2
grad_out; the transposed operands as the recipe defines them), computes each
GEMM in double, and every output must be within the GEMM error bound.  For
delayed scaling the three device histories must equal the oracle's after
each of two calls, bit for bit.  The host-buffer variant must equal the
device variant bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.gpu_helpers import assert_f32_bits_equal, f32, to_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fq():
    import scaled_quantize_fp8_warp_gb300 as fq
    from scaled_quantize_fp8_warp_gb300 import build_lib
    build_lib.build()
    fq.load_library()
    assert fq.device_supported()
    return fq


def check_bound(got, y_ref, absum, what):
    tol = oracle.gemm_bound(y_ref, absum, True)
    err = np.abs(got.astype(np.float64) - y_ref)
    bad = np.nonzero(~(err <= tol))
    assert bad[0].size == 0, f"{what}: {bad[0].size} outputs outside the bound"


def oracle_step(recipe, x, w, g, hist=None):
    """The three GEMMs with the oracle's own quantisation.  hist: list of three
    (ring, next) pairs for delayed scaling, updated in place."""
    xo, wo, go = to_oracle(x), to_oracle(w), to_oracle(g)
    O = oracle.GemmOperand
    if recipe == "current":
        qx, qxt, sx = oracle.quantize_tensor(xo, 0, want_qt=True)
        qw, qwt, sw = oracle.quantize_tensor(wo, 0, want_qt=True)
        qg, qgt, sg = oracle.quantize_tensor(go, 1, want_qt=True)
        ops = [(O.tensor(qx, 0, sx), O.tensor(qw, 0, sw)), (O.tensor(qg, 1, sg), O.tensor(qwt, 0, sw)),
               (O.tensor(qgt, 1, sg), O.tensor(qxt, 0, sx))]
    elif recipe == "delayed":
        out = []
        for i, (t, fmt) in enumerate(((xo, 0), (wo, 0), (go, 1))):
            ring, nxt = hist[i]
            q, qt, s, ring, nxt = oracle.quantize_delayed(t, fmt, ring, nxt, want_qt=True)
            hist[i] = (ring, nxt)
            out.append((q, qt, s))
        (qx, qxt, sx), (qw, qwt, sw), (qg, qgt, sg) = out
        ops = [(O.tensor(qx, 0, sx), O.tensor(qw, 0, sw)), (O.tensor(qg, 1, sg), O.tensor(qwt, 0, sw)),
               (O.tensor(qgt, 1, sg), O.tensor(qxt, 0, sx))]
    elif recipe == "block":
        qx, sx = oracle.quantize_tile_rows(xo, 0)
        qxt, sxt = oracle.quantize_tile_cols(xo, 0)
        qw, qwt, sw = oracle.quantize_block(wo, 0, want_qt=True)
        qg, sg = oracle.quantize_tile_rows(go, 1)
        qgt, sgt = oracle.quantize_tile_cols(go, 1)
        ops = [(O.tile(qx, 0, sx), O.block(qw, 0, sw)),
               (O.tile(qg, 1, sg), O.block(qwt, 0, sw, transposed=True)),   # sw read as [kb][rb]
               (O.tile(qgt, 1, sgt), O.tile(qxt, 0, sxt))]
    else:
        qx, sx = oracle.quantize_mx_rows(xo, 0)
        qxt, sxt = oracle.quantize_mx_cols(xo, 0)
        qw, sw = oracle.quantize_mx_rows(wo, 0)
        qwt, swt = oracle.quantize_mx_cols(wo, 0)
        qg, sg = oracle.quantize_mx_rows(go, 1)
        qgt, sgt = oracle.quantize_mx_cols(go, 1)
        ops = [(O.mx(qx, 0, sx), O.mx(qw, 0, sw)), (O.mx(qg, 1, sg), O.mx(qwt, 0, swt)),
               (O.mx(qgt, 1, sgt), O.mx(qxt, 0, sxt))]
    return [oracle.gemm_rows(a, b) for a, b in ops]


RECIPES = {"current": "RECIPE_TENSOR_CURRENT", "delayed": "RECIPE_TENSOR_DELAYED",
           "block": "RECIPE_BLOCK", "mxfp8": "RECIPE_MXFP8"}


@pytest.mark.parametrize("recipe", list(RECIPES))
@pytest.mark.parametrize("in_dtype", [torch.bfloat16, torch.float32])
def test_linear_train_vs_oracle(fq, recipe, in_dtype):
    M, N, K = 384, 272, 320
    code = getattr(fq, RECIPES[recipe])
    h0 = [[2.0 + 0.4 * i for i in range(16)], [0.02 + 0.008 * i for i in range(16)],
          [0.005 + 0.0003 * i for i in range(16)]]   # maxima 8.0, 0.14, 0.0095 cover the data
    hists = [fq.History(initial=h) for h in h0] if recipe == "delayed" else [None] * 3
    ohist = [(np.array(h, np.float32), 0) for h in h0]
    for call in range(2):
        x = workloads.normal((M, K), 1.0, 60 + call, dtype=in_dtype)
        w = workloads.normal((N, K), 0.02, 62 + call, dtype=in_dtype)
        g, _ = workloads.with_spikes((M, N), 1e-3, 40.0 if recipe != "delayed" else 0.0, 1e4,
                                     64 + call, dtype=in_dtype)
        y, dx, dw = fq.fp8_linear_train(x.cuda(), w.cuda(), g.cuda(), recipe=code,
                                        hist_x=hists[0], hist_w=hists[1], hist_g=hists[2])
        assert fq.device_status() == 0
        refs = oracle_step(recipe, x, w, g, ohist)
        for got, (yr, ab), nm in zip((y, dx, dw), refs, ("fprop", "dgrad", "wgrad")):
            check_bound(f32(got), yr, ab, f"{recipe} {in_dtype} call {call} {nm}")
        if recipe == "delayed":
            for h, (ring, nxt), nm in zip(hists, ohist, "xwg"):
                got_ring, got_next, _ = h.state()
                assert_f32_bits_equal(np.array(got_ring, np.float32), ring, f"hist_{nm}")
                assert got_next == nxt


@pytest.mark.parametrize("recipe", list(RECIPES))
def test_linear_train_host_equals_device(fq, recipe):
    """The host-buffer call copies in, runs the same kernels and copies out:
    its outputs equal the device call's bit for bit, twice in a row (the
    second call reuses the library's copy streams and events)."""
    M, N, K = 512, 384, 256
    code = getattr(fq, RECIPES[recipe])
    mk = lambda: [fq.History(initial=[8.0] * 16), fq.History(initial=[0.2] * 16),
                  fq.History(initial=[0.05] * 16)] if recipe == "delayed" else [None] * 3
    hd, hh = mk(), mk()
    ws = torch.empty(fq.linear_train_host_workspace_size(code, torch.bfloat16, torch.bfloat16,
                                                         M, N, K), dtype=torch.uint8,
                     device="cuda")
    st = torch.cuda.Stream()
    for call in range(2):
        x = workloads.normal((M, K), 1.0, 70 + call)
        w = workloads.normal((N, K), 0.02, 72 + call)
        g = workloads.normal((M, N), 1e-3, 74 + call)
        yd, dxd, dwd = fq.fp8_linear_train(x.cuda(), w.cuda(), g.cuda(), recipe=code,
                                           hist_x=hd[0], hist_w=hd[1], hist_g=hd[2])
        xh, wh, gh = x.pin_memory(), w.pin_memory(), g.pin_memory()
        yh = torch.empty((M, N), dtype=torch.bfloat16).pin_memory()
        dxh = torch.empty((M, K), dtype=torch.bfloat16).pin_memory()
        dwh = torch.empty((N, K), dtype=torch.bfloat16).pin_memory()
        fq.fp8_linear_train_host(xh, wh, gh, yh, dxh, dwh, ws, recipe=code, hist_x=hh[0],
                                 hist_w=hh[1], hist_g=hh[2], stream=st)
        st.synchronize()
        assert fq.device_status() == 0
        for a, b, nm in ((yd, yh, "y"), (dxd, dxh, "dx"), (dwd, dwh, "dw")):
            assert torch.equal(a.cpu().view(torch.int16), b.view(torch.int16)), (recipe, nm, call)
        if recipe == "delayed":
            for a, b in zip(hd, hh):
                assert torch.equal(a.buf.cpu(), b.buf.cpu())
