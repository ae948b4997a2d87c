"""FP8 training parity on a small MLP ("fp8_parity.py", smoke step 5), with
every FP8 matmul running through this library's kernels.

The page trains a 32 -> 64 -> 16 MLP for 300 AdamW steps (lr 3e-3, fp32
master weights and optimizer state) twice -- once with fp32 matmuls, once
with FP8 matmuls (E4M3 x and w forward, E5M2 output gradient backward, per-
tensor current scaling) -- and asserts that the final losses agree within
10%.  Here the FP8 run's Fprop, Dgrad and Wgrad are fp8_gemm_fprop /
fp8_gemm_dgrad / fp8_gemm_wgrad on operands from fp8_amax +
fp8_quantize_tensor (the transposed copies feed the backward GEMMs), with
fp32 outputs; the loss, ReLU and AdamW stay in torch fp32 as on the page.
Inputs are the page's shapes drawn from seeded generators (the page's exact
random stream is not reproduced).
"""
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fq():
    import scaled_quantize_fp8_warp_gb300 as fq
    from scaled_quantize_fp8_warp_gb300 import build_lib
    build_lib.build()
    fq.load_library()
    assert fq.device_supported()
    return fq


def make_fp8_matmul(fq):
    T = fq.GemmOperand.tensor

    class FP8Matmul(torch.autograd.Function):
        """y = x @ w.T with E4M3 operands forward, E5M2 grad_out backward."""

        @staticmethod
        def forward(ctx, x, w):
            x, w = x.contiguous(), w.contiguous()
            qx, qxt, sx = fq.fp8_quantize_tensor(x, fq.E4M3, fq.fp8_amax(x), want_qt=True)
            qw, qwt, sw = fq.fp8_quantize_tensor(w, fq.E4M3, fq.fp8_amax(w), want_qt=True)
            ctx.save_for_backward(qxt, sx, qwt, sw)
            return fq.fp8_gemm_fprop(T(qx, fq.E4M3, sx), T(qw, fq.E4M3, sw),
                                     out_dtype=torch.float32)

        @staticmethod
        def backward(ctx, g):
            qxt, sx, qwt, sw = ctx.saved_tensors
            g = g.contiguous()
            qg, qgt, sg = fq.fp8_quantize_tensor(g, fq.E5M2, fq.fp8_amax(g), want_qt=True)
            dx = fq.fp8_gemm_dgrad(T(qg, fq.E5M2, sg), T(qwt, fq.E4M3, sw),
                                   out_dtype=torch.float32)
            dw = fq.fp8_gemm_wgrad(T(qgt, fq.E5M2, sg), T(qxt, fq.E4M3, sx),
                                   out_dtype=torch.float32)
            return dx, dw

    return FP8Matmul.apply


def train(mm, X, Y, steps=300):
    g = torch.Generator()
    g.manual_seed(1)
    W1 = (torch.randn(64, 32, generator=g) / 6).cuda().requires_grad_()
    W2 = (torch.randn(16, 64, generator=g) / 8).cuda().requires_grad_()
    opt = torch.optim.AdamW([W1, W2], lr=3e-3)
    first = None
    for _ in range(steps):
        loss = ((mm(torch.relu(mm(X, W1)), W2) - Y) ** 2).mean()
        opt.zero_grad()
        loss.backward()
        opt.step()
        if first is None:
            first = loss.item()
    return first, loss.item()


def test_fp8_mlp_training_matches_fp32(fq):
    X = workloads.normal((512, 32), 1.0, 50, dtype=torch.float32).cuda()
    Wt = workloads.normal((16, 32), 1.0, 51, dtype=torch.float32).cuda() / 6
    Y = torch.tanh(X @ Wt.T)
    f32_first, l32 = train(lambda a, w: a @ w.T, X, Y)
    f8_first, l8 = train(make_fp8_matmul(fq), X, Y)
    assert fq.device_status() == 0
    assert l32 < 0.5 * f32_first and l8 < 0.5 * f8_first, "training did not make progress"
    gap = abs(l8 - l32) / l32
    assert gap < 0.10, f"final loss fp32 {l32:.5f} vs FP8 {l8:.5f} (gap {100 * gap:.1f}%)"
