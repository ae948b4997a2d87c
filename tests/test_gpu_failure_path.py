"""Failure detection without a GPU fault: a bounded barrier wait that runs
out is reported as FP8Q_ERR_TIMEOUT through the device error word, once, and
the CUDA context stays usable afterwards.  The wait runs out because nothing
ever arrives at the barrier (no trap, no bad address, no endless loop)."""
import time

import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fq():
    import scaled_quantize_fp8_warp_gb300 as fq
    from scaled_quantize_fp8_warp_gb300 import build_lib
    build_lib.build()
    fq.load_library()
    assert fq.device_supported()
    return fq


def test_bounded_wait_reports_timeout_and_context_survives(fq):
    assert fq.device_status() == 0
    t0 = time.time()
    fq.selftest_barrier_timeout()
    assert fq.device_status() == 5          # FP8Q_ERR_TIMEOUT, read and cleared
    waited = time.time() - t0
    assert 1.0 < waited < 30.0
    assert fq.device_status() == 0          # cleared
    # the context still runs the path
    x = torch.randn(256, 256, device="cuda", dtype=torch.bfloat16)
    q, qs, _, _ = fq.fp8_quantize_tile1x128(x, fq.E4M3)
    torch.cuda.synchronize()
    assert fq.device_status() == 0 and q.shape == (256, 256)
