"""The workspace-free autocast forward, fp8_linear_autocast_noalloc.

Callers that cannot call cudaMalloc (a plugin given only its tensors by a
host application that owns device memory, a serving loop that forbids
allocation after start-up) use this entry point; the library keeps the FP8
copies and scales in its own static 64 MiB device array.  The test calls it
through the C ABI, twice in a row on different inputs so that the second call
runs on scratch the first one left behind, and compares each result with the
existing entry point, fp8_linear_autocast, given a freshly allocated
workspace.  Both run the same kernels on the same data, so the results agree
bit for bit, which is stricter than the GEMM error bound of the other tests.

This file sorts last so that a run stopping at the first failure has run
every other test already.
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


@pytest.mark.parametrize("recipe_name",
                         ["RECIPE_TENSOR_CURRENT", "RECIPE_TENSOR_DELAYED", "RECIPE_BLOCK"])
def test_noalloc_matches_workspace_entry_point_twice(fq, recipe_name):
    recipe = getattr(fq, recipe_name)
    delayed = recipe == fq.RECIPE_TENSOR_DELAYED
    # The delayed recipe reads and updates amax histories: each entry point
    # gets its own pair, started from the same state, so after every call the
    # two pairs must still hold the same bits.
    hist0_x = [0.5 + 0.25 * i for i in range(fq.HISTORY_LEN)]
    hist0_w = [0.01 + 0.002 * i for i in range(fq.HISTORY_LEN)]
    ref_h = (fq.History(initial=hist0_x), fq.History(initial=hist0_w)) if delayed else (None, None)
    got_h = (fq.History(initial=hist0_x), fq.History(initial=hist0_w)) if delayed else (None, None)
    shapes = [(1024, 512, 1024, 10), (512, 768, 2048, 20)]   # (M, N, K, seed): two calls
    for M, N, K, seed in shapes:
        x = workloads.normal((M, K), 1.0, seed).cuda()
        w = workloads.normal((N, K), 0.02, seed + 1).cuda()
        ref = fq.fp8_linear_autocast(x, w, recipe=recipe, hist_x=ref_h[0], hist_w=ref_h[1])
        out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        got = fq.fp8_linear_autocast_noalloc(x, w, recipe=recipe, hist_x=got_h[0],
                                             hist_w=got_h[1], out=out)
        assert got.data_ptr() == out.data_ptr()
        assert fq.device_status() == 0
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16)), (recipe_name, M, N, K)
        if delayed:
            for r, g in zip(ref_h, got_h):
                assert torch.equal(r.buf.cpu(), g.buf.cpu()), (M, N, K)


def test_noalloc_rejects_sizes_over_the_limit(fq):
    M, N, K = 8192, 8192, 8192           # needs 128 MiB of FP8 copies
    need = fq.linear_workspace_size(fq.RECIPE_TENSOR_CURRENT, M, N, K)
    assert need > fq.NOALLOC_SCRATCH_BYTES
    x = torch.empty((1, 16), dtype=torch.bfloat16, device="cuda")   # never read
    rc = fq.lib().fp8_linear_autocast_noalloc(
        fq._ptr(x), fq._ptr(x), fq.DT_BF16, M, N, K, fq.RECIPE_TENSOR_CURRENT, None, None,
        fq._ptr(x), fq.DT_BF16, fq._stream(None))
    assert rc == 4   # FP8Q_ERR_WORKSPACE
