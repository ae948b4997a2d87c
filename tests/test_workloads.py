"""The seeded input recipes: shapes, distributions, outlier and spike
placement, and the layer's GEMM list, checked against the numbers the
workload is defined by (the fp8_parity page's sizes; the blog repost's
15872-token layer with hidden 4096 and FFN 16384; one 40.0 spike per 1e6
gradient entries; 1% outlier rows x 1e4)."""
import torch

import workloads


def test_layer_gemms_and_flops():
    probs = workloads.gemm_problems()
    assert len(probs) == 12
    shapes = {(n, r): (m, nn, k) for n, r, m, nn, k in probs}
    assert shapes[("qkv", "fprop")] == (15872, 12288, 4096)
    assert shapes[("qkv", "dgrad")] == (15872, 4096, 12288)
    assert shapes[("qkv", "wgrad")] == (12288, 4096, 15872)
    assert shapes[("mlp_down", "fprop")] == (15872, 4096, 16384)
    assert shapes[("mlp_down", "wgrad")] == (4096, 16384, 15872)
    # 6.391e12 FLOP per pass of the four linears, 1.917e13 per 12-GEMM layer
    assert abs(workloads.gemm_flops() - 1.917e13) / 1.917e13 < 1e-3
    fprop = sum(2 * m * n * k for _, r, m, n, k in probs if r == "fprop")
    assert abs(fprop - 6.391e12) / 6.391e12 < 1e-3


def test_spike_counts_per_layer():
    """floor(numel / 1e6) spikes in each linear's grad_out [M, N]."""
    counts = {s.name: (workloads.TOKENS * s.N) // 10**6 for s in workloads.LAYER}
    assert counts == {"qkv": 195, "attn_out": 65, "mlp_up": 260, "mlp_down": 65}


def test_with_spikes_places_distinct_exact_spikes():
    t, pos = workloads.with_spikes((300, 700), 1e-3, 40.0, 1e3, 7)
    assert t.dtype == torch.bfloat16 and t.shape == (300, 700)
    assert pos.numel() == 210 and torch.unique(pos).numel() == 210
    flat = t.view(-1).float()
    assert torch.all(flat[pos] == 40.0)
    rest = torch.ones(flat.numel(), dtype=torch.bool)
    rest[pos] = False
    assert flat[rest].abs().max() < 0.01          # N(0, 1e-3) stays far below the spike
    assert 0.9e-3 < flat[rest].std() < 1.1e-3
    t2, pos2 = workloads.with_spikes((300, 700), 1e-3, 40.0, 1e3, 7)
    assert torch.equal(t.view(torch.int16), t2.view(torch.int16)) and torch.equal(pos, pos2)


def test_spike_positions_cover_the_range():
    g = torch.Generator()
    g.manual_seed(3)
    pos = workloads.spike_positions(1000, 999, g)
    assert torch.unique(pos).numel() == 999 and int(pos.min()) >= 0 and int(pos.max()) < 1000
    assert workloads.spike_positions(10, 0, g).numel() == 0


def test_quantize_activation_recipe():
    x, rows = workloads.quantize_activation()
    assert x.shape == (8192, 4096) and x.dtype == torch.bfloat16
    assert rows.numel() == 82 and torch.unique(rows).numel() == 82     # round(0.01 * 8192)
    xf = x.float()
    mask = torch.zeros(8192, dtype=torch.bool)
    mask[rows] = True
    assert 90 < xf[mask].std() < 110            # N(0, 0.01) x 1e4
    assert 0.0095 < xf[~mask].std() < 0.0105
    x2, rows2 = workloads.quantize_activation()
    assert torch.equal(x.view(torch.int16), x2.view(torch.int16)) and torch.equal(rows, rows2)


def test_tiny_linear_recipe():
    x, w, g = workloads.tiny_linear()
    assert (x.shape, w.shape, g.shape) == ((512, 32), (64, 32), (512, 64))
    assert x.dtype == w.dtype == g.dtype == torch.float32
    assert 0.9 < x.std() < 1.1
    assert 0.9 / 6 < w.std() < 1.1 / 6
    assert 0.9e-2 < g.std() < 1.1e-2
    x2, _, _ = workloads.tiny_linear(1)
    assert not torch.equal(x, x2)


def test_layer_inputs_small_m():
    """The layer recipe at a small token count (the full one is too large for
    a CPU test): shapes, dtypes, spreads and the spike count."""
    s = workloads.LAYER[0]
    x, w, g = workloads.layer_inputs(s, 0, M=256)
    assert x.shape == (256, 4096) and w.shape == (12288, 4096) and g.shape == (256, 12288)
    assert x.dtype == w.dtype == g.dtype == torch.bfloat16
    assert 0.95 < x.float().std() < 1.05 and 0.019 < w.float().std() < 0.021
    assert int((g.float() == 40.0).sum()) == (256 * 12288) // 10**6
