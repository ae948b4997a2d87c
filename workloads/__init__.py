"""Seeded synthetic inputs shared by the oracle side and the CUDA side.

This module holds the input recipe only -- distributions, shapes, seeds and
outlier placement -- and none of the quantisation or GEMM arithmetic.  Every
tensor is drawn on the CPU with ``torch.Generator().manual_seed(seed)`` in
fp32, shaped as below, then cast once to its storage type, so both sides see
identical bytes.

Workloads (names used by the tests and the benchmark):

* ``tiny_linear`` -- the MLP sizes of the fp8_parity page's smoke step 5:
  x 512x32 ~ N(0,1), w 64x32 ~ N(0,1)/6, grad_out 512x64 ~ N(0,1)*1e-2, fp32.
* ``quantize_8192x4096`` -- an activation 8192x4096 ~ N(0,1)*0.01 with 1% of
  its rows (82, uniformly without replacement) multiplied by 1e4 in fp32,
  then cast to bf16 (the outlier-row construction of smoke step 4, at scale).
* ``layer`` -- the transformer layer of the low-precision-training blog
  repost: M = 31 x 512 = 15872 tokens, hidden 4096, FFN 16384, four linear
  layers (QKV, attention out, MLP up, MLP down).  Per layer: x [M, K] bf16
  ~ N(0,1); w [N, K] bf16 ~ N(0, 0.02); grad_out [M, N] bf16 ~ N(0, 1e-3)
  with floor(numel / 1e6) entries (uniform, without replacement) set to 40.0.
  Delayed-scaling history: 16 amax values of spike-free draws of the same
  grad_out distribution (seeds 4000 + i).

The second number in N(mu, sigma) is a standard deviation: the draw is
``randn * sigma``.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

TOKENS = 31 * 512          # 15872
HIDDEN = 4096
FFN = 16384


@dataclass(frozen=True)
class LinearShape:
    name: str
    K: int   # input features (contraction of Fprop)
    N: int   # output features


LAYER = (
    LinearShape("qkv", HIDDEN, 3 * HIDDEN),
    LinearShape("attn_out", HIDDEN, HIDDEN),
    LinearShape("mlp_up", HIDDEN, FFN),
    LinearShape("mlp_down", FFN, HIDDEN),
)


def gemm_problems(M: int = TOKENS):
    """The 12 GEMMs of one layer as (name, role, out_rows, out_cols, contraction).

    Fprop  y  = x w^T : [M, N] over K
    Dgrad  dx = g w   : [M, K] over N
    Wgrad  dw = g^T x : [N, K] over M
    """
    out = []
    for s in LAYER:
        out.append((s.name, "fprop", M, s.N, s.K))
        out.append((s.name, "dgrad", M, s.K, s.N))
        out.append((s.name, "wgrad", s.N, s.K, M))
    return out


def gemm_flops(M: int = TOKENS) -> float:
    return float(sum(2 * m * n * k for _, _, m, n, k in gemm_problems(M)))


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def normal(shape, std: float, seed: int, dtype=torch.bfloat16) -> torch.Tensor:
    """randn(shape) * std drawn in fp32, cast once to dtype."""
    g = _gen(seed)
    t = torch.randn(*shape, generator=g, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def with_outlier_rows(shape, std: float, frac: float, factor: float, seed: int,
                      dtype=torch.bfloat16):
    """randn * std with round(frac * rows) rows (seeded permutation) multiplied
    by ``factor`` in fp32 before the single cast.  Returns (tensor, rows)."""
    g = _gen(seed)
    t = torch.randn(*shape, generator=g, dtype=torch.float32)
    t.mul_(std)
    n_out = int(round(frac * shape[0]))
    rows = torch.randperm(shape[0], generator=g)[:n_out]
    t[rows] *= factor
    return t.to(dtype), torch.sort(rows).values


def spike_positions(numel: int, count: int, g: torch.Generator) -> torch.Tensor:
    """``count`` distinct flat positions in [0, numel), uniform."""
    if count == 0:
        return torch.empty(0, dtype=torch.int64)
    chosen = torch.empty(0, dtype=torch.int64)
    while chosen.numel() < count:
        extra = torch.randint(numel, (2 * (count - chosen.numel()),), generator=g)
        merged = torch.cat([chosen, extra])
        # keep first occurrences in draw order
        uniq, inv = torch.unique(merged, return_inverse=True)
        first = torch.full((uniq.numel(),), merged.numel(), dtype=torch.int64)
        first.scatter_reduce_(0, inv, torch.arange(merged.numel()), reduce="amin")
        chosen = merged[torch.sort(first).values]
    return chosen[:count]


def with_spikes(shape, std: float, spike: float, per: float, seed: int,
                dtype=torch.bfloat16):
    """randn * std with floor(numel / per) entries set to ``spike``.
    Returns (tensor, flat spike positions)."""
    g = _gen(seed)
    t = torch.randn(*shape, generator=g, dtype=torch.float32)
    t.mul_(std)
    numel = t.numel()
    pos = spike_positions(numel, int(numel // per), g)
    t.view(-1)[pos] = spike
    return t.to(dtype), pos


# ------------------------------------------------------------ named workloads

def tiny_linear(seed: int = 0):
    """x 512x32, w 64x32, grad_out 512x64, fp32 (seed 0)."""
    g = _gen(seed)
    x = torch.randn(512, 32, generator=g)
    w = torch.randn(64, 32, generator=g) / 6
    gout = torch.randn(512, 64, generator=g) * 1e-2
    return x, w, gout


def quantize_activation(seed: int = 1, rows: int = 8192, cols: int = 4096):
    """8192x4096 bf16 ~ N(0,1)*0.01 with 1% of rows x 1e4 (seed 1)."""
    return with_outlier_rows((rows, cols), 0.01, 0.01, 1e4, seed)


def layer_inputs(shape: LinearShape, index: int, M: int = TOKENS):
    """(x, w, grad_out) for one linear layer of the transformer workload."""
    x = normal((M, shape.K), 1.0, 3000 + index)
    w = normal((shape.N, shape.K), 0.02, 3100 + index)
    g, _ = with_spikes((M, shape.N), 1e-3, 40.0, 1e6, 3200 + index)
    return x, w, g


def history_draws(shape, count: int = 16, std: float = 1e-3, max_numel: int = 1 << 22):
    """Spike-free draws for the delayed-scaling history (seeds 4000 + i), each
    with the distribution of grad_out and min(numel, max_numel) elements."""
    numel = 1
    for d in shape:
        numel *= d
    n = min(numel, max_numel)
    return [normal((n,), std, 4000 + i) for i in range(count)]
