"""Shared helpers for the GPU parity tests: tensor <-> oracle array plumbing."""
import numpy as np
import torch


def to_oracle(x: torch.Tensor) -> np.ndarray:
    """CPU copy in the oracle's input convention (fp32, or bf16 bit patterns)."""
    x = x.detach().cpu().contiguous()
    if x.dtype == torch.bfloat16:
        return x.view(torch.int16).numpy().view(np.uint16)
    assert x.dtype == torch.float32
    return x.numpy()


def u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def assert_bytes_equal(got: np.ndarray, ref: np.ndarray, what: str):
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    bad = np.nonzero(got != ref)
    if bad[0].size:
        idx = tuple(b[0] for b in bad)
        raise AssertionError(f"{what}: {bad[0].size} mismatching bytes, first at {idx}: "
                             f"got {got[idx]:#04x} want {ref[idx]:#04x}")


def assert_f32_bits_equal(got: np.ndarray, ref: np.ndarray, what: str):
    g = np.ascontiguousarray(got, dtype=np.float32).view(np.uint32)
    r = np.ascontiguousarray(ref, dtype=np.float32).view(np.uint32)
    gn = np.isnan(got)
    rn = np.isnan(ref)
    assert np.array_equal(gn, rn), f"{what}: NaN positions differ"
    ok = ~rn
    bad = np.nonzero(g[ok] != r[ok])[0]
    assert bad.size == 0, f"{what}: {bad.size} scales differ, e.g. {got[ok][bad[0]]} vs {ref[ok][bad[0]]}"
