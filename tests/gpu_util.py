"""Helpers shared by the GPU tests: numpy bf16 bits <-> torch tensors, and the
parity bar against the fp64 oracle (max-abs 1e-2 beyond the output's own bf16
rounding, mean-abs 1e-3)."""
import numpy as np
import torch

from synthetic import bf16_to_f32

MAX_ABS = 1e-2
MEAN_ABS = 1e-3
BF16_HALF_ULP_REL = 2.0 ** -8  # largest relative rounding error of a bf16 value


def dev():
    return torch.device("cuda:0")


def bf(x: np.ndarray) -> torch.Tensor:
    """uint16 bf16 bits (numpy) -> bf16 CUDA tensor with the same bits."""
    return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).to(dev())


def f32(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(dev())


def i32(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.int32)).to(dev())


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 CUDA tensor -> uint16 bits (numpy)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def val(t: torch.Tensor) -> np.ndarray:
    return bf16_to_f32(bits(t)).astype(np.float64)


def assert_parity(got: np.ndarray, ref: np.ndarray, what: str = "") -> None:
    """max-abs 1e-2 on the error beyond the output's own bf16 rounding, mean-abs 1e-3 raw.

    A bf16 output can be no closer to the exact value than half an ulp, which is up to
    2**-8 * |o| (0.0156 for |o| in [4, 8)), so the max bar is applied to
    |got - ref| - 2**-8 * |ref|; the mean bar is applied to |got - ref| itself."""
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    if got.size == 0:
        return
    d = np.abs(got - ref)
    excess = float((d - BF16_HALF_ULP_REL * np.abs(ref)).max())
    mx, mn = float(d.max()), float(d.mean())
    assert excess <= MAX_ABS and mn <= MEAN_ABS, (
        f"{what}: max|err| {mx:.3e} (beyond bf16 output rounding {excess:.3e}) mean|err| {mn:.3e}")


class ParityAccumulator:
    """assert_parity over an output compared in chunks: the max bar on the largest excess over
    all chunks, the mean bar on the mean over every element."""

    def __init__(self, what: str = ""):
        self.what, self.excess, self.mx, self.total, self.n = what, -np.inf, 0.0, 0.0, 0

    def add(self, got: np.ndarray, ref: np.ndarray) -> None:
        assert got.shape == ref.shape, (got.shape, ref.shape)
        assert np.isfinite(got).all(), f"{self.what}: non-finite output"
        if got.size == 0:
            return
        d = np.abs(got - ref)
        self.excess = max(self.excess, float((d - BF16_HALF_ULP_REL * np.abs(ref)).max()))
        self.mx = max(self.mx, float(d.max()))
        self.total += float(d.sum())
        self.n += d.size

    def check(self) -> None:
        assert self.n > 0, f"{self.what}: nothing compared"
        mn = self.total / self.n
        assert self.excess <= MAX_ABS and mn <= MEAN_ABS, (
            f"{self.what}: max|err| {self.mx:.3e} (beyond bf16 output rounding {self.excess:.3e}) "
            f"mean|err| {mn:.3e} over {self.n} values")
