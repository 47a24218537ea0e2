"""Shared helpers for the GPU parity tests: seeded cases, the oracle reference,
and the tolerance from the acceptance rule

    |y_gpu - y_ref| <= 1e-3 * max|y_ref| + 1e-3   (elementwise, max over the call's output)

y_ref is the oracle's binary64 result.  The bound covers fp16 output rounding
(at most 2^-11 |y|, about half of the relative term) and fp32 accumulation.
"""
import numpy as np
import torch

import oracle
import synthetic_inputs as si

RTOL = 1e-3
ATOL = 1e-3


# bf16 outputs: one rounding to 8 significant bits costs up to 2^-9 |y|, more
# than the fp16 rule's relative term allows; the bound doubles that rounding
RTOL_BF16 = 2.0 ** -8
# bf16 outputs of the tcgen05 rungs, which round each restored weight once to
# bf16 ((q - z) * s to 8 significant bits, as a bf16 dequantisation does):
# the output's rounding (up to 2^-8 |y| just above a power of two) plus the
# weights' roundings (up to 2^-9 each, summed with the products)
RTOL_BF16_TC = 2.0 ** -7


def tolerance(y_ref: np.ndarray, rtol: float = RTOL) -> float:
    m = float(np.max(np.abs(y_ref))) if y_ref.size else 0.0
    return rtol * m + ATOL


def assert_close(y_gpu: torch.Tensor, y_ref: np.ndarray, what: str = "", rtol: float = None):
    if rtol is None:
        rtol = RTOL_BF16 if y_gpu.dtype == torch.bfloat16 else RTOL
    y = y_gpu.detach().float().cpu().numpy().astype(np.float64)
    assert y.shape == y_ref.shape, (y.shape, y_ref.shape)
    assert np.all(np.isfinite(y)), f"{what}: non-finite output"
    err = np.abs(y - y_ref)
    tol = tolerance(y_ref, rtol)
    bad = np.argwhere(err > tol)
    assert bad.size == 0, (f"{what}: {len(bad)} elements over tolerance {tol:.3e}; "
                           f"first {bad[:4].tolist()} err {err.max():.3e}")
    return float(err.max()), tol


class Case:
    """A seeded linear: host inputs (torch CPU) and lazily the oracle reference."""

    def __init__(self, seed: int, M: int, N: int, K: int):
        self.seed, self.M, self.N, self.K = seed, M, N, K
        self.qw, self.s, self.zw = si.layer(seed, N, K)
        self.x = si.x(seed, M, K)

    def to(self, dev):
        return (self.x.to(dev), self.qw.to(dev), self.s.to(dev), self.zw.to(dev))

    def reference(self) -> np.ndarray:
        return oracle.linear(si.as_u16(self.x), si.as_u32(self.qw), si.as_u16(self.s),
                             si.as_u32(self.zw))


def sampled_reference(seed: int, x_cpu: torch.Tensor, N: int, K: int, rows) -> np.ndarray:
    """Oracle outputs for selected rows of a (possibly huge) seeded layer, the
    rows regenerated on the host from the counter-based generator."""
    rows = np.asarray(rows, dtype=np.int64)
    qw, s, zw = si.layer(seed, N, K, rows=rows)
    local = np.arange(rows.size)
    return oracle.linear_rows(si.as_u16(x_cpu), si.as_u32(qw), si.as_u16(s), si.as_u32(zw), local)


def sample_rows(N: int, count: int, seed: int = 0) -> np.ndarray:
    rng = np.random.default_rng(seed)
    pick = set([0, N - 1, N // 2])
    pick.update(rng.integers(0, N, size=max(0, count - 3)).tolist())
    return np.array(sorted(pick), dtype=np.int64)
