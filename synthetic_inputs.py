"""Seeded synthetic inputs for the W4A16 linear layer, shared by tests, the
benchmark and the oracle checks.

This module holds no arithmetic of the method itself: it only draws random
bits and values.  Every draw is counter based -- element ``i`` of tensor
``tensor_id`` under ``seed`` is a pure function of ``(seed, tensor_id, i)`` --
so any subset of rows can be regenerated on its own (the oracle recomputes
sampled rows of a multi-gigabyte weight set this way), and the same call gives
the same bits on CPU and on a CUDA device.

Generator: splitmix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014; the 64-bit finaliser as published by Vigna),
applied to ``key(seed, tensor_id) + (i + 1) * gamma``.  It runs in torch int64
tensors (wrap-around multiply, masked logical shifts), so the integer draws are
bit-identical on every device.  ``tests/test_synthetic_inputs.py`` checks the
torch version against a numpy uint64 restatement.

Value recipe, after the decode workload the pages benchmark (packed INT4
weights with per-group fp16 scale and 4-bit zero, fp16 activations):
  * qweight: uniform random 32-bit words = 8 iid uniform nibbles 0..15;
  * zeros:   uniform random words, nibbles past the last group set to 0;
  * scales:  fp16 of U[0.002, 0.02];
  * x:       fp16 of N(0, 1) (Box-Muller, computed on the host only);
  * residual (the epilogue's second input): fp16 of N(0, 4^2), a spread like
    that of the linear's outputs, so that a dropped residual shows;
  * dense 16-bit weights: fp16 of N(0, 0.05^2), the spread of the dequantised
    4-bit weights above.
"""
from __future__ import annotations

import math

import numpy as np
import torch

GAMMA = 0x9E3779B97F4A7C15
MIX1 = 0xBF58476D1CE4E5B9
MIX2 = 0x94D049BB133111EB
_M64 = (1 << 64) - 1

T_QWEIGHT = 1
T_ZEROS = 2
T_SCALES = 3
T_X = 4
T_RESIDUAL = 5
T_DENSE_W = 6


def _signed(c: int) -> int:
    """A 64-bit pattern as the int64 value with the same bits."""
    c &= _M64
    return c - (1 << 64) if c >= (1 << 63) else c


def _mix_int(z: int) -> int:
    z &= _M64
    z = ((z ^ (z >> 30)) * MIX1) & _M64
    z = ((z ^ (z >> 27)) * MIX2) & _M64
    return z ^ (z >> 31)


def key(seed: int, tensor_id: int) -> int:
    """Per-tensor stream key (a Python int in [0, 2^64))."""
    return _mix_int(_mix_int(seed * GAMMA + 0x5851F42D4C957F2D) + tensor_id * GAMMA)


def _lsr(z: torch.Tensor, s: int) -> torch.Tensor:
    return (z >> s) & ((1 << (64 - s)) - 1)


def hash_u64(seed: int, tensor_id: int, idx: torch.Tensor) -> torch.Tensor:
    """splitmix64 output for counters ``idx`` (int64 tensor); result int64 holding uint64 bits."""
    k = key(seed, tensor_id)
    z = idx.to(torch.int64) + 1
    z = z * _signed(GAMMA) + _signed(k)
    z = (z ^ _lsr(z, 30)) * _signed(MIX1)
    z = (z ^ _lsr(z, 27)) * _signed(MIX2)
    return z ^ _lsr(z, 31)


def hash_u64_numpy(seed: int, tensor_id: int, idx: np.ndarray) -> np.ndarray:
    """The same generator in numpy uint64 arithmetic (wrap-around by definition)."""
    k = np.uint64(key(seed, tensor_id))
    with np.errstate(over="ignore"):
        z = idx.astype(np.uint64) + np.uint64(1)
        z = z * np.uint64(GAMMA) + k
        z = (z ^ (z >> np.uint64(30))) * np.uint64(MIX1)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(MIX2)
        return z ^ (z >> np.uint64(31))


def _row_index(N: int, width: int, rows, device) -> torch.Tensor:
    if rows is None:
        r = torch.arange(N, dtype=torch.int64, device=device)
    else:
        r = torch.as_tensor(rows, dtype=torch.int64, device=device)
    return r[:, None] * width + torch.arange(width, dtype=torch.int64, device=device)[None, :]


def _low32(h: torch.Tensor) -> torch.Tensor:
    """Low 32 bits of each value, as int32 holding the uint32 bit pattern."""
    lo = h & 0xFFFFFFFF
    return torch.where(lo >= (1 << 31), lo - (1 << 32), lo).to(torch.int32)


def qweight(seed: int, N: int, K: int, rows=None, device="cpu") -> torch.Tensor:
    """[len(rows) or N, K/8] int32 tensor holding uint32 words (8 nibbles each)."""
    assert K % 8 == 0
    return _low32(hash_u64(seed, T_QWEIGHT, _row_index(N, K // 8, rows, device)))


def zeros(seed: int, N: int, K: int, group: int = 128, rows=None, device="cpu") -> torch.Tensor:
    """[rows, ceil(G/8)] int32 tensor of packed 4-bit zeros; pad nibbles are 0."""
    G = K // group
    ZW = (G + 7) // 8
    w = hash_u64(seed, T_ZEROS, _row_index(N, ZW, rows, device)) & 0xFFFFFFFF
    tail = G - 8 * (ZW - 1)  # groups held by the last word of a row (1..8)
    if tail < 8:
        w[:, ZW - 1] &= (1 << (4 * tail)) - 1
    return torch.where(w >= (1 << 31), w - (1 << 32), w).to(torch.int32)


def scales(seed: int, N: int, K: int, group: int = 128, rows=None, device="cpu",
           lo: float = 0.002, hi: float = 0.02) -> torch.Tensor:
    """[rows, G] float16 tensor, fp16 of U[lo, hi] (binary64 draw -> fp32 -> fp16)."""
    G = K // group
    h = hash_u64(seed, T_SCALES, _row_index(N, G, rows, device))
    u = _lsr(h, 11).to(torch.float64) * (2.0 ** -53)
    v = u * (hi - lo) + lo
    return v.to(torch.float32).to(torch.float16)


def _normal_f16(seed: int, tensor_id: int, M: int, K: int, std: float) -> torch.Tensor:
    n = M * K
    idx = np.arange(2 * ((n + 1) // 2), dtype=np.uint64)
    h = hash_u64_numpy(seed, tensor_id, idx)
    u = (h >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    u1 = 1.0 - u[0::2]          # (0, 1]
    u2 = u[1::2]
    r = np.sqrt(-2.0 * np.log(u1))
    t = 2.0 * math.pi * u2
    z = np.empty(u.size, dtype=np.float64)
    z[0::2] = r * np.cos(t)
    z[1::2] = r * np.sin(t)
    if std != 1.0:
        z *= std
    return torch.from_numpy(z[:n].astype(np.float32).astype(np.float16).reshape(M, K))


def x(seed: int, M: int, K: int) -> torch.Tensor:
    """[M, K] float16 CPU tensor of N(0, 1) draws (Box-Muller on the host)."""
    return _normal_f16(seed, T_X, M, K, 1.0)


def dense_weight(seed: int, N: int, K: int, std: float = 0.05) -> torch.Tensor:
    """[N, K] float16 CPU tensor of N(0, std^2) draws: 16-bit weights of the
    dense linear (the spread of dequantised 4-bit weights here)."""
    return _normal_f16(seed, T_DENSE_W, N, K, std)


def residual(seed: int, M: int, N: int, std: float = 4.0) -> torch.Tensor:
    """[M, N] float16 CPU tensor of N(0, std^2) draws."""
    return _normal_f16(seed, T_RESIDUAL, M, N, std)


def as_u32(t: torch.Tensor) -> np.ndarray:
    """int32 torch tensor of packed words -> numpy uint32 view (on the host)."""
    return t.detach().cpu().contiguous().numpy().view(np.uint32)


def as_u16(t: torch.Tensor) -> np.ndarray:
    """float16 torch tensor -> numpy uint16 bit patterns (on the host)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def layer(seed: int, N: int, K: int, group: int = 128, rows=None, device="cpu"):
    """(qweight, scales, zeros) for one linear layer."""
    return (qweight(seed, N, K, rows, device), scales(seed, N, K, group, rows, device),
            zeros(seed, N, K, group, rows, device))


def config_seed(config: int, layer_index: int = 0, shape_index: int = 0) -> int:
    """Seed for a workload: config id, decode-round layer and shape within the layer."""
    return (config << 20) | (layer_index << 4) | shape_index
