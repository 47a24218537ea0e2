"""CPU oracle for the group-wise INT4 weight-only linear layer (W4A16).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The CUDA library never calls it and shares no code with it.

The arithmetic lives in ``w4a16_oracle.c`` (plain C, binary64); this module
compiles it with gcc into ``oracle/_build/`` and wraps it with ctypes, taking
and returning numpy arrays.  fp16 values travel as their uint16 bit patterns.

Method: forum.sourcefind.cn thread "vLLM on Hygon Z100", section 四 (W4A16):
w = (q - z) * s per group along K, y = x @ w^T.  Every function here is pinned
by ``tests/test_oracle_pins.py`` against exact rationals, closed forms, numpy's
binary16 conversion or an int64 matrix product.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "w4a16_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (portable flags: same results on x86 and Arm)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    # -ffp-contract=off: no fused multiply-add, every binary64 operation rounds
    # exactly as written.
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
           "-o", tmp, _SRC, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(lib):
    """Declare the C signatures on a loaded copy of the oracle library."""
    P = ctypes.c_void_p
    I = ctypes.c_int
    L = ctypes.c_long
    lib.w4o_half_to_double.argtypes = [ctypes.c_uint16]
    lib.w4o_half_to_double.restype = ctypes.c_double
    lib.w4o_double_to_half.argtypes = [ctypes.c_double]
    lib.w4o_double_to_half.restype = ctypes.c_uint16
    lib.w4o_pack.argtypes = [P, P, I, I, I, P, P]
    lib.w4o_unpack.argtypes = [P, P, I, I, I, P, P]
    lib.w4o_dequant.argtypes = [P, P, P, I, I, I, P]
    lib.w4o_silu_mul.argtypes = [P, I, I, P]
    lib.w4o_transpose_u4.argtypes = [P, L, L, ctypes.c_uint32, P]
    lib.w4o_transpose_u16.argtypes = [P, L, L, P]
    lib.w4o_dense_linear.argtypes = [P, P, I, I, I, I, P]
    lib.w4o_dense_linear_rows.argtypes = [P, P, I, I, I, I, P, I, P]
    lib.w4o_moe_align.argtypes = [P, I, I, P, P, P]
    lib.w4o_moe_linear.argtypes = [P, I, P, P, P, P, I, I, I, I, I, I, I, P]
    lib.w4o_moe_sum.argtypes = [P, P, I, I, I, P]
    lib.w4o_round_to_half.argtypes = [P, L, P]
    lib.w4o_half_array_to_double.argtypes = [P, L, P]
    lib.w4o_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.w4o_bf16_to_double.restype = ctypes.c_double
    lib.w4o_double_to_bf16.argtypes = [ctypes.c_double]
    lib.w4o_double_to_bf16.restype = ctypes.c_uint16
    lib.w4o_round_to_bf16.argtypes = [P, L, P]
    lib.w4o_bf16_array_to_double.argtypes = [P, L, P]
    lib.w4o_linear_dt.argtypes = [P, P, P, P, I, I, I, I, I, P, I]
    lib.w4o_linear_rows_dt.argtypes = [P, P, P, P, I, I, I, I, I, P, I, P, I]
    lib.w4o_add_residual_dt.argtypes = [P, P, L, I, P]
    for f in (lib.w4o_pack, lib.w4o_unpack, lib.w4o_dequant, lib.w4o_round_to_half,
              lib.w4o_half_array_to_double, lib.w4o_round_to_bf16,
              lib.w4o_bf16_array_to_double, lib.w4o_linear_dt, lib.w4o_linear_rows_dt,
              lib.w4o_silu_mul, lib.w4o_add_residual_dt,
              lib.w4o_transpose_u4, lib.w4o_transpose_u16, lib.w4o_dense_linear,
              lib.w4o_dense_linear_rows, lib.w4o_moe_align, lib.w4o_moe_linear,
              lib.w4o_moe_sum):
        f.restype = None
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
        return _lib


def _c(a: np.ndarray, dtype) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {np.dtype(dtype)}, got {a.dtype}")
    return a


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check_shape(K: int, group: int):
    if K % group or K % 8 or group <= 0:
        raise ValueError("K must be a multiple of group and of 8")


def zero_words(G: int) -> int:
    return (G + 7) // 8


def half_to_double(bits) -> np.ndarray:
    h = _c(np.asarray(bits, dtype=np.uint16).reshape(-1), np.uint16)
    out = np.empty(h.size, dtype=np.float64)
    _load().w4o_half_array_to_double(_ptr(h), h.size, _ptr(out))
    return out.reshape(np.shape(bits))


def double_to_half(v) -> np.ndarray:
    d = _c(np.asarray(v, dtype=np.float64).reshape(-1), np.float64)
    out = np.empty(d.size, dtype=np.uint16)
    _load().w4o_round_to_half(_ptr(d), d.size, _ptr(out))
    return out.reshape(np.shape(v))


def bf16_to_double(bits) -> np.ndarray:
    b = _c(np.asarray(bits, dtype=np.uint16).reshape(-1), np.uint16)
    out = np.empty(b.size, dtype=np.float64)
    _load().w4o_bf16_array_to_double(_ptr(b), b.size, _ptr(out))
    return out.reshape(np.shape(bits))


def double_to_bf16(v) -> np.ndarray:
    d = _c(np.asarray(v, dtype=np.float64).reshape(-1), np.float64)
    out = np.empty(d.size, dtype=np.uint16)
    _load().w4o_round_to_bf16(_ptr(d), d.size, _ptr(out))
    return out.reshape(np.shape(v))


_DTYPES = {"f16": 0, "bf16": 1}


def pack(q: np.ndarray, z: np.ndarray, group: int = 128):
    """q [N, K] uint8 (0..15), z [N, K/group] uint8 -> (qweight [N, K/8], zeros [N, ceil(G/8)]) uint32."""
    q = _c(q, np.uint8)
    z = _c(z, np.uint8)
    N, K = q.shape
    _check_shape(K, group)
    G = K // group
    assert z.shape == (N, G)
    qw = np.empty((N, K // 8), dtype=np.uint32)
    zw = np.empty((N, zero_words(G)), dtype=np.uint32)
    _load().w4o_pack(_ptr(q), _ptr(z), N, K, group, _ptr(qw), _ptr(zw))
    return qw, zw


def unpack(qweight: np.ndarray, zeros: np.ndarray, K: int, group: int = 128):
    qweight = _c(qweight, np.uint32)
    zeros = _c(zeros, np.uint32)
    N = qweight.shape[0]
    _check_shape(K, group)
    G = K // group
    assert qweight.shape == (N, K // 8) and zeros.shape == (N, zero_words(G))
    q = np.empty((N, K), dtype=np.uint8)
    z = np.empty((N, G), dtype=np.uint8)
    _load().w4o_unpack(_ptr(qweight), _ptr(zeros), N, K, group, _ptr(q), _ptr(z))
    return q, z


def dequant(qweight: np.ndarray, scales: np.ndarray, zeros: np.ndarray, K: int,
            group: int = 128) -> np.ndarray:
    """Exact w[n, k] = (q - z) * s in binary64, [N, K]."""
    qweight = _c(qweight, np.uint32)
    scales = _c(scales, np.uint16)
    zeros = _c(zeros, np.uint32)
    N = qweight.shape[0]
    _check_shape(K, group)
    G = K // group
    assert scales.shape == (N, G)
    w = np.empty((N, K), dtype=np.float64)
    _load().w4o_dequant(_ptr(qweight), _ptr(scales), _ptr(zeros), N, K, group, _ptr(w))
    return w


def linear(x: np.ndarray, qweight: np.ndarray, scales: np.ndarray, zeros: np.ndarray,
           group: int = 128, nthreads: int | None = None, dtype: str = "f16") -> np.ndarray:
    """y[M, N] = x @ dequant(W)^T in binary64.  x is [M, K] and scales [N, G]
    16-bit bit patterns (uint16) of type dtype: "f16" (IEEE binary16) or "bf16"."""
    x = _c(x, np.uint16)
    qweight = _c(qweight, np.uint32)
    scales = _c(scales, np.uint16)
    zeros = _c(zeros, np.uint32)
    M, K = x.shape
    N = qweight.shape[0]
    _check_shape(K, group)
    G = K // group
    assert qweight.shape == (N, K // 8) and scales.shape == (N, G)
    assert zeros.shape == (N, zero_words(G))
    y = np.empty((M, N), dtype=np.float64)
    nt = nthreads if nthreads is not None else (os.cpu_count() or 1)
    _load().w4o_linear_dt(_ptr(x), _ptr(qweight), _ptr(scales), _ptr(zeros), M, N, K,
                          group, _DTYPES[dtype], _ptr(y), nt)
    return y


def linear_rows(x: np.ndarray, qweight: np.ndarray, scales: np.ndarray,
                zeros: np.ndarray, rows, group: int = 128,
                nthreads: int | None = None, dtype: str = "f16") -> np.ndarray:
    """y[M, len(rows)] for the listed output rows; the weight arrays hold all N rows."""
    x = _c(x, np.uint16)
    qweight = _c(qweight, np.uint32)
    scales = _c(scales, np.uint16)
    zeros = _c(zeros, np.uint32)
    rows = _c(np.asarray(rows, dtype=np.int64), np.int64)
    M, K = x.shape
    N = qweight.shape[0]
    _check_shape(K, group)
    G = K // group
    assert qweight.shape == (N, K // 8) and scales.shape == (N, G)
    assert zeros.shape == (N, zero_words(G))
    if rows.size and (rows.min() < 0 or rows.max() >= N):
        raise IndexError("row index out of range")
    y = np.empty((M, rows.size), dtype=np.float64)
    nt = nthreads if nthreads is not None else (os.cpu_count() or 1)
    _load().w4o_linear_rows_dt(_ptr(x), _ptr(qweight), _ptr(scales), _ptr(zeros), M, N,
                               K, group, _DTYPES[dtype], _ptr(rows), int(rows.size), _ptr(y), nt)
    return y



def silu_mul(y: np.ndarray) -> np.ndarray:
    """out[M, I] = silu(y[:, :I]) * y[:, I:] in binary64 (y is [M, 2I], gate
    columns first): the epilogue of a fused gate+up projection."""
    y = _c(y, np.float64)
    M, N2 = y.shape
    assert N2 % 2 == 0
    out = np.empty((M, N2 // 2), dtype=np.float64)
    _load().w4o_silu_mul(_ptr(y), M, N2 // 2, _ptr(out))
    return out


def add_residual(y: np.ndarray, residual: np.ndarray, dtype: str = "f16") -> np.ndarray:
    """out = y + residual in binary64; residual as 16-bit bits (uint16) of type
    dtype ("f16" or "bf16"), same shape."""
    y = _c(y, np.float64)
    r = _c(residual, np.uint16)
    assert r.shape == y.shape
    out = np.empty_like(y)
    _load().w4o_add_residual_dt(_ptr(y), _ptr(r), int(y.size), _DTYPES[dtype], _ptr(out))
    return out


SEQUENTIAL_ORDER = 0x76543210


def transpose_u4(src: np.ndarray, rows: int, cols: int, order: int = SEQUENTIAL_ORDER) -> np.ndarray:
    """Packed 4-bit transpose: src [rows, cols/8] uint32 packed along cols (nibble
    order `order`) -> [cols, ceil(rows/8)] uint32 packed along rows, sequential."""
    src = _c(src, np.uint32)
    assert cols % 8 == 0 and src.size == rows * cols // 8
    dst = np.empty((cols, (rows + 7) // 8), dtype=np.uint32)
    _load().w4o_transpose_u4(_ptr(src), rows, cols, order, _ptr(dst))
    return dst


def transpose_u16(src: np.ndarray) -> np.ndarray:
    """[rows, cols] uint16 (fp16 bits) -> [cols, rows]."""
    src = _c(src, np.uint16)
    rows, cols = src.shape
    dst = np.empty((cols, rows), dtype=np.uint16)
    _load().w4o_transpose_u16(_ptr(src), rows, cols, _ptr(dst))
    return dst


def dense_linear(x: np.ndarray, w: np.ndarray, dtype: str = "f16", rows=None) -> np.ndarray:
    """y[M, N] = x @ w^T in binary64 for 16-bit x [M, K] and w [N, K] (bit
    patterns, type dtype); with rows, only those output rows: y[M, len(rows)]."""
    x = _c(x, np.uint16)
    w = _c(w, np.uint16)
    M, K = x.shape
    N = w.shape[0]
    assert w.shape == (N, K)
    if rows is None:
        y = np.empty((M, N), dtype=np.float64)
        _load().w4o_dense_linear(_ptr(x), _ptr(w), M, N, K, _DTYPES[dtype], _ptr(y))
        return y
    rows = _c(np.asarray(rows, dtype=np.int64), np.int64)
    if rows.size and (rows.min() < 0 or rows.max() >= N):
        raise IndexError("row index out of range")
    y = np.empty((M, rows.size), dtype=np.float64)
    _load().w4o_dense_linear_rows(_ptr(x), _ptr(w), M, N, K, _DTYPES[dtype], _ptr(rows),
                                  int(rows.size), _ptr(y))
    return y


def moe_align(ids: np.ndarray, E: int):
    """Slots grouped by expert (stable): (sorted [S], pos [S], offsets [E+1]) int32."""
    ids = _c(np.asarray(ids, dtype=np.int32).reshape(-1), np.int32)
    assert ids.size == 0 or (ids.min() >= 0 and ids.max() < E)
    S = ids.size
    srt = np.empty(S, dtype=np.int32)
    pos = np.empty(S, dtype=np.int32)
    off = np.empty(E + 1, dtype=np.int32)
    _load().w4o_moe_align(_ptr(ids), S, E, _ptr(srt), _ptr(pos), _ptr(off))
    return srt, pos, off


def moe_linear(x: np.ndarray, qweight: np.ndarray, scales: np.ndarray, zeros: np.ndarray,
               ids: np.ndarray, per_slot: bool = False, group: int = 128,
               dtype: str = "f16") -> np.ndarray:
    """Expert linears per slot: y [T*k, N] (binary64).  qweight [E, N, K/8],
    scales [E, N, G], zeros [E, N, ceil(G/8)]; ids [T, k]; x [T, K] by token,
    or [T*k, K] by slot when per_slot."""
    ids = _c(np.asarray(ids, dtype=np.int32), np.int32)
    T, k = ids.shape
    qweight = _c(qweight, np.uint32)
    scales = _c(scales, np.uint16)
    zeros = _c(zeros, np.uint32)
    E, N, KW = qweight.shape
    K = KW * 8
    x = _c(x, np.uint16)
    assert x.shape == ((T * k if per_slot else T), K)
    assert ids.size == 0 or (ids.min() >= 0 and ids.max() < E)
    y = np.empty((T * k, N), dtype=np.float64)
    _load().w4o_moe_linear(_ptr(x), int(per_slot), _ptr(qweight), _ptr(scales), _ptr(zeros),
                           _ptr(ids), T, k, E, N, K, group, _DTYPES[dtype], _ptr(y))
    return y


def moe_sum(y: np.ndarray, weights: np.ndarray) -> np.ndarray:
    """out [T, N] = sum_j weights[t, j] * y[t*k + j] in binary64."""
    w = _c(np.asarray(weights, dtype=np.float64), np.float64)
    T, k = w.shape
    y = _c(y, np.float64)
    N = y.shape[1]
    assert y.shape == (T * k, N)
    out = np.empty((T, N), dtype=np.float64)
    _load().w4o_moe_sum(_ptr(y), _ptr(w), T, k, N, _ptr(out))
    return out
