"""Thin ctypes binding over the C ABI in ``include/w4a16.h``.

Argument marshalling only: every step of the computation runs in the CUDA
library ``_lib/libw4a16.so``.  Tensors are torch CUDA tensors (device memory
and streams come from PyTorch); fp16 data crosses the ABI as uint16 bit
patterns.  Importing this module fails loudly if the library has not been
built: there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libw4a16.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"W4A16 CUDA library not built ({LIB_PATH} missing). Build it with "
        "`python weight_only_int4_w4a16_gb300/build.py` or __graft_entry__.build().")

lib = ctypes.CDLL(LIB_PATH)

GROUP = 128

W4A16_OK = 0
W4A16_ERR_INVALID_ARG = 1
W4A16_ERR_UNSUPPORTED = 2
W4A16_ERR_MISALIGNED = 3
W4A16_ERR_WORKSPACE = 4
W4A16_ERR_NOT_INITIALIZED = 5
W4A16_ERR_CUDA = 6
W4A16_ERR_DEVICE = 7

RUNG_AUTO = -1
RUNG_GEMV = 0
RUNG_GEMV_SPLITK = 1
RUNG_TC = 2
RUNG_TC_SPLITK = 3
RUNG_MMA = 4
RUNG_MMA_SPLITK = 5
NUM_RUNGS = 6

EPILOGUE_NONE = 0
EPILOGUE_RESIDUAL = 1
EPILOGUE_SILU_MUL = 2

DTYPE_F16 = 0
DTYPE_BF16 = 1

MOE_PATH_AUTO = 0
MOE_PATH_CHAIN = 1
MOE_PATH_DECODE = 2
_DTYPE_OF = {torch.float16: DTYPE_F16, torch.bfloat16: DTYPE_BF16}

_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t


class LinearDesc(ctypes.Structure):
    """Mirror of ``w4a16_linear_desc``."""
    _fields_ = [("x", _P), ("qweight", _P), ("scales", _P), ("zeros", _P), ("y", _P),
                ("N", _I), ("K", _I), ("group", _I), ("epilogue", _I), ("residual", _P),
                ("dtype", _I)]


def _sig(name, args, res=_I):
    f = getattr(lib, name)
    f.argtypes = args
    f.restype = res
    return f


_sig("w4a16_init", [_I, _SZ])
_sig("w4a16_shutdown", [])
_sig("w4a16_workspace_bytes", [_I, _I, _I, _I], _SZ)
_sig("w4a16_pack", [_P, _P, _I, _I, _I, _P, _P, _P])
_sig("w4a16_unpack", [_P, _P, _I, _I, _I, _P, _P, _P])
_sig("w4a16_dequant", [_P, _P, _P, _I, _I, _I, _P, _P, _P])
_sig("w4a16_repack_transpose", [_P, _I, _I, ctypes.c_uint32, _P, _P])
_sig("w4a16_transpose_f16", [_P, _I, _I, _P, _P])
_sig("w4a16_linear", [_P, _P, _P, _P, _I, _I, _I, _I, _P, _P])
_sig("w4a16_linear_noalloc", [_P, _P, _P, _P, _I, _I, _I, _I, _P, _P])
_sig("w4a16_linear_epilogue", [_P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P])
_sig("w4a16_linear_ex", [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _P])
_sig("w4a16_dense_linear", [_P, _P, _I, _I, _I, _I, _P, _P])
_sig("w4a16_moe_align", [_P, _I, _I, _P, _P, _P, _P])
_sig("w4a16_moe_create", [_I, _I, _I, _I, _P, _P, _P, _I, _I, _I, ctypes.POINTER(_P)])
_sig("w4a16_moe_destroy", [_P])
_sig("w4a16_moe_linear", [_P, _P, _I, _P, _P, _I, _P, _P])
_sig("w4a16_moe_sum", [_P, _P, _P, _I, _I, _I, _I, _P, _P])
_sig("w4a16_moe_mlp_set_path", [_P, _I])
_sig("w4a16_moe_mlp_path", [_P, _I, ctypes.POINTER(_I)])
_sig("w4a16_moe_mlp_buffers", [_P, ctypes.POINTER(_P), ctypes.POINTER(_P)])
_sig("w4a16_wait_probe", [_P])
_sig("w4a16_moe_mlp_create", [_P, _P, _I, _I, ctypes.POINTER(_P)])
_sig("w4a16_moe_mlp_destroy", [_P])
_sig("w4a16_moe_mlp", [_P, _P, _P, _P, _I, _P, _P])
_sig("w4a16_decode_round", [ctypes.POINTER(LinearDesc), _I, _I, _P])
_sig("w4a16_round_graph_create", [ctypes.POINTER(LinearDesc), _I, _I, ctypes.POINTER(_P)])
_sig("w4a16_round_graph_launch", [_P, _P])
_sig("w4a16_round_graph_destroy", [_P])
_sig("w4a16_select_rung", [_I, _I, _I, _I])
_sig("w4a16_plan_info", [_I, _I, _I, _I, _I, _I, ctypes.POINTER(ctypes.c_int32)])
_sig("w4a16_set_forced_rung", [_I])
_sig("w4a16_probe_counts", [ctypes.POINTER(ctypes.c_uint64), _I])
_sig("w4a16_probe_reset", [], None)
_sig("w4a16_kernel_launches", [], ctypes.c_uint64)
_sig("w4a16_rung_name", [_I], ctypes.c_char_p)
_sig("w4a16_status_string", [_I], ctypes.c_char_p)
_sig("w4a16_device_status", [_P, ctypes.POINTER(_I)])
_sig("w4a16_last_cuda_error", [])
_sig("w4a16_device_sm_count", [])

EXPORTED = ["w4a16_init", "w4a16_shutdown", "w4a16_workspace_bytes", "w4a16_pack",
            "w4a16_unpack", "w4a16_dequant", "w4a16_repack_transpose", "w4a16_transpose_f16",
            "w4a16_linear", "w4a16_linear_noalloc",
            "w4a16_linear_epilogue", "w4a16_linear_ex", "w4a16_dense_linear",
            "w4a16_moe_align", "w4a16_moe_create", "w4a16_moe_destroy", "w4a16_moe_linear",
            "w4a16_moe_sum", "w4a16_moe_mlp_create", "w4a16_moe_mlp_destroy", "w4a16_moe_mlp",
            "w4a16_moe_mlp_set_path", "w4a16_moe_mlp_path", "w4a16_moe_mlp_buffers",
            "w4a16_decode_round",
            "w4a16_round_graph_create", "w4a16_round_graph_launch", "w4a16_round_graph_destroy",
            "w4a16_select_rung", "w4a16_plan_info", "w4a16_set_forced_rung", "w4a16_probe_counts",
            "w4a16_probe_reset", "w4a16_kernel_launches", "w4a16_rung_name", "w4a16_status_string",
            "w4a16_device_status", "w4a16_wait_probe", "w4a16_last_cuda_error",
            "w4a16_device_sm_count"]


class W4A16Error(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        msg = lib.w4a16_status_string(status).decode()
        if status == W4A16_ERR_CUDA:
            msg += f" (cudaError {lib.w4a16_last_cuda_error()})"
        super().__init__(f"{what}: {msg} [status {status}]")


def _check(status: int, what: str):
    if status != W4A16_OK:
        raise W4A16Error(status, what)


def _stream_ptr(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _dev(t: torch.Tensor, dtype, name: str, host_ok: bool = False):
    """The tensor's address after checks.  host_ok: an output that may also be
    page-locked host memory (pin_memory()), which the kernels write directly."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if not t.is_cuda and not (host_ok and t.is_pinned()):
        raise ValueError(f"{name} must live on a CUDA device" +
                         (" or in page-locked host memory" if host_ok else ""))
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def rung_name(rung: int) -> str:
    return lib.w4a16_rung_name(rung).decode()


# ---------------------------------------------------------------------------
# Same names as the C ABI
# ---------------------------------------------------------------------------
def w4a16_init(device: int = 0, workspace_bytes: int = 0) -> None:
    _check(lib.w4a16_init(device, workspace_bytes), "w4a16_init")


def w4a16_shutdown() -> None:
    _check(lib.w4a16_shutdown(), "w4a16_shutdown")


def w4a16_workspace_bytes(M: int, N: int, K: int, group: int = GROUP) -> int:
    return int(lib.w4a16_workspace_bytes(M, N, K, group))


def w4a16_pack(q: torch.Tensor, z: torch.Tensor, group: int = GROUP, qweight=None, zeros=None,
               stream=None):
    """q [N, K] uint8, z [N, K/group] uint8 -> (qweight [N, K/8], zeros [N, ceil(G/8)]) int32 (uint32 bits)."""
    N, K = q.shape
    G = K // group if group else 0
    if qweight is None:
        qweight = torch.empty((N, K // 8), dtype=torch.int32, device=q.device)
    if zeros is None:
        zeros = torch.empty((N, (G + 7) // 8), dtype=torch.int32, device=q.device)
    _check(lib.w4a16_pack(_dev(q, torch.uint8, "q"), _dev(z, torch.uint8, "z"), N, K, group,
                          _dev(qweight, torch.int32, "qweight"), _dev(zeros, torch.int32, "zeros"),
                          _stream_ptr(stream)), "w4a16_pack")
    return qweight, zeros


def w4a16_unpack(qweight: torch.Tensor, zeros: torch.Tensor, K: int, group: int = GROUP,
                 stream=None):
    N = qweight.shape[0]
    G = K // group if group else 0
    q = torch.empty((N, K), dtype=torch.uint8, device=qweight.device)
    z = torch.empty((N, G), dtype=torch.uint8, device=qweight.device)
    _check(lib.w4a16_unpack(_dev(qweight, torch.int32, "qweight"), _dev(zeros, torch.int32, "zeros"),
                            N, K, group, q.data_ptr(), z.data_ptr(), _stream_ptr(stream)),
           "w4a16_unpack")
    return q, z


def w4a16_dequant(qweight: torch.Tensor, scales: torch.Tensor, zeros: torch.Tensor, K: int,
                  group: int = GROUP, f32: bool = True, f16: bool = True, stream=None):
    N = qweight.shape[0]
    w32 = torch.empty((N, K), dtype=torch.float32, device=qweight.device) if f32 else None
    w16 = torch.empty((N, K), dtype=torch.float16, device=qweight.device) if f16 else None
    _check(lib.w4a16_dequant(_dev(qweight, torch.int32, "qweight"),
                             _dev(scales, torch.float16, "scales"), _dev(zeros, torch.int32, "zeros"),
                             N, K, group, w32.data_ptr() if f32 else None,
                             w16.data_ptr() if f16 else None, _stream_ptr(stream)), "w4a16_dequant")
    return w32, w16


SEQUENTIAL_ORDER = 0x76543210


def w4a16_repack_transpose(src: torch.Tensor, rows: int, cols: int,
                           src_order: int = SEQUENTIAL_ORDER, dst=None, stream=None) -> torch.Tensor:
    """src [rows, cols/8] int32 (4-bit values packed along cols, nibble order
    src_order) -> [cols, ceil(rows/8)] int32 packed along rows (sequential)."""
    if dst is None:
        dst = torch.empty((cols, (rows + 7) // 8), dtype=torch.int32, device=src.device)
    _check(lib.w4a16_repack_transpose(_dev(src, torch.int32, "src"), rows, cols, src_order,
                                      _dev(dst, torch.int32, "dst"), _stream_ptr(stream)),
           "w4a16_repack_transpose")
    return dst


def w4a16_transpose_f16(src: torch.Tensor, dst=None, stream=None) -> torch.Tensor:
    """[rows, cols] fp16 -> [cols, rows]."""
    rows, cols = src.shape
    if dst is None:
        dst = torch.empty((cols, rows), dtype=torch.float16, device=src.device)
    _check(lib.w4a16_transpose_f16(_dev(src, torch.float16, "src"), rows, cols,
                                   _dev(dst, torch.float16, "dst"), _stream_ptr(stream)),
           "w4a16_transpose_f16")
    return dst


def w4a16_linear(x: torch.Tensor, qweight: torch.Tensor, scales: torch.Tensor,
                 zeros: torch.Tensor, group: int = GROUP, y=None, stream=None) -> torch.Tensor:
    """y [M, N] fp16 = x [M, K] fp16 @ dequant(qweight, scales, zeros)^T.

    y (here and in the other linear calls and round descriptors) may be a
    pinned host tensor: the kernels then store the result straight into host
    memory, and it is there once the stream has passed the call."""
    M, K = x.shape
    N = qweight.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.float16, device=x.device)
    _check(lib.w4a16_linear(_dev(x, torch.float16, "x"), _dev(qweight, torch.int32, "qweight"),
                            _dev(scales, torch.float16, "scales"), _dev(zeros, torch.int32, "zeros"),
                            M, N, K, group, _dev(y, torch.float16, "y", True),
                            _stream_ptr(stream)),
           "w4a16_linear")
    return y


def w4a16_linear_noalloc(x: torch.Tensor, qweight: torch.Tensor, scales: torch.Tensor,
                         zeros: torch.Tensor, y: torch.Tensor, group: int = GROUP,
                         stream=None) -> torch.Tensor:
    """w4a16_linear for M <= 8 that allocates nothing (y must be given) and needs
    no w4a16_init: its split-K scratch is static device memory of the library."""
    M, K = x.shape
    N = qweight.shape[0]
    _check(lib.w4a16_linear_noalloc(_dev(x, torch.float16, "x"),
                                    _dev(qweight, torch.int32, "qweight"),
                                    _dev(scales, torch.float16, "scales"),
                                    _dev(zeros, torch.int32, "zeros"), M, N, K, group,
                                    _dev(y, torch.float16, "y", True), _stream_ptr(stream)),
           "w4a16_linear_noalloc")
    return y


def w4a16_linear_epilogue(x: torch.Tensor, qweight: torch.Tensor, scales: torch.Tensor,
                          zeros: torch.Tensor, epilogue: int, residual=None, group: int = GROUP,
                          y=None, stream=None) -> torch.Tensor:
    """w4a16_linear followed in the same kernel by an epilogue: EPILOGUE_RESIDUAL
    (y [M, N] = h + residual [M, N]; residual may be y itself) or EPILOGUE_SILU_MUL
    (y [M, N/2] = silu(h[:, :N/2]) * h[:, N/2:]), h = x @ W^T in fp32."""
    M, K = x.shape
    N = qweight.shape[0]
    cols = N // 2 if epilogue == EPILOGUE_SILU_MUL else N
    if y is None:
        y = torch.empty((M, cols), dtype=torch.float16, device=x.device)
    r = _dev(residual, torch.float16, "residual") if residual is not None else None
    _check(lib.w4a16_linear_epilogue(_dev(x, torch.float16, "x"),
                                     _dev(qweight, torch.int32, "qweight"),
                                     _dev(scales, torch.float16, "scales"),
                                     _dev(zeros, torch.int32, "zeros"), M, N, K, group, epilogue,
                                     r, _dev(y, torch.float16, "y", True), _stream_ptr(stream)),
           "w4a16_linear_epilogue")
    return y


def w4a16_linear_ex(x: torch.Tensor, qweight: torch.Tensor, scales: torch.Tensor,
                    zeros: torch.Tensor, epilogue: int = EPILOGUE_NONE, residual=None,
                    group: int = GROUP, y=None, stream=None) -> torch.Tensor:
    """w4a16_linear_epilogue for fp16 or bf16 data: x, scales, residual and y
    share one dtype (torch.float16 or torch.bfloat16)."""
    M, K = x.shape
    N = qweight.shape[0]
    if x.dtype not in _DTYPE_OF:
        raise TypeError(f"x must be float16 or bfloat16, got {x.dtype}")
    dt = x.dtype
    cols = N // 2 if epilogue == EPILOGUE_SILU_MUL else N
    if y is None:
        y = torch.empty((M, cols), dtype=dt, device=x.device)
    r = _dev(residual, dt, "residual") if residual is not None else None
    _check(lib.w4a16_linear_ex(_dev(x, dt, "x"), _dev(qweight, torch.int32, "qweight"),
                               _dev(scales, dt, "scales"), _dev(zeros, torch.int32, "zeros"),
                               M, N, K, group, _DTYPE_OF[dt], epilogue, r, _dev(y, dt, "y", True),
                               _stream_ptr(stream)),
           "w4a16_linear_ex")
    return y


def w4a16_dense_linear(x: torch.Tensor, w: torch.Tensor, y=None, stream=None) -> torch.Tensor:
    """y [M, N] = x [M, K] @ w [N, K]^T for fp16 or bf16 weights (x, w and y of
    one dtype), fp32 accumulation."""
    M, K = x.shape
    N = w.shape[0]
    if x.dtype not in _DTYPE_OF:
        raise TypeError(f"x must be float16 or bfloat16, got {x.dtype}")
    dt = x.dtype
    if y is None:
        y = torch.empty((M, N), dtype=dt, device=x.device)
    _check(lib.w4a16_dense_linear(_dev(x, dt, "x"), _dev(w, dt, "w"), M, N, K, _DTYPE_OF[dt],
                                  _dev(y, dt, "y"), _stream_ptr(stream)),
           "w4a16_dense_linear")
    return y


def w4a16_moe_align(topk_ids: torch.Tensor, E: int, stream=None):
    """topk_ids [T, k] int32 -> (sorted [T*k], pos [T*k], offsets [E+1]) int32."""
    n = topk_ids.numel()
    dev = topk_ids.device
    srt = torch.empty(n, dtype=torch.int32, device=dev)
    pos = torch.empty(n, dtype=torch.int32, device=dev)
    off = torch.empty(E + 1, dtype=torch.int32, device=dev)
    _check(lib.w4a16_moe_align(_dev(topk_ids, torch.int32, "topk_ids"), n, E, srt.data_ptr(),
                               pos.data_ptr(), off.data_ptr(), _stream_ptr(stream)),
           "w4a16_moe_align")
    return srt, pos, off


class _DeviceRows:
    """A device pointer seen as 16-bit rows (the CUDA array interface), for
    torch.as_tensor: no copy, no ownership."""

    def __init__(self, ptr: int, shape):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": "<i2",
                                          "data": (ptr, False), "version": 3, "strides": None}


def _view_device(ptr: int, shape, dt, dev) -> torch.Tensor:
    return torch.as_tensor(_DeviceRows(ptr, shape), device=dev).view(dt)


class MoeExperts:
    """E stacked W4A16 experts (qweight [E, N, K/8], scales [E, N, G], zeros
    [E, N, ceil(G/8)]) prepared for w4a16_moe_linear."""

    def __init__(self, qweight, scales, zeros, epilogue: int = EPILOGUE_NONE,
                 max_slots: int = 64, group: int = GROUP):
        E, N, KW = qweight.shape
        self.E, self.N, self.K, self.epilogue = E, N, KW * 8, epilogue
        self.dtype = scales.dtype
        self._keep = (qweight, scales, zeros)
        h = _P()
        _check(lib.w4a16_moe_create(E, N, self.K, group, _dev(qweight, torch.int32, "qweight"),
                                    _dev(scales, self.dtype, "scales"),
                                    _dev(zeros, torch.int32, "zeros"), epilogue,
                                    _DTYPE_OF[self.dtype], max_slots, ctypes.byref(h)),
               "w4a16_moe_create")
        self.handle = h.value

    def linear(self, x, sorted_slots, offsets, n_slots: int, gather_k: int = 0, y=None,
               stream=None):
        cols = self.N // 2 if self.epilogue == EPILOGUE_SILU_MUL else self.N
        if y is None:
            y = torch.empty((n_slots, cols), dtype=self.dtype, device=x.device)
        _check(lib.w4a16_moe_linear(self.handle, _dev(x, self.dtype, "x"), gather_k,
                                    _dev(sorted_slots, torch.int32, "sorted"),
                                    _dev(offsets, torch.int32, "offsets"), n_slots,
                                    _dev(y, self.dtype, "y"), _stream_ptr(stream)),
               "w4a16_moe_linear")
        return y

    def destroy(self):
        if self.handle:
            _check(lib.w4a16_moe_destroy(self.handle), "w4a16_moe_destroy")
            self.handle = None


class MoeMlp:
    """gate+up then down over one routing (two MoeExperts): the one-launch
    decode kernel when a call fits it, else the chain (path: MOE_PATH_*)."""

    def __init__(self, gate_up: MoeExperts, down: MoeExperts, max_tokens: int, k: int,
                 path: int = 0):
        self.gate_up, self.down, self.k = gate_up, down, k
        h = _P()
        _check(lib.w4a16_moe_mlp_create(gate_up.handle, down.handle, max_tokens, k,
                                        ctypes.byref(h)), "w4a16_moe_mlp_create")
        self.handle = h.value
        self.set_path(path)

    def set_path(self, path: int):
        _check(lib.w4a16_moe_mlp_set_path(self.handle, path), "w4a16_moe_mlp_set_path")

    def path(self, T: int) -> int:
        """The path (MOE_PATH_CHAIN or MOE_PATH_DECODE) a call with T tokens takes."""
        p = _I()
        _check(lib.w4a16_moe_mlp_path(self.handle, T, ctypes.byref(p)), "w4a16_moe_mlp_path")
        return p.value

    def intermediates(self, n_slots: int):
        """The last call's intermediate rows h [n_slots, I] and expert outputs
        o [n_slots, N] in sorted order, as views of the handle's device buffers."""
        hp, op = _P(), _P()
        _check(lib.w4a16_moe_mlp_buffers(self.handle, ctypes.byref(hp), ctypes.byref(op)),
               "w4a16_moe_mlp_buffers")
        dt = self.gate_up.dtype
        dev = torch.device("cuda", torch.cuda.current_device())
        I, N = self.down.K, self.down.N
        return (_view_device(hp.value, (n_slots, I), dt, dev),
                _view_device(op.value, (n_slots, N), dt, dev))

    def __call__(self, x, topk_ids, weights, out=None, stream=None):
        T = x.shape[0]
        dt = self.gate_up.dtype
        if out is None:
            out = torch.empty((T, self.down.N), dtype=dt, device=x.device)
        _check(lib.w4a16_moe_mlp(self.handle, _dev(x, dt, "x"), _dev(topk_ids, torch.int32, "topk_ids"),
                                 _dev(weights, torch.float32, "weights"), T, _dev(out, dt, "out"),
                                 _stream_ptr(stream)), "w4a16_moe_mlp")
        return out

    def destroy(self):
        if self.handle:
            _check(lib.w4a16_moe_mlp_destroy(self.handle), "w4a16_moe_mlp_destroy")
            self.handle = None


def w4a16_moe_sum(y_sorted: torch.Tensor, pos: torch.Tensor, weights: torch.Tensor, out=None,
                  stream=None) -> torch.Tensor:
    """out [T, N] = sum_j weights[t, j] * y_sorted[pos[t*k + j]] (weights fp32 [T, k])."""
    T, k = weights.shape
    N = y_sorted.shape[1]
    dt = y_sorted.dtype
    if out is None:
        out = torch.empty((T, N), dtype=dt, device=y_sorted.device)
    _check(lib.w4a16_moe_sum(_dev(y_sorted, dt, "y_sorted"), _dev(pos, torch.int32, "pos"),
                             _dev(weights, torch.float32, "weights"), T, k, N, _DTYPE_OF[dt],
                             _dev(out, dt, "out"), _stream_ptr(stream)),
           "w4a16_moe_sum")
    return out


def make_descs(layers) -> ctypes.Array:
    """layers: iterable of dicts with x, qweight, scales, zeros, y tensors (and
    optionally an epilogue code and a residual tensor) -> host desc array.
    A y may be a pinned host tensor (never another layer's x or residual:
    those must be CUDA tensors)."""
    layers = list(layers)
    arr = (LinearDesc * len(layers))()
    for i, L in enumerate(layers):
        N, K = L["qweight"].shape[0], L["x"].shape[1]
        res = L.get("residual")
        dt = L["x"].dtype
        if dt not in _DTYPE_OF:
            raise TypeError(f"x must be float16 or bfloat16, got {dt}")
        arr[i] = LinearDesc(_dev(L["x"], dt, "x"), _dev(L["qweight"], torch.int32, "qweight"),
                            _dev(L["scales"], dt, "scales"),
                            _dev(L["zeros"], torch.int32, "zeros"), _dev(L["y"], dt, "y", True),
                            N, K, L.get("group", GROUP), L.get("epilogue", EPILOGUE_NONE),
                            _dev(res, dt, "residual") if res is not None else None,
                            _DTYPE_OF[dt])
    return arr


def w4a16_decode_round(descs, M: int, stream=None) -> None:
    _check(lib.w4a16_decode_round(descs, len(descs), M, _stream_ptr(stream)), "w4a16_decode_round")


class RoundGraph:
    """A decode round captured once into a CUDA graph and replayed."""

    def __init__(self, descs, M: int):
        self._descs = descs  # keep the host array alive for the graph's lifetime
        h = _P()
        _check(lib.w4a16_round_graph_create(descs, len(descs), M, ctypes.byref(h)),
               "w4a16_round_graph_create")
        self.handle = h.value

    def launch(self, stream=None) -> None:
        _check(lib.w4a16_round_graph_launch(self.handle, _stream_ptr(stream)),
               "w4a16_round_graph_launch")

    def destroy(self) -> None:
        if self.handle:
            _check(lib.w4a16_round_graph_destroy(self.handle), "w4a16_round_graph_destroy")
            self.handle = None


def w4a16_select_rung(M: int, N: int, K: int, group: int = GROUP) -> int:
    return int(lib.w4a16_select_rung(M, N, K, group))


def w4a16_plan_info(M: int, N: int, K: int, group: int = GROUP, epilogue: int = 0,
                    dtype: int = 0) -> dict:
    """The plan of a linear's first tile: rung, threads per CTA, K slices, CTAs."""
    info = (ctypes.c_int32 * 4)()
    _check(lib.w4a16_plan_info(M, N, K, group, epilogue, dtype, info), "w4a16_plan_info")
    return {"rung": info[0], "threads": info[1], "k_slices": info[2], "grid": info[3]}


def w4a16_set_forced_rung(rung: int) -> int:
    prev = int(lib.w4a16_set_forced_rung(rung))
    if prev == -2:
        raise ValueError(f"invalid rung {rung}")
    return prev


def w4a16_probe_counts() -> list[int]:
    buf = (ctypes.c_uint64 * NUM_RUNGS)()
    n = lib.w4a16_probe_counts(buf, NUM_RUNGS)
    return [int(buf[i]) for i in range(n)]


def w4a16_probe_reset() -> None:
    lib.w4a16_probe_reset()


def w4a16_kernel_launches() -> int:
    return int(lib.w4a16_kernel_launches())


def w4a16_device_status(stream=None) -> int:
    """Synchronise `stream`; return (and clear) the device error code (0 = none)."""
    code = _I(0)
    st = lib.w4a16_device_status(_stream_ptr(stream), ctypes.byref(code))
    if st not in (W4A16_OK, W4A16_ERR_DEVICE):
        _check(st, "w4a16_device_status")
    return int(code.value)


def w4a16_wait_probe(stream=None):
    """Run the library's bounded waits on a counter and an mbarrier that nothing
    completes; each expires (200 ms) and sets its bit in the device status
    word (4096, 8192)."""
    _check(lib.w4a16_wait_probe(_stream_ptr(stream)), "w4a16_wait_probe")


def w4a16_device_sm_count() -> int:
    return int(lib.w4a16_device_sm_count())
