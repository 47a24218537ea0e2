"""Host-side checks of the C ABI (no GPU needed, no device work).

The library must load, export every function ``include/w4a16.h`` declares,
and reject bad arguments on the host, before any CUDA call, with the status
codes the header documents.
"""
import ctypes
import os
import re

import pytest

import __graft_entry__

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def w4():
    __graft_entry__.build()
    import weight_only_int4_w4a16_gb300 as w4
    return w4


def header_functions():
    text = open(os.path.join(ROOT, "include", "w4a16.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(w4a16_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(w4):
    names = header_functions()
    assert len(names) >= 19
    for n in names:
        assert hasattr(w4.lib, n), f"{n} declared in include/w4a16.h but not exported"
    assert set(names) == set(w4.binding.EXPORTED)


def test_status_and_rung_strings(w4):
    assert w4.lib.w4a16_status_string(0) == b"ok"
    assert w4.lib.w4a16_status_string(99) == b"?"
    assert [w4.rung_name(i) for i in range(6)] == ["gemv", "gemv_splitk", "tc", "tc_splitk",
                                                   "mma", "mma_splitk"]
    assert w4.rung_name(-1) == "auto" and w4.rung_name(9) == "?"


A = 1 << 20  # a fake, 16-byte aligned "device address": never dereferenced on these paths


def _lin(w4, x=A, qw=2 * A, s=3 * A, z=4 * A, M=1, N=64, K=256, group=128, y=5 * A):
    return w4.lib.w4a16_linear(x, qw, s, z, M, N, K, group, y, None)


def test_linear_validation_codes(w4):
    assert _lin(w4, x=None) == w4.W4A16_ERR_INVALID_ARG
    assert _lin(w4, y=None) == w4.W4A16_ERR_INVALID_ARG
    assert _lin(w4, M=0) == w4.W4A16_ERR_INVALID_ARG
    assert _lin(w4, M=70000) == w4.W4A16_ERR_INVALID_ARG
    assert _lin(w4, N=0) == w4.W4A16_ERR_INVALID_ARG
    assert _lin(w4, K=200) == w4.W4A16_ERR_INVALID_ARG
    assert _lin(w4, group=64) == w4.W4A16_ERR_UNSUPPORTED
    assert _lin(w4, x=A + 8) == w4.W4A16_ERR_MISALIGNED
    assert _lin(w4, qw=2 * A + 4) == w4.W4A16_ERR_MISALIGNED
    assert _lin(w4, s=3 * A + 1) == w4.W4A16_ERR_MISALIGNED
    assert _lin(w4, z=4 * A + 2) == w4.W4A16_ERR_MISALIGNED
    # x and y overlapping
    assert _lin(w4, y=A + 64) == w4.W4A16_ERR_INVALID_ARG
    # valid arguments, but no successful w4a16_init in this process
    if w4.lib.w4a16_device_sm_count() == 0:
        assert _lin(w4) == w4.W4A16_ERR_NOT_INITIALIZED


def _epi(w4, epi, res=None, M=1, N=64, K=256, y=5 * A, group=128):
    return w4.lib.w4a16_linear_epilogue(A, 2 * A, 3 * A, 4 * A, M, N, K, group, epi, res, y, None)


def test_linear_epilogue_validation_codes(w4):
    R, S = w4.EPILOGUE_RESIDUAL, w4.EPILOGUE_SILU_MUL
    assert _epi(w4, 3) == w4.W4A16_ERR_INVALID_ARG           # no such epilogue
    assert _epi(w4, -1) == w4.W4A16_ERR_INVALID_ARG
    assert _epi(w4, R) == w4.W4A16_ERR_INVALID_ARG           # residual epilogue without one
    assert _epi(w4, 0, res=6 * A) == w4.W4A16_ERR_INVALID_ARG  # a residual nobody adds
    assert _epi(w4, S, res=6 * A) == w4.W4A16_ERR_INVALID_ARG
    assert _epi(w4, S, N=48) == w4.W4A16_ERR_UNSUPPORTED     # N/2 not a multiple of 16
    assert _epi(w4, R, res=6 * A + 1) == w4.W4A16_ERR_MISALIGNED
    # the residual partly over y (y itself is allowed)
    assert _epi(w4, R, res=5 * A + 2) == w4.W4A16_ERR_INVALID_ARG
    # y of SiLU-and-mul is [M, N/2]: 64 bytes just below x do not overlap it,
    # the 128 bytes of a plain y do
    assert _epi(w4, S, y=A - 64) == _epi(w4, S, y=5 * A)
    assert _epi(w4, 0, y=A - 64) == w4.W4A16_ERR_INVALID_ARG
    if w4.lib.w4a16_device_sm_count() == 0:
        assert _epi(w4, R, res=5 * A) == w4.W4A16_ERR_NOT_INITIALIZED  # in place
        assert _epi(w4, R, res=6 * A) == w4.W4A16_ERR_NOT_INITIALIZED
        assert _epi(w4, S) == w4.W4A16_ERR_NOT_INITIALIZED
        assert _epi(w4, 0) == w4.W4A16_ERR_NOT_INITIALIZED


def test_linear_ex_validation_codes(w4):
    L = w4.lib
    args = (A, 2 * A, 3 * A, 4 * A, 1, 64, 256, 128)
    assert L.w4a16_linear_ex(*args, 2, 0, None, 5 * A, None) == w4.W4A16_ERR_INVALID_ARG
    assert L.w4a16_linear_ex(*args, -1, 0, None, 5 * A, None) == w4.W4A16_ERR_INVALID_ARG
    assert L.w4a16_linear_ex(*args, 1, 3, None, 5 * A, None) == w4.W4A16_ERR_INVALID_ARG
    assert L.w4a16_linear_ex(*args, 1, 1, None, 5 * A, None) == w4.W4A16_ERR_INVALID_ARG
    if w4.lib.w4a16_device_sm_count() == 0:
        assert L.w4a16_linear_ex(*args, 1, 0, None, 5 * A, None) == w4.W4A16_ERR_NOT_INITIALIZED
        assert L.w4a16_linear_ex(*args, 1, 1, 6 * A, 5 * A, None) == w4.W4A16_ERR_NOT_INITIALIZED


def test_dense_linear_validation_codes(w4):
    L = w4.lib
    assert L.w4a16_dense_linear(None, 2 * A, 1, 64, 256, 0, 5 * A, None) == w4.W4A16_ERR_INVALID_ARG
    assert L.w4a16_dense_linear(A, 2 * A, 0, 64, 256, 0, 5 * A, None) == w4.W4A16_ERR_INVALID_ARG
    assert L.w4a16_dense_linear(A, 2 * A, 1, 64, 200, 0, 5 * A, None) == w4.W4A16_ERR_INVALID_ARG
    assert L.w4a16_dense_linear(A, 2 * A, 1, 64, 256, 2, 5 * A, None) == w4.W4A16_ERR_INVALID_ARG
    assert L.w4a16_dense_linear(A + 8, 2 * A, 1, 64, 256, 0, 5 * A, None) == w4.W4A16_ERR_MISALIGNED
    assert L.w4a16_dense_linear(A, 2 * A, 1, 64, 256, 0, 2 * A + 64, None) == w4.W4A16_ERR_INVALID_ARG
    if w4.lib.w4a16_device_sm_count() == 0:
        assert L.w4a16_dense_linear(A, 2 * A, 1, 64, 256, 1, 5 * A, None) == w4.W4A16_ERR_NOT_INITIALIZED


def test_moe_validation_codes(w4):
    L = w4.lib
    assert L.w4a16_moe_align(None, 8, 4, A, 2 * A, 3 * A, None) == w4.W4A16_ERR_INVALID_ARG
    assert L.w4a16_moe_align(A, 8, 0, A, 2 * A, 3 * A, None) == w4.W4A16_ERR_INVALID_ARG
    assert L.w4a16_moe_align(A, 8, 2000, A, 2 * A, 3 * A, None) == w4.W4A16_ERR_INVALID_ARG
    assert L.w4a16_moe_align(A + 2, 8, 4, A, 2 * A, 3 * A, None) == w4.W4A16_ERR_MISALIGNED
    h = ctypes.c_void_p()
    assert L.w4a16_moe_create(0, 64, 256, 128, A, 2 * A, 3 * A, 0, 0, 8,
                              ctypes.byref(h)) == w4.W4A16_ERR_INVALID_ARG
    assert L.w4a16_moe_create(4, 64, 256, 128, A, 2 * A, 3 * A, 1, 0, 8,
                              ctypes.byref(h)) == w4.W4A16_ERR_UNSUPPORTED  # residual
    assert L.w4a16_moe_create(4, 48, 256, 128, A, 2 * A, 3 * A, 2, 0, 8,
                              ctypes.byref(h)) == w4.W4A16_ERR_UNSUPPORTED  # N/2 % 16
    assert L.w4a16_moe_create(4, 64, 256, 64, A, 2 * A, 3 * A, 0, 0, 8,
                              ctypes.byref(h)) == w4.W4A16_ERR_UNSUPPORTED  # group
    assert L.w4a16_moe_linear(None, A, 1, A, A, 8, A, None) == w4.W4A16_ERR_INVALID_ARG
    assert L.w4a16_moe_destroy(None) == w4.W4A16_ERR_INVALID_ARG
    assert L.w4a16_moe_sum(A, 2 * A, 3 * A, 0, 2, 8, 0, 4 * A, None) == w4.W4A16_ERR_INVALID_ARG
    assert L.w4a16_moe_sum(A, 2 * A, 3 * A, 2, 2, 8, 5, 4 * A, None) == w4.W4A16_ERR_INVALID_ARG
    assert L.w4a16_moe_sum(A, 2 * A, 3 * A, 2, 2, 8, 0, A + 8, None) == w4.W4A16_ERR_INVALID_ARG
    p = ctypes.c_int()
    assert L.w4a16_moe_mlp_set_path(None, 0) == w4.W4A16_ERR_INVALID_ARG
    assert L.w4a16_moe_mlp_path(None, 1, ctypes.byref(p)) == w4.W4A16_ERR_INVALID_ARG
    assert (w4.MOE_PATH_AUTO, w4.MOE_PATH_CHAIN, w4.MOE_PATH_DECODE) == (0, 1, 2)
    if w4.lib.w4a16_device_sm_count() == 0:
        assert L.w4a16_moe_align(A, 8, 4, A, 2 * A, 3 * A, None) == w4.W4A16_ERR_NOT_INITIALIZED
        assert L.w4a16_moe_create(4, 64, 256, 128, A, 2 * A, 3 * A, 2, 1, 8,
                                  ctypes.byref(h)) == w4.W4A16_ERR_NOT_INITIALIZED


def test_repack_validation_codes(w4):
    L, seq = w4.lib, 0x76543210
    assert L.w4a16_repack_transpose(None, 8, 8, seq, A, None) == w4.W4A16_ERR_INVALID_ARG
    assert L.w4a16_repack_transpose(A, 0, 8, seq, 2 * A, None) == w4.W4A16_ERR_INVALID_ARG
    assert L.w4a16_repack_transpose(A, 8, 12, seq, 2 * A, None) == w4.W4A16_ERR_INVALID_ARG
    assert L.w4a16_repack_transpose(A, 8, 8, 0x76543211, 2 * A, None) == w4.W4A16_ERR_INVALID_ARG
    assert L.w4a16_repack_transpose(A, 8, 8, 0x86543210, 2 * A, None) == w4.W4A16_ERR_INVALID_ARG
    assert L.w4a16_repack_transpose(A + 2, 8, 8, seq, 2 * A, None) == w4.W4A16_ERR_MISALIGNED
    assert L.w4a16_repack_transpose(A, 64, 64, seq, A + 64, None) == w4.W4A16_ERR_INVALID_ARG
    assert L.w4a16_transpose_f16(A, 0, 4, 2 * A, None) == w4.W4A16_ERR_INVALID_ARG
    assert L.w4a16_transpose_f16(A + 1, 4, 4, 2 * A, None) == w4.W4A16_ERR_MISALIGNED
    assert L.w4a16_transpose_f16(A, 4, 4, A + 8, None) == w4.W4A16_ERR_INVALID_ARG


def test_pack_dequant_validation_codes(w4):
    L = w4.lib
    assert L.w4a16_pack(None, A, 4, 256, 128, A, A, None) == w4.W4A16_ERR_INVALID_ARG
    assert L.w4a16_pack(A, A, 4, 256, 32, A, A, None) == w4.W4A16_ERR_UNSUPPORTED
    assert L.w4a16_pack(A + 4, A, 4, 256, 128, A, A, None) == w4.W4A16_ERR_MISALIGNED
    assert L.w4a16_unpack(A, A, 4, 100, 128, A, A, None) == w4.W4A16_ERR_INVALID_ARG
    assert L.w4a16_dequant(A, A, A, 4, 256, 128, None, None, None) == w4.W4A16_ERR_INVALID_ARG
    assert L.w4a16_dequant(A, A, A, 4, 256, 128, A + 4, None, None) == w4.W4A16_ERR_MISALIGNED


def test_decode_round_validates_every_descriptor(w4):
    descs = (w4.LinearDesc * 2)()
    descs[0] = w4.LinearDesc(A, 2 * A, 3 * A, 4 * A, 5 * A, 64, 256, 128)
    descs[1] = w4.LinearDesc(A, 2 * A, 3 * A, 4 * A, 5 * A, 64, 250, 128)  # bad K
    assert w4.lib.w4a16_decode_round(descs, 2, 4, None) == w4.W4A16_ERR_INVALID_ARG
    descs[1] = w4.LinearDesc(A, 2 * A, 3 * A, 4 * A, 5 * A, 64, 256, 128, w4.EPILOGUE_RESIDUAL,
                             None)  # residual epilogue without a residual
    assert w4.lib.w4a16_decode_round(descs, 2, 4, None) == w4.W4A16_ERR_INVALID_ARG
    descs[1] = w4.LinearDesc(A, 2 * A, 3 * A, 4 * A, 5 * A, 48, 256, 128, w4.EPILOGUE_SILU_MUL,
                             None)  # N/2 not a multiple of 16
    assert w4.lib.w4a16_decode_round(descs, 2, 4, None) == w4.W4A16_ERR_UNSUPPORTED
    assert w4.lib.w4a16_decode_round(descs, 0, 4, None) == w4.W4A16_ERR_INVALID_ARG
    h = ctypes.c_void_p()
    assert w4.lib.w4a16_round_graph_create(descs, 2, 4, None) == w4.W4A16_ERR_INVALID_ARG
    assert w4.lib.w4a16_round_graph_launch(None, None) == w4.W4A16_ERR_INVALID_ARG
    del h


def test_dispatch_table_host_queries(w4):
    # Pure host queries: the table picks a rung for every valid shape and
    # rejects invalid ones.
    assert 0 <= w4.w4a16_select_rung(1, 34816, 5120) < w4.NUM_RUNGS
    assert w4.w4a16_select_rung(16, 27648, 5120) in (w4.RUNG_TC, w4.RUNG_TC_SPLITK)
    assert w4.w4a16_select_rung(1, 1024, 500) == -1
    assert w4.w4a16_select_rung(0, 1024, 512) == -1
    # small fp16 linears launched alone take the CUDA-core gemv kernel: up to
    # 24 Mi weights at 1..2 tokens, 16 Mi at 3..4, 8 Mi at 5..8 (K split
    # where one warp cannot hold the whole K); larger ones the warp-MMA kernel
    gemv = (w4.RUNG_GEMV, w4.RUNG_GEMV_SPLITK)
    mma = (w4.RUNG_MMA, w4.RUNG_MMA_SPLITK)
    assert w4.w4a16_select_rung(1, 1024, 512) == w4.RUNG_GEMV
    assert w4.w4a16_select_rung(2, 6144, 4096) in gemv
    assert w4.w4a16_select_rung(2, 8192, 4096) in mma
    assert w4.w4a16_select_rung(4, 4096, 4096) in gemv
    assert w4.w4a16_select_rung(4, 6144, 4096) in mma
    assert w4.w4a16_select_rung(8, 512, 16384) in gemv
    assert w4.w4a16_select_rung(8, 4096, 4096) in mma
    assert w4.w4a16_select_rung(1, 34816, 5120) in mma
    # epilogues and bf16 stay on the MMA kernels
    assert w4.w4a16_plan_info(1, 1024, 512, epilogue=w4.EPILOGUE_RESIDUAL)["rung"] in mma
    assert w4.w4a16_plan_info(1, 1024, 512, dtype=w4.DTYPE_BF16)["rung"] in mma
    prev = w4.w4a16_set_forced_rung(w4.RUNG_GEMV_SPLITK)
    try:
        assert w4.w4a16_select_rung(4, 5120, 17408) == w4.RUNG_GEMV_SPLITK
        assert w4.w4a16_workspace_bytes(4, 5120, 17408) >= 2 * 4 * 5120 * 4
    finally:
        w4.w4a16_set_forced_rung(prev)
    with pytest.raises(ValueError):
        w4.w4a16_set_forced_rung(9)


def test_plan_info_names_the_cta_shape(w4):
    # Pure host queries (152 SMs assumed before init).  Up to 4 tokens the
    # warp-MMA kernel runs 8-warp CTAs; at 8 tokens a K 5120 linear's x only
    # fits a 16-warp CTA (one per SM), which keeps K whole; K 17408 splits
    # either way and stays on 8 warps.
    assert w4.w4a16_set_forced_rung(w4.RUNG_AUTO) == w4.RUNG_AUTO
    p = w4.w4a16_plan_info(4, 27648, 5120)
    assert p["rung"] == w4.RUNG_MMA and p["threads"] == 256 and p["k_slices"] == 1
    p = w4.w4a16_plan_info(8, 27648, 5120)
    assert p["rung"] == w4.RUNG_MMA and p["threads"] == 512 and p["k_slices"] == 1
    assert p["grid"] <= 152
    p = w4.w4a16_plan_info(8, 5120, 17408)
    assert p["rung"] == w4.RUNG_MMA_SPLITK and p["threads"] == 256 and p["k_slices"] > 1
    p = w4.w4a16_plan_info(8, 34816, 5120, epilogue=w4.EPILOGUE_SILU_MUL)
    assert p["threads"] == 512
    p = w4.w4a16_plan_info(16, 27648, 5120)
    assert p["rung"] in (w4.RUNG_TC, w4.RUNG_TC_SPLITK) and p["threads"] == 800
    with pytest.raises(w4.W4A16Error):
        w4.w4a16_plan_info(4, 1024, 500)
    with pytest.raises(w4.W4A16Error):
        w4.w4a16_plan_info(4, 1000, 512, epilogue=w4.EPILOGUE_SILU_MUL)  # N/2 not a multiple of 16


def test_tc_plan_keeps_short_single_wave_tiles_whole(w4):
    # From 17 tokens on, a single wave of tiles with fewer than 12 stages
    # stays whole (the pieces' partial sums cost more than idle SMs); long
    # tiles, and shapes of more than one wave, are split (stream-K)
    assert w4.w4a16_set_forced_rung(w4.RUNG_AUTO) == w4.RUNG_AUTO
    assert w4.w4a16_plan_info(24, 8192, 4096)["rung"] == w4.RUNG_TC          # 64 tiles, 8 stages
    assert w4.w4a16_plan_info(64, 2048, 5120)["rung"] == w4.RUNG_TC          # 16 tiles, 10 stages
    assert w4.w4a16_plan_info(24, 1024, 8192)["rung"] == w4.RUNG_TC_SPLITK   # 16 stages a tile
    assert w4.w4a16_plan_info(32, 27648, 5120)["rung"] == w4.RUNG_TC_SPLITK  # 216 tiles
    assert w4.w4a16_plan_info(16, 8192, 4096)["rung"] == w4.RUNG_TC_SPLITK   # 16 tokens: split


def test_probe_counters_reset(w4):
    w4.w4a16_probe_reset()
    assert w4.w4a16_probe_counts() == [0] * 6


def test_binding_output_may_be_pinned_host_memory_inputs_may_not(w4):
    # Only an output may live in (page-locked) host memory; the check runs in
    # the binding before the library is called.  Here nothing is pinned (no
    # GPU), so every CPU tensor is refused, and the message names the rule.
    import torch
    x = torch.zeros((1, 256), dtype=torch.float16)
    qw = torch.zeros((64, 32), dtype=torch.int32)
    s = torch.zeros((64, 2), dtype=torch.float16)
    z = torch.zeros((64, 1), dtype=torch.int32)
    y = torch.zeros((1, 64), dtype=torch.float16)
    with pytest.raises(ValueError, match="page-locked host memory"):
        w4.binding._dev(y, torch.float16, "y", True)
    with pytest.raises(ValueError, match="must live on a CUDA device$"):
        w4.binding._dev(x, torch.float16, "x")
    with pytest.raises(ValueError, match="x must live on a CUDA device$"):
        w4.w4a16_linear(x, qw, s, z, y=y)
    with pytest.raises(ValueError, match="x must live on a CUDA device$"):
        w4.make_descs([dict(x=x, qweight=qw, scales=s, zeros=z, y=y)])
