"""The fused epilogues and bf16 layers on the tcgen05 rung (more than 8 tokens).

A layer of more than 8 tokens runs on the tcgen05 rung, which reads the
weights once for up to 64 tokens.  That holds for a residual add (the output
projections: haowenji.com V100 decode article, the add-back merged into the
matmul's output stage), for SiLU-and-mul after a fused gate+up projection
(forum.sourcefind.cn thread "vLLM on Hygon Z100", section 二), and for bf16
activations and scales (the same thread: activations "fp16 or bf16").  The
rung restores each weight to the layer's 16-bit type ((q - z) * s rounded
once) and accumulates the tensor-core products in fp32.  A SiLU-and-mul tile
holds 64 gate rows and their up rows N/2 below.  The probe counters show which
rung computed the layer; every output is compared with the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic_inputs as si
from helpers import RTOL_BF16_TC, assert_close

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def w4():
    import __graft_entry__
    __graft_entry__.build()
    import weight_only_int4_w4a16_gb300 as w4
    if w4.w4a16_device_sm_count() == 0:
        w4.w4a16_init(0, 256 << 20)
    yield w4
    w4.w4a16_set_forced_rung(w4.RUNG_AUTO)


@pytest.fixture(autouse=True)
def no_device_errors(request):
    yield
    if "w4" in request.fixturenames:
        import weight_only_int4_w4a16_gb300 as w4
        assert w4.w4a16_device_status() == 0, "a kernel reported an expired bounded wait"


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _case(seed, M, N, K, dt):
    qw, s, zw = si.layer(seed, N, K)
    x = si.x(seed, M, K).float().to(dt)
    if dt == torch.bfloat16:
        s = s.float().to(dt)
    return x, qw, s, zw


def _reference(x, qw, s, zw, dt, residual=None):
    name = "bf16" if dt == torch.bfloat16 else "f16"
    h = oracle.linear(_bits(x), si.as_u32(qw), _bits(s), si.as_u32(zw), dtype=name)
    return h if residual is None else oracle.add_residual(h, _bits(residual), name)


def _rtol(dt):
    # bf16 on this rung: each weight is restored to bf16 once
    return RTOL_BF16_TC if dt == torch.bfloat16 else None


def _tc_count(w4):
    c = w4.w4a16_probe_counts()
    return c[w4.RUNG_TC] + c[w4.RUNG_TC_SPLITK], sum(c)


# token counts past the warp-MMA rungs (one tcgen05 tile of 16, 32, 64 tokens,
# and two tiles at 100), ragged N, K from a few groups to the down projection's
SHAPES = [(9, 300, 1024), (16, 1024, 2048), (33, 777, 1408), (64, 5120, 6144),
          (100, 640, 17408)]


@pytest.mark.parametrize("dt", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_residual_on_the_tc_rung(w4, dt, M, N, K):
    seed = si.config_seed(87, M, N % 16)
    x, qw, s, zw = _case(seed, M, N, K, dt)
    r = si.residual(seed, M, N).float().to(dt)
    y = torch.full((M, N), float("nan"), dtype=dt, device=DEV)
    w4.w4a16_probe_reset()
    w4.w4a16_linear_ex(x.to(DEV), qw.to(DEV), s.to(DEV), zw.to(DEV),
                       epilogue=w4.EPILOGUE_RESIDUAL, residual=r.to(DEV), y=y)
    torch.cuda.synchronize()
    tc, total = _tc_count(w4)
    assert tc == total == (M + 63) // 64, "the layer ran on another rung"
    assert_close(y, _reference(x, qw, s, zw, dt, r), f"residual {dt} M={M} N={N} K={K}",
                 rtol=_rtol(dt))
    # in place: the residual is y itself (y += x W^T)
    y2 = r.to(DEV).clone()
    w4.w4a16_linear_ex(x.to(DEV), qw.to(DEV), s.to(DEV), zw.to(DEV),
                       epilogue=w4.EPILOGUE_RESIDUAL, residual=y2, y=y2)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(y2.cpu()), _bits(y.cpu()))


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_bf16_on_the_tc_rung(w4, M, N, K):
    dt = torch.bfloat16
    seed = si.config_seed(88, M, N % 16)
    x, qw, s, zw = _case(seed, M, N, K, dt)
    w4.w4a16_probe_reset()
    y = w4.w4a16_linear_ex(x.to(DEV), qw.to(DEV), s.to(DEV), zw.to(DEV))
    torch.cuda.synchronize()
    tc, total = _tc_count(w4)
    assert tc == total == (M + 63) // 64
    assert_close(y, _reference(x, qw, s, zw, dt), f"bf16 M={M} N={N} K={K}", rtol=_rtol(dt))


# SiLU-and-mul tiles: 64 outputs each (N/2 a multiple of 16; ragged last
# tile), the fused gate+up shape of the 27B decode layer, tiles of 64 tokens
SILU_SHAPES = [(9, 320, 1024), (16, 2048, 2048), (33, 1056, 1408), (64, 34816, 5120),
               (100, 640, 6144)]


@pytest.mark.parametrize("dt", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("M,N,K", SILU_SHAPES)
def test_silu_mul_on_the_tc_rung(w4, dt, M, N, K):
    seed = si.config_seed(91, M, N % 16)
    x, qw, s, zw = _case(seed, M, N, K, dt)
    y = torch.full((M, N // 2), float("nan"), dtype=dt, device=DEV)
    w4.w4a16_probe_reset()
    w4.w4a16_linear_ex(x.to(DEV), qw.to(DEV), s.to(DEV), zw.to(DEV),
                       epilogue=w4.EPILOGUE_SILU_MUL, y=y)
    torch.cuda.synchronize()
    tc, total = _tc_count(w4)
    assert tc == total == (M + 63) // 64, "the layer ran on another rung"
    ref = oracle.silu_mul(_reference(x, qw, s, zw, dt))
    assert_close(y, ref, f"silu_mul {dt} M={M} N={N} K={K}", rtol=_rtol(dt))


@pytest.mark.parametrize("rung", [2, 3])
@pytest.mark.parametrize("dt", [torch.float16, torch.bfloat16])
def test_forced_tc_rungs_with_epilogue_and_bf16(w4, rung, dt):
    # whole tiles (tc) and stream-K (tc_splitk), from 4 tokens up
    for M, N, K in [(4, 1024, 2048), (24, 320, 5120)]:
        seed = si.config_seed(89, M, rung)
        x, qw, s, zw = _case(seed, M, N, K, dt)
        r = si.residual(seed, M, N).float().to(dt)
        prev = w4.w4a16_set_forced_rung(rung)
        try:
            w4.w4a16_probe_reset()
            y = w4.w4a16_linear_ex(x.to(DEV), qw.to(DEV), s.to(DEV), zw.to(DEV),
                                   epilogue=w4.EPILOGUE_RESIDUAL, residual=r.to(DEV))
            torch.cuda.synchronize()
            assert w4.w4a16_probe_counts()[rung] >= 1
            ys = w4.w4a16_linear_ex(x.to(DEV), qw.to(DEV), s.to(DEV), zw.to(DEV),
                                    epilogue=w4.EPILOGUE_SILU_MUL)
            torch.cuda.synchronize()
        finally:
            w4.w4a16_set_forced_rung(prev)
        assert_close(y, _reference(x, qw, s, zw, dt, r), f"forced rung {rung} {dt} M={M}",
                     rtol=_rtol(dt))
        assert_close(ys, oracle.silu_mul(_reference(x, qw, s, zw, dt)),
                     f"forced rung {rung} {dt} M={M} SiLU-and-mul", rtol=_rtol(dt))


def test_large_scales_with_residual_on_the_tc_rung(w4):
    # scales that the fp16 restore cannot hold ((q - z) * 65504 overflows):
    # those rows are recomputed exactly on the CUDA cores, residual included
    M, N, K = 16, 320, 1024
    rng = np.random.default_rng(90)
    seed = si.config_seed(90)
    qw, s, zw = si.layer(seed, N, K)
    v = s.double().numpy().copy()
    for row in range(0, N, 37):
        v[row, int(rng.integers(0, K // 128))] = 65504.0 if row % 2 == 0 else -65504.0
    s = torch.from_numpy(v.astype(np.float16))
    x = (si.x(seed, M, K).double() / 1024.0).to(torch.float16)
    r = si.residual(seed, M, N)
    w4.w4a16_probe_reset()
    y = w4.w4a16_linear_ex(x.to(DEV), qw.to(DEV), s.to(DEV), zw.to(DEV),
                           epilogue=w4.EPILOGUE_RESIDUAL, residual=r.to(DEV))
    torch.cuda.synchronize()
    assert _tc_count(w4)[0] == 1
    ref = _reference(x, qw, s, zw, torch.float16, r)
    assert np.isfinite(ref).all() and np.abs(ref).max() < 60000
    assert_close(y, ref, "large scales with the residual")
    # and through SiLU-and-mul (the exact rows' sums meet their partner rows)
    x2 = (x.double() / 64.0).to(torch.float16)
    ys = w4.w4a16_linear_ex(x2.to(DEV), qw.to(DEV), s.to(DEV), zw.to(DEV),
                            epilogue=w4.EPILOGUE_SILU_MUL)
    torch.cuda.synchronize()
    refs = oracle.silu_mul(_reference(x2, qw, s, zw, torch.float16))
    assert np.isfinite(refs).all() and np.abs(refs).max() < 60000
    assert_close(ys, refs, "large scales with SiLU-and-mul")
