"""The warp-MMA kernel on 16-warp CTAs (one per SM).

From 5 tokens on, the activations of a K 5120 slice no longer fit beside an
8-warp CTA's weight rings, and two such CTAs share an SM; a 16-warp CTA has
the SM's whole shared memory and keeps K whole (the method is unchanged:
forum.sourcefind.cn thread "vLLM on Hygon Z100", sections 四 and 五, weights
streamed once for all M rows).  Every case below first checks, with
w4a16_plan_info, that the shape takes the 16-warp CTA, then compares every
output with the oracle: plain linears (K whole and split), the residual and
SiLU-and-mul epilogues, bf16, the forced warp-MMA rungs, the allocation-free
entry point, and a fused round whose linears wait on each other.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic_inputs as si
from helpers import assert_close

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
WIDE = 512  # threads of a 16-warp CTA


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


def _case(seed, M, N, K, dt=torch.float16):
    qw, s, zw = si.layer(seed, N, K)
    x = si.x(seed, M, K).float().to(dt)
    if dt == torch.bfloat16:
        s = s.float().to(dt)
    return x, qw, s, zw


def _ref(x, qw, s, zw, dt=torch.float16):
    name = "bf16" if dt == torch.bfloat16 else "f16"
    return oracle.linear(_bits(x), si.as_u32(qw), _bits(s), si.as_u32(zw), dtype=name)


# K whole (k_slices 1) and split for balance (small N): both on 16 warps
# (above 8 Mi weights: smaller linears at 5..8 tokens go to the gemv rung)
SHAPES = [(5, 3000, 4608), (6, 1800, 5120), (7, 4096, 4096), (8, 2048, 5120), (8, 1900, 4608)]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_wide_linear_full_output(w4, M, N, K):
    assert w4.w4a16_plan_info(M, N, K)["threads"] == WIDE
    seed = si.config_seed(95, M, K // 128)
    x, qw, s, zw = _case(seed, M, N, K)
    y = torch.full((M, N), float("nan"), dtype=torch.float16, device=DEV)
    w4.w4a16_linear(x.to(DEV), qw.to(DEV), s.to(DEV), zw.to(DEV), y=y)
    torch.cuda.synchronize()
    assert_close(y, _ref(x, qw, s, zw), f"16-warp CTA M={M} N={N} K={K}")
    # run to run: the same bits (the split-K sums in slice order)
    y2 = w4.w4a16_linear(x.to(DEV), qw.to(DEV), s.to(DEV), zw.to(DEV))
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))


@pytest.mark.parametrize("dt", [torch.float16, torch.bfloat16])
def test_wide_epilogues(w4, dt):
    dtype = w4.DTYPE_BF16 if dt == torch.bfloat16 else w4.DTYPE_F16
    # residual add, out of place and in place
    M, N, K = 8, 2048, 5120
    assert w4.w4a16_plan_info(M, N, K, epilogue=w4.EPILOGUE_RESIDUAL, dtype=dtype)["threads"] == WIDE
    seed = si.config_seed(96, 1)
    x, qw, s, zw = _case(seed, M, N, K, dt)
    r = si.residual(seed, M, N).float().to(dt)
    name = "bf16" if dt == torch.bfloat16 else "f16"
    ref = oracle.add_residual(_ref(x, qw, s, zw, dt), _bits(r), name)
    y = w4.w4a16_linear_ex(x.to(DEV), qw.to(DEV), s.to(DEV), zw.to(DEV),
                           epilogue=w4.EPILOGUE_RESIDUAL, residual=r.to(DEV))
    yi = r.to(DEV).clone()
    w4.w4a16_linear_ex(x.to(DEV), qw.to(DEV), s.to(DEV), zw.to(DEV),
                       epilogue=w4.EPILOGUE_RESIDUAL, residual=yi, y=yi)
    torch.cuda.synchronize()
    rtol = 2.0 ** -8 if dt == torch.bfloat16 else None
    assert_close(y, ref, f"16-warp residual {dt}", rtol=rtol)
    assert torch.equal(y.view(torch.int16), yi.view(torch.int16))
    # SiLU-and-mul over the fused gate+up rows
    M, N, K = 6, 4096, 5120
    assert w4.w4a16_plan_info(M, N, K, epilogue=w4.EPILOGUE_SILU_MUL, dtype=dtype)["threads"] == WIDE
    seed = si.config_seed(96, 2)
    x, qw, s, zw = _case(seed, M, N, K, dt)
    y = w4.w4a16_linear_ex(x.to(DEV), qw.to(DEV), s.to(DEV), zw.to(DEV),
                           epilogue=w4.EPILOGUE_SILU_MUL)
    torch.cuda.synchronize()
    assert_close(y, oracle.silu_mul(_ref(x, qw, s, zw, dt)), f"16-warp SiLU-and-mul {dt}",
                 rtol=rtol)


@pytest.mark.parametrize("rung", [4, 5])  # mma, mma_splitk
def test_wide_forced_rungs(w4, rung):
    M, N, K = 8, 1000, 5120
    prev = w4.w4a16_set_forced_rung(rung)
    try:
        info = w4.w4a16_plan_info(M, N, K)
        assert info["threads"] == WIDE and (info["k_slices"] > 1) == (rung == w4.RUNG_MMA_SPLITK)
        seed = si.config_seed(97, rung)
        x, qw, s, zw = _case(seed, M, N, K)
        w4.w4a16_probe_reset()
        y = w4.w4a16_linear(x.to(DEV), qw.to(DEV), s.to(DEV), zw.to(DEV))
        torch.cuda.synchronize()
        assert w4.w4a16_probe_counts()[rung] == 1
    finally:
        w4.w4a16_set_forced_rung(prev)
    assert_close(y, _ref(x, qw, s, zw), f"16-warp forced rung {rung}")


def test_wide_noalloc(w4):
    M, N, K = 8, 3000, 5120
    assert w4.w4a16_plan_info(M, N, K)["threads"] == WIDE
    seed = si.config_seed(98)
    x, qw, s, zw = _case(seed, M, N, K)
    ref = _ref(x, qw, s, zw)
    for i in range(2):
        y = torch.full((M, N), float("nan"), dtype=torch.float16, device=DEV)
        w4.w4a16_linear_noalloc(x.to(DEV), qw.to(DEV), s.to(DEV), zw.to(DEV), y)
        torch.cuda.synchronize()
        assert_close(y, ref, f"16-warp no-alloc call {i}")


@pytest.mark.parametrize("graph", [False, True])
def test_wide_round_with_waits(w4, graph):
    # A chain whose K all lie between what an 8-warp CTA holds unsplit at
    # 8 tokens (2560) and what a 16-warp CTA holds (5120): the round runs on
    # 16-warp CTAs, cooperative, with waits between the linears (each reads
    # the previous one's output, the last writes over the first input).
    M = 8
    dims = [4096, 3072, 5120, 4608, 3584]
    acts = [torch.zeros((M, d), dtype=torch.float16, device=DEV) for d in dims]
    acts[0].copy_(si.x(si.config_seed(99), M, dims[0]).to(DEV))
    layers = []
    for l in range(len(dims) - 1):
        K, N = dims[l], dims[l + 1]
        assert w4.w4a16_plan_info(M, N, K)["threads"] == WIDE
        seed = si.config_seed(99, l + 1)
        qw, s, zw = si.layer(seed, N, K, device=DEV)
        layers.append(dict(x=acts[l], qweight=qw, scales=s, zeros=zw, y=acts[l + 1], N=N, K=K,
                           seed=seed))
    qw, s, zw = si.layer(si.config_seed(99, 9), dims[0], dims[-1], device=DEV)
    layers.append(dict(x=acts[-1], qweight=qw, scales=s, zeros=zw, y=acts[0], N=dims[0],
                       K=dims[-1], seed=si.config_seed(99, 9)))
    descs = w4.make_descs(layers)
    x0 = acts[0].clone()
    for rep in range(2):
        acts[0].copy_(x0)
        for a in acts[1:]:
            a.fill_(float("nan"))
        w4.w4a16_probe_reset()
        if graph:
            g = w4.RoundGraph(descs, M)
            g.launch()
            torch.cuda.synchronize()
            g.destroy()
        else:
            w4.w4a16_decode_round(descs, M)
            torch.cuda.synchronize()
            assert w4.w4a16_kernel_launches() == 1
        chain = [x0] + [acts[l + 1].clone() for l in range(len(dims) - 1)]
        for l in range(len(dims) - 1):
            L = layers[l]
            qh, sh, zh = si.layer(L["seed"], L["N"], L["K"])
            ref = oracle.linear(si.as_u16(chain[l].cpu()), si.as_u32(qh), si.as_u16(sh),
                                si.as_u32(zh))
            assert_close(chain[l + 1], ref, f"16-warp round linear {l} rep {rep}")
        L = layers[-1]
        qh, sh, zh = si.layer(L["seed"], L["N"], L["K"])
        ref = oracle.linear(si.as_u16(chain[-1].cpu()), si.as_u32(qh), si.as_u16(sh),
                            si.as_u32(zh))
        assert_close(acts[0], ref, f"16-warp round write-after-read rep {rep}")
