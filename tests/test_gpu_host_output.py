"""Outputs written straight into page-locked host memory.

The linear calls and the decode round's descriptors accept a pinned host
tensor as y: the kernels store the result into host memory themselves (on a
Grace-Blackwell part, over the NVLink-C2C link), so a caller that wants the
result on the host needs no copy back.  Every case compares the host result
with the oracle and with the same call writing device memory, bit for bit:
only where y lives differs, not the arithmetic.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic_inputs as si
from helpers import assert_close

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
ALL_RUNGS = [0, 1, 2, 3, 4, 5]  # gemv, gemv_splitk, tc, tc_splitk, mma, mma_splitk


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


def _host(shape, dt=torch.float16):
    return torch.full(shape, float("nan"), dtype=dt).pin_memory()


def _same_bits(a, b):
    return torch.equal(a.cpu().view(torch.int16), b.cpu().view(torch.int16))


@pytest.mark.parametrize("rung", ALL_RUNGS + [-1])
def test_linear_host_y_every_rung(w4, rung):
    M = 16 if rung in (2, 3) else 4
    N, K = 1000, 2048
    seed = si.config_seed(111, rung + 1)
    qw, s, zw = si.layer(seed, N, K)
    x = si.x(seed, M, K)
    args = (x.to(DEV), qw.to(DEV), s.to(DEV), zw.to(DEV))
    prev = w4.w4a16_set_forced_rung(rung)
    try:
        y_host = _host((M, N))
        assert y_host.is_pinned()
        w4.w4a16_probe_reset()
        w4.w4a16_linear(*args, y=y_host)
        torch.cuda.synchronize()
        if rung >= 0:
            assert w4.w4a16_probe_counts()[rung] == 1
        y_dev = w4.w4a16_linear(*args)
        torch.cuda.synchronize()
    finally:
        w4.w4a16_set_forced_rung(prev)
    ref = oracle.linear(_bits(x), si.as_u32(qw), _bits(s), si.as_u32(zw))
    assert_close(y_host, ref, f"host y, rung {rung}")
    assert _same_bits(y_host, y_dev)


@pytest.mark.parametrize("M", [4, 16])
@pytest.mark.parametrize("dt", [torch.float16, torch.bfloat16])
def test_linear_ex_host_y_epilogues(w4, M, dt):
    name = "bf16" if dt == torch.bfloat16 else "f16"
    rtol = (2.0 ** -7 if M > 8 else 2.0 ** -8) if dt == torch.bfloat16 else None
    K = 1536
    # residual add (the residual in device memory, y on the host)
    N = 1152
    seed = si.config_seed(112, M, 1)
    qw, s, zw = si.layer(seed, N, K)
    x = si.x(seed, M, K).float().to(dt)
    s = s.float().to(dt) if dt == torch.bfloat16 else s
    r = si.residual(seed, M, N).float().to(dt)
    y_host = _host((M, N), dt)
    w4.w4a16_linear_ex(x.to(DEV), qw.to(DEV), s.to(DEV), zw.to(DEV),
                       epilogue=w4.EPILOGUE_RESIDUAL, residual=r.to(DEV), y=y_host)
    y_dev = w4.w4a16_linear_ex(x.to(DEV), qw.to(DEV), s.to(DEV), zw.to(DEV),
                               epilogue=w4.EPILOGUE_RESIDUAL, residual=r.to(DEV))
    torch.cuda.synchronize()
    h = oracle.linear(_bits(x), si.as_u32(qw), _bits(s), si.as_u32(zw), dtype=name)
    assert_close(y_host, oracle.add_residual(h, _bits(r), name), f"host y + residual {dt} M={M}",
                 rtol=rtol)
    assert _same_bits(y_host, y_dev)
    # SiLU-and-mul over the fused gate+up rows
    N = 2048
    seed = si.config_seed(112, M, 2)
    qw, s, zw = si.layer(seed, N, K)
    x = si.x(seed, M, K).float().to(dt)
    s = s.float().to(dt) if dt == torch.bfloat16 else s
    y_host = _host((M, N // 2), dt)
    w4.w4a16_linear_ex(x.to(DEV), qw.to(DEV), s.to(DEV), zw.to(DEV),
                       epilogue=w4.EPILOGUE_SILU_MUL, y=y_host)
    y_dev = w4.w4a16_linear_ex(x.to(DEV), qw.to(DEV), s.to(DEV), zw.to(DEV),
                               epilogue=w4.EPILOGUE_SILU_MUL)
    torch.cuda.synchronize()
    h = oracle.linear(_bits(x), si.as_u32(qw), _bits(s), si.as_u32(zw), dtype=name)
    assert_close(y_host, oracle.silu_mul(h), f"host y SiLU-and-mul {dt} M={M}", rtol=rtol)
    assert _same_bits(y_host, y_dev)


def test_noalloc_host_y(w4):
    M, N, K = 8, 3000, 5120
    seed = si.config_seed(113)
    qw, s, zw = si.layer(seed, N, K)
    x = si.x(seed, M, K)
    ref = oracle.linear(_bits(x), si.as_u32(qw), _bits(s), si.as_u32(zw))
    for i in range(2):
        y_host = _host((M, N))
        w4.w4a16_linear_noalloc(x.to(DEV), qw.to(DEV), s.to(DEV), zw.to(DEV), y_host)
        torch.cuda.synchronize()
        assert_close(y_host, ref, f"no-alloc host y, call {i}")


@pytest.mark.parametrize("M", [4, 16])
@pytest.mark.parametrize("graph", [False, True])
def test_round_host_y(w4, M, graph):
    # a round of four linears (one decoder layer's shapes, scaled down) whose
    # outputs all go to one pinned host buffer, against the same round into
    # device memory and against the oracle
    shapes = [(1024, 2048), (2048, 1536), (1536, 3000), (3072, 1024)]  # (K, N)
    total = sum(M * N for _, N in shapes)
    y_host = _host((total,))
    y_dev = torch.full((total,), float("nan"), dtype=torch.float16, device=DEV)
    host_layers, dev_layers, refs, off = [], [], [], 0
    for j, (K, N) in enumerate(shapes):
        seed = si.config_seed(114, M, j)
        qw, s, zw = si.layer(seed, N, K)
        x = si.x(seed, M, K)
        refs.append(oracle.linear(_bits(x), si.as_u32(qw), _bits(s), si.as_u32(zw)))
        common = dict(x=x.to(DEV), qweight=qw.to(DEV), scales=s.to(DEV), zeros=zw.to(DEV))
        host_layers.append(dict(common, y=y_host[off:off + M * N].view(M, N)))
        dev_layers.append(dict(common, y=y_dev[off:off + M * N].view(M, N)))
        off += M * N
    descs = w4.make_descs(host_layers)
    if graph:
        g = w4.RoundGraph(descs, M)
        g.launch()
        torch.cuda.synchronize()
        g.destroy()
    else:
        launches0 = w4.w4a16_kernel_launches()
        w4.w4a16_decode_round(descs, M)
        torch.cuda.synchronize()
        assert w4.w4a16_kernel_launches() - launches0 == 1
    w4.w4a16_decode_round(w4.make_descs(dev_layers), M)
    torch.cuda.synchronize()
    for L, ref, (K, N) in zip(host_layers, refs, shapes):
        assert_close(L["y"], ref, f"host y round M={M} K={K} N={N}")
    assert _same_bits(y_host, y_dev)
