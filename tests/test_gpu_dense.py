"""GPU parity of the dense 16-bit linear (w4a16_dense_linear) against the
oracle's dense_linear: fp16 and bf16, split and unsplit K, ragged N, tiles of
8 tokens, a bit-exact integer case, and agreement with the 4-bit rung over
the 4-bit weights dequantised to fp16 on the device.

Tolerance: the linear's rule (bf16 outputs: relative term 2^-8, helpers).
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic_inputs as si
from helpers import assert_close, sample_rows

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def w4():
    import __graft_entry__
    __graft_entry__.build()
    import weight_only_int4_w4a16_gb300 as w4
    w4.w4a16_init(0, 256 << 20)
    return w4


@pytest.fixture(autouse=True)
def no_device_errors(request):
    yield
    if "w4" in request.fixturenames:
        import weight_only_int4_w4a16_gb300 as w4
        assert w4.w4a16_device_status() == 0, "a kernel reported an expired bounded wait"


def bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def case(seed, M, N, K, dt):
    x = si.x(seed, M, K).float().to(dt)
    w = si.dense_weight(seed, N, K).float().to(dt)
    return x, w


def run(w4, x, w):
    M, N = x.shape[0], w.shape[0]
    y = torch.full((M, N), float("nan"), dtype=x.dtype, device=DEV)
    w4.w4a16_dense_linear(x.to(DEV), w.to(DEV), y=y)
    torch.cuda.synchronize()
    return y


def name(dt):
    return "bf16" if dt == torch.bfloat16 else "f16"


# the pages' dense shape (N 8192, K 5120, M 2/4/8), a split-K shape, ragged N,
# a single stage of K, more than 8 tokens
SHAPES = [(1, 1024, 512), (2, 8192, 5120), (4, 8192, 5120), (8, 8192, 5120), (4, 5120, 17408),
          (3, 777, 1408), (1, 100, 128), (12, 512, 1024)]


@pytest.mark.parametrize("dt", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_dense_matches_oracle(w4, M, N, K, dt):
    x, w = case(si.config_seed(110, 0, M), M, N, K, dt)
    y = run(w4, x, w)
    ref = oracle.dense_linear(bits(x), bits(w), name(dt))
    assert_close(y, ref, f"dense {name(dt)} M={M} N={N} K={K}")


def test_dense_integer_case_bit_exact(w4):
    # x in {-1, 0, 1} and integer weights: every fp32 partial sum is an exact
    # integer, so y is the exact product rounded once to fp16
    M, N, K = 4, 1000, 2048
    gen = torch.Generator().manual_seed(9)
    X = torch.randint(-1, 2, (M, K), generator=gen).to(torch.float16)
    W = torch.randint(-8, 9, (N, K), generator=gen).to(torch.float16)
    y = run(w4, X, W)
    want = oracle.double_to_half(oracle.dense_linear(bits(X), bits(W)))
    assert np.array_equal(bits(y), want)


def test_dense_over_dequantised_weights_matches_the_4bit_rung(w4):
    # the 4-bit layer dequantised on the device (exact to fp16 when the scale
    # is a power of two) through the dense path, against the 4-bit path
    M, N, K = 4, 4096, 5120
    seed = si.config_seed(111)
    qw, _, zw = si.layer(seed, N, K, device=DEV)
    s = torch.full((N, K // 128), 2.0 ** -6, dtype=torch.float16, device=DEV)
    x = si.x(seed, M, K).to(DEV)
    _, w16 = w4.w4a16_dequant(qw, s, zw, K, f32=False)
    y_dense = run(w4, x, w16)
    y_4bit = w4.w4a16_linear(x, qw, s, zw)
    torch.cuda.synchronize()
    ref = oracle.linear(si.as_u16(x), si.as_u32(qw), si.as_u16(s), si.as_u32(zw))
    assert_close(y_dense, ref, "dense over dequantised weights")
    assert_close(y_4bit, ref, "4-bit")


@pytest.mark.parametrize("dt", [torch.float16, torch.bfloat16])
def test_dense_run_to_run_bit_identical(w4, dt):
    x, w = case(si.config_seed(112), 4, 5120, 17408, dt)
    xd, wd = x.to(DEV), w.to(DEV)
    ys = [w4.w4a16_dense_linear(xd, wd) for _ in range(5)]
    torch.cuda.synchronize()
    for y in ys[1:]:
        assert torch.equal(y.view(torch.int16), ys[0].view(torch.int16))


@pytest.mark.parametrize("M", [1, 8])
def test_dense_full_size_sampled(w4, M):
    # a gate+up-sized dense layer (K 5120, N 34816: 356 MB of fp16 weights,
    # made on the device by dequantising a seeded 4-bit layer); sampled rows
    # are copied back for the oracle
    N, K = 34816, 5120
    seed = si.config_seed(113, 0, M)
    qw, s, zw = si.layer(seed, N, K, device=DEV)
    _, w16 = w4.w4a16_dequant(qw, s, zw, K, f32=False)
    del qw, s, zw
    x = si.x(seed, M, K)
    y = run(w4, x, w16)
    rows = sample_rows(N, 6, seed=M)
    w_rows = w16[torch.from_numpy(rows).to(DEV)]
    ref = oracle.dense_linear(bits(x), bits(w_rows))
    assert_close(y[:, torch.from_numpy(rows).to(DEV)], ref, f"dense full size M={M}")
