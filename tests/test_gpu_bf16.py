"""GPU parity of bf16 activations (w4a16_linear_ex with W4A16_DTYPE_BF16, and
bf16 decode rounds) against the oracle's bf16 linear.

x, scales, residual and y are bfloat16; the oracle decodes the same bit
patterns and works in binary64.  Tolerance: the linear's rule with the
relative term raised to 2^-8 (helpers.RTOL_BF16), since one rounding of y to
bf16's 8 significant bits already costs up to 2^-9 |y|.  Layers of more than 8
tokens run on the tcgen05 rung, which also rounds each restored weight once to
bf16: there the relative term is 2^-7 (helpers.RTOL_BF16_TC).
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic_inputs as si
from helpers import RTOL_BF16_TC, assert_close, sample_rows

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
AUTO, MMA, MMA_SPLITK = -1, 4, 5
BF = torch.bfloat16


@pytest.fixture(scope="module")
def w4():
    import __graft_entry__
    __graft_entry__.build()
    import weight_only_int4_w4a16_gb300 as w4
    w4.w4a16_init(0, 256 << 20)
    yield w4
    w4.w4a16_set_forced_rung(w4.RUNG_AUTO)


@pytest.fixture(autouse=True)
def no_device_errors(request):
    yield
    if "w4" in request.fixturenames:
        import weight_only_int4_w4a16_gb300 as w4
        assert w4.w4a16_device_status() == 0, "a kernel reported an expired bounded wait"


def bits(t):
    """bf16 tensor -> numpy uint16 bit patterns (host)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def case(seed, M, N, K, x_scale=1.0):
    """Seeded bf16 layer: x (times x_scale, a power of two) and scales are the
    fp16 draws rounded to bf16."""
    qw, s16, zw = si.layer(seed, N, K)
    x = (si.x(seed, M, K).float() * x_scale).to(BF)
    return x, qw, s16.float().to(BF), zw


def reference(x, qw, s, zw, rows=None):
    if rows is None:
        return oracle.linear(bits(x), si.as_u32(qw), bits(s), si.as_u32(zw), dtype="bf16")
    return oracle.linear_rows(bits(x), si.as_u32(qw), bits(s), si.as_u32(zw), rows,
                              dtype="bf16")


def run(w4, rung, x, qw, s, zw, epi=0, residual=None, cols=None):
    M, N = x.shape[0], qw.shape[0]
    y = torch.full((M, cols or N), float("nan"), dtype=BF, device=DEV)
    prev = w4.w4a16_set_forced_rung(rung)
    try:
        w4.w4a16_linear_ex(x.to(DEV), qw.to(DEV), s.to(DEV), zw.to(DEV), epi,
                           residual=None if residual is None else residual.to(DEV), y=y)
    except w4.W4A16Error as e:
        if e.status == w4.W4A16_ERR_UNSUPPORTED and rung != AUTO:
            return None
        raise
    finally:
        w4.w4a16_set_forced_rung(prev)
    torch.cuda.synchronize()
    return y


SHAPES = [(1, 1024, 512), (4, 5120, 6144), (4, 5120, 17408), (8, 1000, 2560), (3, 777, 1408),
          (2, 8192, 5120), (12, 512, 1024)]


@pytest.mark.parametrize("rung", [AUTO, MMA, MMA_SPLITK])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_bf16_linear_matches_oracle(w4, rung, M, N, K):
    x, qw, s, zw = case(si.config_seed(100, 0, M), M, N, K)
    y = run(w4, rung, x, qw, s, zw)
    if y is None:
        pytest.skip("rung cannot run this shape")
    # more than 8 tokens run on the tcgen05 rung (weights restored to bf16)
    rtol = RTOL_BF16_TC if rung == AUTO and M > 8 else None
    assert_close(y, reference(x, qw, s, zw), f"bf16 M={M} N={N} K={K} rung={rung}", rtol=rtol)


def test_bf16_range_beyond_fp16(w4):
    # activations of 2^20 times N(0, 1): far outside fp16's range, ordinary in bf16
    M, N, K = 4, 2048, 2048
    x, qw, s, zw = case(si.config_seed(101), M, N, K, x_scale=2.0 ** 20)
    assert float(x.abs().max()) > 65504
    y = run(w4, AUTO, x, qw, s, zw)
    assert_close(y, reference(x, qw, s, zw), "bf16 large activations")


def test_bf16_integer_case_bit_exact(w4):
    # x in {-1, 0, 1}, s = 2^-4: every partial sum on the GPU is an integer
    # (times 2^-4) below 2^24, so its fp32 result is exact and its one bf16
    # rounding must equal the oracle's exact value rounded to bf16
    M, N, K = 4, 1024, 1024
    gen = torch.Generator().manual_seed(5)
    X = torch.randint(-1, 2, (M, K), generator=gen).to(BF)
    qw, _, zw = si.layer(7, N, K)
    s = torch.full((N, K // 128), 2.0 ** -4, dtype=BF)
    y = run(w4, AUTO, X, qw, s, zw)
    ref = reference(X, qw, s, zw)
    want = oracle.double_to_bf16(ref)
    assert np.array_equal(bits(y), want)


@pytest.mark.parametrize("M,N,K", [(4, 5120, 17408), (1, 5120, 6144), (8, 1000, 2560)])
def test_bf16_residual(w4, M, N, K):
    x, qw, s, zw = case(si.config_seed(102, 0, M), M, N, K)
    r = si.residual(si.config_seed(102, 0, M), M, N).float().to(BF)
    y = run(w4, AUTO, x, qw, s, zw, w4.EPILOGUE_RESIDUAL, r)
    ref = oracle.add_residual(reference(x, qw, s, zw), bits(r), dtype="bf16")
    assert_close(y, ref, f"bf16 residual M={M}")


@pytest.mark.parametrize("rung", [AUTO, MMA_SPLITK])
@pytest.mark.parametrize("M,N,K", [(4, 2048, 1024), (1, 1056, 1408), (8, 4096, 5120)])
def test_bf16_silu_mul(w4, rung, M, N, K):
    x, qw, s, zw = case(si.config_seed(103, 0, M), M, N, K)
    y = run(w4, rung, x, qw, s, zw, w4.EPILOGUE_SILU_MUL, cols=N // 2)
    if y is None:
        pytest.skip("rung cannot run this shape")
    assert_close(y, oracle.silu_mul(reference(x, qw, s, zw)), f"bf16 silu M={M}")


@pytest.mark.parametrize("M", [1, 4, 8])
def test_bf16_full_size_sampled(w4, M):
    # the 27B layer's gate+up (5120 -> 34816), sampled output rows
    N, K = 34816, 5120
    seed = si.config_seed(104, 0, M)
    qw, s16, zw = si.layer(seed, N, K, device=DEV)
    x = si.x(seed, M, K).float().to(BF)
    s = s16.float().to(BF)
    y = run(w4, AUTO, x, qw, s, zw)
    rows = sample_rows(N, 6, seed=M)
    qh, sh, zh = si.layer(seed, N, K, rows=rows)
    ref = oracle.linear_rows(bits(x), si.as_u32(qh), bits(sh.float().to(BF)), si.as_u32(zh),
                             np.arange(rows.size), dtype="bf16")
    assert_close(y[:, torch.from_numpy(rows).to(DEV)], ref, f"bf16 gate+up M={M}")


@pytest.mark.parametrize("graph", [False, True])
def test_bf16_decode_round(w4, graph):
    # four linears of a layer in bf16, one fused launch; then a round mixing
    # fp16 and bf16, which runs linear by linear with the same results
    M = 4
    shapes = [(8192, 5120), (5120, 6144), (34816, 5120), (5120, 17408)]
    layers, refs = [], []
    for j, (N, K) in enumerate(shapes):
        seed = si.config_seed(105, 0, j)
        x, qw, s, zw = case(seed, M, N, K)
        y = torch.full((M, N), float("nan"), dtype=BF, device=DEV)
        layers.append(dict(x=x.to(DEV), qweight=qw.to(DEV), scales=s.to(DEV),
                           zeros=zw.to(DEV), y=y))
        rows = sample_rows(N, 4, seed=j)
        refs.append((rows, reference(x, qw, s, zw, rows)))
    descs = w4.make_descs(layers)
    w4.w4a16_probe_reset()
    if graph:
        g = w4.RoundGraph(descs, M)
        g.launch()
        torch.cuda.synchronize()
        g.destroy()
    else:
        w4.w4a16_decode_round(descs, M)
        torch.cuda.synchronize()
        assert w4.w4a16_kernel_launches() == 1  # one fused launch
    for L, (rows, ref) in zip(layers, refs):
        assert_close(L["y"][:, torch.from_numpy(rows).to(DEV)], ref, "bf16 round")
    # mixed types: the fp16 linear and the bf16 ones side by side
    seed = si.config_seed(106)
    qw, s16, zw = si.layer(seed, 1024, 2048, device=DEV)
    x16 = si.x(seed, M, 2048).to(DEV)
    y16 = torch.full((M, 1024), float("nan"), dtype=torch.float16, device=DEV)
    mixed = w4.make_descs(layers[:2] + [dict(x=x16, qweight=qw, scales=s16, zeros=zw, y=y16)])
    w4.w4a16_decode_round(mixed, M)
    torch.cuda.synchronize()
    ref16 = oracle.linear(si.as_u16(x16), si.as_u32(qw), si.as_u16(s16), si.as_u32(zw))
    assert_close(y16, ref16, "fp16 linear in a mixed round")
    for L, (rows, ref) in zip(layers[:2], refs[:2]):
        assert_close(L["y"][:, torch.from_numpy(rows).to(DEV)], ref, "bf16 in a mixed round")


def test_bf16_on_forced_rungs(w4):
    # the CUDA-core rungs have no bf16 path; the tcgen05 rung has one (bf16
    # restore and bf16 tensor-core products), also below 9 tokens when forced
    x, qw, s, zw = case(1, 2, 64, 256)
    prev = w4.w4a16_set_forced_rung(0)
    try:
        with pytest.raises(w4.W4A16Error) as e:
            w4.w4a16_linear_ex(x.to(DEV), qw.to(DEV), s.to(DEV), zw.to(DEV))
        assert e.value.status == w4.W4A16_ERR_UNSUPPORTED
        w4.w4a16_set_forced_rung(2)
        y = w4.w4a16_linear_ex(x.to(DEV), qw.to(DEV), s.to(DEV), zw.to(DEV))
        torch.cuda.synchronize()
        assert_close(y, reference(x, qw, s, zw), "bf16 on the forced tcgen05 rung",
                     rtol=RTOL_BF16_TC)
    finally:
        w4.w4a16_set_forced_rung(prev)
