"""GPU parity of the fused epilogues (w4a16_linear_epilogue and epilogues in a
decode round) against the oracle.

The oracle computes the linear in binary64 and then its epilogue (residual add,
SiLU-and-mul) in binary64; the kernel keeps h = x @ W^T in fp32, applies the
epilogue in fp32 and rounds once to fp16.  The acceptance rule of the linear,
|y_gpu - y_ref| <= 1e-3 * max|y_ref| + 1e-3, is applied to the epilogue's
output: its fp16 rounding (2^-11 relative at most) dominates, as it does for
the plain linear, and h is never rounded to fp16 on the GPU side.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic_inputs as si
from helpers import assert_close, sample_rows, sampled_reference

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
AUTO, MMA, MMA_SPLITK = -1, 4, 5


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


def _epilogue(w4, rung, x, qw, s, zw, epi, residual, y):
    """Run on a forced rung (AUTO: the dispatch table); None if that rung
    cannot run the shape."""
    prev = w4.w4a16_set_forced_rung(rung)
    try:
        w4.w4a16_linear_epilogue(x, qw, s, zw, epi, residual=residual, y=y)
    except w4.W4A16Error as e:
        if e.status == w4.W4A16_ERR_UNSUPPORTED and rung != AUTO:
            return None
        raise
    finally:
        w4.w4a16_set_forced_rung(prev)
    torch.cuda.synchronize()
    return y


def _oracle_linear(seed, x_cpu, N, K):
    qw, s, zw = si.layer(seed, N, K)
    return oracle.linear(si.as_u16(x_cpu), si.as_u32(qw), si.as_u16(s), si.as_u32(zw))


def _nan(M, N):
    return torch.full((M, N), float("nan"), dtype=torch.float16, device=DEV)


# o-projection and down-projection shapes of the 27B decode layer (K = 6144,
# 17408: split K), ragged N and K (partial strips, a partial last stage), M
# from 1 to 8
RES_SHAPES = [(4, 5120, 6144), (4, 5120, 17408), (1, 777, 1408), (8, 1000, 2560), (3, 64, 640)]


@pytest.mark.parametrize("rung", [AUTO, MMA, MMA_SPLITK])
@pytest.mark.parametrize("M,N,K", RES_SHAPES)
def test_residual_matches_oracle(w4, rung, M, N, K):
    seed = si.config_seed(80, 0, M)
    x = si.x(seed, M, K)
    r = si.residual(seed, M, N)
    qw, s, zw = si.layer(seed, N, K, device=DEV)
    xd, rd = x.to(DEV), r.to(DEV)
    y = _epilogue(w4, rung, xd, qw, s, zw, w4.EPILOGUE_RESIDUAL, rd, _nan(M, N))
    if y is None:
        pytest.skip("rung cannot run this shape")
    ref = oracle.add_residual(_oracle_linear(seed, x, N, K), si.as_u16(r))
    assert_close(y, ref, f"residual M={M} N={N} K={K} rung={rung}")
    # in place (y += x W^T): the same kernel and arithmetic, the same bits
    y2 = rd.clone()
    _epilogue(w4, rung, xd, qw, s, zw, w4.EPILOGUE_RESIDUAL, y2, y2)
    assert torch.equal(y2.view(torch.int16), y.view(torch.int16))
    assert torch.equal(rd.view(torch.int16), r.to(DEV).view(torch.int16))  # input untouched


# fused gate+up shapes: N = 2 * intermediate, gate rows first
SILU_SHAPES = [(4, 2048, 1024), (1, 1056, 1408), (8, 2560, 2560), (3, 4096, 5120),
               (4, 6144, 17408)]


@pytest.mark.parametrize("rung", [AUTO, MMA, MMA_SPLITK])
@pytest.mark.parametrize("M,N,K", SILU_SHAPES)
def test_silu_mul_matches_oracle(w4, rung, M, N, K):
    seed = si.config_seed(81, 0, M)
    x = si.x(seed, M, K)
    qw, s, zw = si.layer(seed, N, K, device=DEV)
    y = _epilogue(w4, rung, x.to(DEV), qw, s, zw, w4.EPILOGUE_SILU_MUL, None, _nan(M, N // 2))
    if y is None:
        pytest.skip("rung cannot run this shape")
    ref = oracle.silu_mul(_oracle_linear(seed, x, N, K))
    assert_close(y, ref, f"silu_mul M={M} N={N} K={K} rung={rung}")


@pytest.mark.parametrize("rung", [AUTO, MMA_SPLITK])
@pytest.mark.parametrize("M", [1, 4, 8])
def test_silu_mul_full_gate_up_sampled(w4, rung, M):
    # the 27B layer's fused gate+up (5120 -> 2 x 17408): sampled output
    # columns, each from its gate row and its up row
    N, K = 34816, 5120
    I = N // 2
    seed = si.config_seed(82, 0, M)
    x = si.x(seed, M, K)
    qw, s, zw = si.layer(seed, N, K, device=DEV)
    y = _epilogue(w4, rung, x.to(DEV), qw, s, zw, w4.EPILOGUE_SILU_MUL, None, _nan(M, I))
    assert y is not None
    cols = sample_rows(I, 6, seed=M)
    h = sampled_reference(seed, x, N, K, np.concatenate([cols, cols + I]))
    ref = oracle.silu_mul(h)
    assert_close(y[:, torch.from_numpy(cols).to(DEV)], ref, f"gate+up M={M} rung={rung}")
    assert torch.isfinite(y).all()


@pytest.mark.parametrize("M", [9, 20])
def test_epilogues_beyond_8_tokens(w4, M):
    # more than 8 tokens: both epilogues on the tcgen05 rung (one reading of
    # the weights for up to 64 tokens)
    N, K = 1024, 2048
    seed = si.config_seed(86, 0, M)
    x = si.x(seed, M, K)
    r = si.residual(seed, M, N)
    qw, s, zw = si.layer(seed, N, K, device=DEV)
    w4.w4a16_probe_reset()
    y = _epilogue(w4, AUTO, x.to(DEV), qw, s, zw, w4.EPILOGUE_RESIDUAL, r.to(DEV), _nan(M, N))
    c = w4.w4a16_probe_counts()
    assert c[w4.RUNG_TC] + c[w4.RUNG_TC_SPLITK] == 1 and sum(c) == 1
    h = _oracle_linear(seed, x, N, K)
    assert_close(y, oracle.add_residual(h, si.as_u16(r)), f"residual M={M}")
    w4.w4a16_probe_reset()
    y = _epilogue(w4, AUTO, x.to(DEV), qw, s, zw, w4.EPILOGUE_SILU_MUL, None, _nan(M, N // 2))
    c = w4.w4a16_probe_counts()
    assert c[w4.RUNG_TC] + c[w4.RUNG_TC_SPLITK] == 1 and sum(c) == 1
    assert_close(y, oracle.silu_mul(h), f"silu_mul M={M}")


def test_epilogue_rejections_on_device(w4):
    qw, s, zw = si.layer(1, 64, 256, device=DEV)
    x = torch.zeros((2, 256), dtype=torch.float16, device=DEV)
    prev = w4.w4a16_set_forced_rung(0)  # a CUDA-core rung has no epilogue
    try:
        with pytest.raises(w4.W4A16Error) as e:
            w4.w4a16_linear_epilogue(x, qw, s, zw, w4.EPILOGUE_RESIDUAL,
                                     residual=torch.zeros((2, 64), dtype=torch.float16, device=DEV))
        assert e.value.status == w4.W4A16_ERR_UNSUPPORTED
        # EPILOGUE_NONE is w4a16_linear, on any rung
        w4.w4a16_linear_epilogue(x, qw, s, zw, w4.EPILOGUE_NONE)
    finally:
        w4.w4a16_set_forced_rung(prev)


@pytest.mark.parametrize("graph", [False, True])
def test_decode_round_with_epilogues(w4, graph):
    # Two decoder layers as one round (M = 4, hidden 1024, intermediate 2048):
    #   qkv:     q_l = x_l @ Wqkv                      (no epilogue)
    #   o:       h_l = a_l @ Wo + x_l                  (residual; a_l a seeded input)
    #   gate+up: g_l = silu(h_l Wg) * (h_l Wu)         (SiLU-and-mul)
    #   down:    x_{l+1} = g_l @ Wd + h_l              (residual; the last layer
    #            writes it over h_l in place, after gate+up has read h_l)
    # Linears wait for the ones whose outputs they read as x or as residual,
    # and the in-place write waits for the read of h_l.  Every output is
    # checked against the oracle applied to the inputs the GPU used; the round
    # runs twice.  Without the normalisations of a real decoder the values
    # grow with every SiLU-and-mul: x_0 and a_l are N(0, 1/16), which keeps
    # the second layer's outputs (a few hundred) well inside fp16.
    M, H, I, QKV = 4, 1024, 2048, 1536
    n_layers = 2
    x0 = (si.x(si.config_seed(83), M, H) * 0.25).to(DEV)
    x_in = x0.clone()
    layers, spec = [], []
    for l in range(n_layers):
        a = (si.x(si.config_seed(84, l), M, H) * 0.25).to(DEV)
        q, h, g = _nan(M, QKV), _nan(M, H), _nan(M, I)
        inplace = l == n_layers - 1
        x_out = h if inplace else _nan(M, H)

        def add(x, N, K, y, epi, res, key):
            seed = si.config_seed(85, l, key)
            qw, s, zw = si.layer(seed, N, K, device=DEV)
            layers.append(dict(x=x, qweight=qw, scales=s, zeros=zw, y=y, epilogue=epi,
                               residual=res))
            spec.append((seed, N, K))

        add(x_in, QKV, H, q, w4.EPILOGUE_NONE, None, 0)
        add(a, H, H, h, w4.EPILOGUE_RESIDUAL, x_in, 1)
        add(h, 2 * I, H, g, w4.EPILOGUE_SILU_MUL, None, 2)
        add(g, H, I, x_out, w4.EPILOGUE_RESIDUAL, h, 3)
        x_in = x_out
    descs = w4.make_descs(layers)
    x_first = layers[0]["x"]
    for rep in range(2):
        x_first.copy_(x0)
        for L in layers:
            L["y"].fill_(float("nan"))
        if graph:
            gr = w4.RoundGraph(descs, M)
            gr.launch()
            torch.cuda.synchronize()
            gr.destroy()
        else:
            w4.w4a16_decode_round(descs, M)
            torch.cuda.synchronize()
        assert w4.w4a16_device_status() == 0
        x_cur = x0.cpu()
        for l in range(n_layers):
            Lq, Lo, Lg, Ld = layers[4 * l:4 * l + 4]
            sq, so, sg, sd = spec[4 * l:4 * l + 4]
            assert_close(Lq["y"], _oracle_linear(sq[0], x_cur, sq[1], sq[2]), f"qkv {l} rep {rep}")
            h_ref = oracle.add_residual(_oracle_linear(so[0], Lo["x"].cpu(), so[1], so[2]),
                                        si.as_u16(x_cur))
            if Ld["y"].data_ptr() == Lo["y"].data_ptr():
                # h_l is gone (overwritten in place): the GPU used h_ref
                # rounded to fp16, up to an ulp in a few elements, which moves
                # the next outputs far less than the tolerance
                h_used = torch.from_numpy(h_ref.astype(np.float16))
            else:
                assert_close(Lo["y"], h_ref, f"o-proj {l} rep {rep}")
                h_used = Lo["y"].cpu()
            g_gpu = Lg["y"].cpu()
            assert_close(g_gpu, oracle.silu_mul(_oracle_linear(sg[0], h_used, sg[1], sg[2])),
                         f"gate+up {l} rep {rep}")
            x_next = Ld["y"].cpu()
            down_ref = oracle.add_residual(_oracle_linear(sd[0], g_gpu, sd[1], sd[2]),
                                           si.as_u16(h_used))
            assert_close(x_next, down_ref, f"down {l} rep {rep}")
            x_cur = x_next
