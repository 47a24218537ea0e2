"""Fused rounds of 9..64 tokens on the tcgen05 rung: one launch per round.

A round of linears (the 27B decode layer's qkv, o, gate+up and down shapes, or
a chain whose linears read each other's outputs) with more tokens than the
warp-MMA kernel takes runs as one stream-K sequence of (linear, tile, stage)
work on the tcgen05 kernel (forum.sourcefind.cn thread "vLLM on Hygon Z100",
section 七: past the small-M GEMV, the prefill-like shapes go to a GEMM path).
Every output is compared with the oracle; a round whose linears wait on each
other must give the results of running them one after another.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic_inputs as si
from helpers import assert_close

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
SHAPES = [(5120, 8192), (6144, 5120), (5120, 34816), (17408, 5120)]  # (K, N)


@pytest.fixture(scope="module")
def w4():
    import __graft_entry__
    __graft_entry__.build()
    import weight_only_int4_w4a16_gb300 as w4
    if w4.w4a16_device_sm_count() == 0:
        w4.w4a16_init(0, 256 << 20)
    yield w4


@pytest.fixture(autouse=True)
def no_device_errors(request):
    yield
    if "w4" in request.fixturenames:
        import weight_only_int4_w4a16_gb300 as w4
        assert w4.w4a16_device_status() == 0, "a kernel reported an expired bounded wait"


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _round(n_layers, M, seed_cfg, shapes=SHAPES):
    layers, xs = [], {}
    for j, (K, N) in enumerate(shapes):
        xs[j] = si.x(si.config_seed(seed_cfg, 0, 8 + j), M, K)
    for l in range(n_layers):
        for j, (K, N) in enumerate(shapes):
            seed = si.config_seed(seed_cfg, l, j)
            qw, s, zw = si.layer(seed, N, K, device=DEV)
            layers.append(dict(x=xs[j].to(DEV), qweight=qw, scales=s, zeros=zw,
                               y=torch.full((M, N), float("nan"), dtype=torch.float16, device=DEV),
                               N=N, K=K, j=j))
    return layers, xs


def _ref(L, x_cpu):
    return oracle.linear(si.as_u16(x_cpu), si.as_u32(L["qweight"]), si.as_u16(L["scales"]),
                         si.as_u32(L["zeros"]))


@pytest.mark.parametrize("M,n_layers", [(16, 2), (33, 2), (64, 1)])
def test_tc_round_full_output(w4, M, n_layers):
    layers, xs = _round(n_layers, M, 101)
    descs = w4.make_descs(layers)
    w4.w4a16_probe_reset()
    launches0 = w4.w4a16_kernel_launches()
    w4.w4a16_decode_round(descs, M)
    torch.cuda.synchronize()
    assert w4.w4a16_kernel_launches() - launches0 == 1, "the round is one launch"
    counts = w4.w4a16_probe_counts()
    assert counts[w4.RUNG_TC_SPLITK] == len(layers) and sum(counts) == len(layers)
    first = [L["y"].clone() for L in layers]
    for L in layers:
        assert_close(L["y"], _ref(L, xs[L["j"]]), f"tc round M={M} linear j={L['j']}")
    # again (the arrival counters are left zeroed), and as a CUDA graph:
    # the same bits
    for L in layers:
        L["y"].fill_(float("nan"))
    g = w4.RoundGraph(descs, M)
    g.launch()
    torch.cuda.synchronize()
    g.destroy()
    for L, f in zip(layers, first):
        assert torch.equal(L["y"].view(torch.int16), f.view(torch.int16))


@pytest.mark.parametrize("graph", [False, True])
def test_tc_round_chained_waits(w4, graph):
    # each linear reads the previous one's output; the last writes over the
    # first input (write after read); a cooperative launch with waits
    M = 24
    dims = [1024, 2048, 1536, 1024, 3072, 2048]
    acts = [torch.zeros((M, d), dtype=torch.float16, device=DEV) for d in dims]
    acts[0].copy_(si.x(si.config_seed(102), M, dims[0]).to(DEV))
    layers = []
    for l in range(len(dims) - 1):
        K, N = dims[l], dims[l + 1]
        seed = si.config_seed(102, l + 1)
        qw, s, zw = si.layer(seed, N, K, device=DEV)
        layers.append(dict(x=acts[l], qweight=qw, scales=s, zeros=zw, y=acts[l + 1], N=N, K=K,
                           seed=seed))
    qw, s, zw = si.layer(si.config_seed(102, 9), dims[0], dims[-1], device=DEV)
    layers.append(dict(x=acts[-1], qweight=qw, scales=s, zeros=zw, y=acts[0], N=dims[0],
                       K=dims[-1], seed=si.config_seed(102, 9)))
    descs = w4.make_descs(layers)
    x0 = acts[0].clone()
    for rep in range(2):
        acts[0].copy_(x0)
        for a in acts[1:]:
            a.fill_(float("nan"))
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
        chain = [x0] + [acts[l + 1].clone() for l in range(len(dims) - 1)]
        for l in range(len(dims) - 1):
            L = layers[l]
            qh, sh, zh = si.layer(L["seed"], L["N"], L["K"])
            ref = oracle.linear(si.as_u16(chain[l].cpu()), si.as_u32(qh), si.as_u16(sh),
                                si.as_u32(zh))
            assert_close(chain[l + 1], ref, f"tc chained linear {l} rep {rep}")
        L = layers[-1]
        qh, sh, zh = si.layer(L["seed"], L["N"], L["K"])
        ref = oracle.linear(si.as_u16(chain[-1].cpu()), si.as_u32(qh), si.as_u16(sh),
                            si.as_u32(zh))
        assert_close(acts[0], ref, f"tc chained write-after-read rep {rep}")


@pytest.mark.parametrize("dt", [torch.float16, torch.bfloat16])
def test_tc_round_epilogues(w4, dt):
    # a decoder layer's tail: o + residual (in place), gate+up with
    # SiLU-and-mul, down + residual (in place), the down projection reading
    # the SiLU output: waits, epilogues and the 16-bit type in one launch
    M, H, I = 20, 1024, 1536
    name = "bf16" if dt == torch.bfloat16 else "f16"
    attn = si.x(si.config_seed(103, 1), M, 2048).float().to(dt).to(DEV)
    hidden = si.residual(si.config_seed(103, 2), M, H).float().to(dt).to(DEV)
    act = torch.full((M, I), float("nan"), dtype=dt, device=DEV)
    shapes = [(2048, H, w4.EPILOGUE_RESIDUAL), (H, 2 * I, w4.EPILOGUE_SILU_MUL),
              (I, H, w4.EPILOGUE_RESIDUAL)]
    ws = []
    for i, (K, N, _) in enumerate(shapes):
        qw, s, zw = si.layer(si.config_seed(103, 10 + i), N, K)
        ws.append((qw, s.float().to(dt) if dt == torch.bfloat16 else s, zw))
    h0 = hidden.clone()
    layers = [
        dict(x=attn, qweight=ws[0][0].to(DEV), scales=ws[0][1].to(DEV), zeros=ws[0][2].to(DEV),
             y=hidden, epilogue=w4.EPILOGUE_RESIDUAL, residual=hidden),
        dict(x=hidden, qweight=ws[1][0].to(DEV), scales=ws[1][1].to(DEV), zeros=ws[1][2].to(DEV),
             y=act, epilogue=w4.EPILOGUE_SILU_MUL),
        dict(x=act, qweight=ws[2][0].to(DEV), scales=ws[2][1].to(DEV), zeros=ws[2][2].to(DEV),
             y=hidden, epilogue=w4.EPILOGUE_RESIDUAL, residual=hidden),
    ]
    descs = w4.make_descs(layers)
    launches0 = w4.w4a16_kernel_launches()
    w4.w4a16_decode_round(descs, M)
    torch.cuda.synchronize()
    assert w4.w4a16_kernel_launches() - launches0 == 1
    # the oracle, step by step, on the values the GPU used (each rounded once)
    h1 = oracle.add_residual(oracle.linear(_bits(attn.cpu()), si.as_u32(ws[0][0]),
                                           _bits(ws[0][1]), si.as_u32(ws[0][2]), dtype=name),
                             _bits(h0.cpu()), name)
    rtol = 2.0 ** -7 if dt == torch.bfloat16 else None
    # the intermediate values the GPU produced feed the next step's reference
    out_cols = act.cpu()
    h_used = torch.from_numpy(h1.astype(np.float32)).to(dt)
    a_ref = oracle.silu_mul(oracle.linear(_bits(h_used), si.as_u32(ws[1][0]), _bits(ws[1][1]),
                                          si.as_u32(ws[1][2]), dtype=name))
    assert_close(act, a_ref, f"tc round SiLU-and-mul {dt}", rtol=rtol)
    h2 = oracle.add_residual(oracle.linear(_bits(out_cols), si.as_u32(ws[2][0]), _bits(ws[2][1]),
                                           si.as_u32(ws[2][2]), dtype=name),
                             _bits(h_used), name)
    assert_close(hidden, h2, f"tc round down + residual {dt}", rtol=rtol)


def test_tc_round_ragged(w4):
    # ragged tiles in one stream-K sequence: N not a multiple of 128 (and a
    # SiLU-and-mul layer whose N/2 is not a multiple of 64), K of 11 groups
    # (a short last stage), 9 tokens (7 padding columns of the MMA)
    M = 9
    specs = [(1408, 777, w4.EPILOGUE_NONE), (1408, 1000, w4.EPILOGUE_RESIDUAL),
             (1408, 320, w4.EPILOGUE_SILU_MUL), (2048, 4100, w4.EPILOGUE_NONE)]
    layers, refs = [], []
    for i, (K, N, epi) in enumerate(specs):
        seed = si.config_seed(104, i)
        qw, s, zw = si.layer(seed, N, K)
        x = si.x(seed, M, K)
        cols = N // 2 if epi == w4.EPILOGUE_SILU_MUL else N
        r = si.residual(seed, M, N) if epi == w4.EPILOGUE_RESIDUAL else None
        h = oracle.linear(_bits(x), si.as_u32(qw), _bits(s), si.as_u32(zw))
        if epi == w4.EPILOGUE_RESIDUAL:
            h = oracle.add_residual(h, _bits(r))
        elif epi == w4.EPILOGUE_SILU_MUL:
            h = oracle.silu_mul(h)
        refs.append(h)
        layers.append(dict(x=x.to(DEV), qweight=qw.to(DEV), scales=s.to(DEV), zeros=zw.to(DEV),
                           y=torch.full((M, cols), float("nan"), dtype=torch.float16, device=DEV),
                           epilogue=epi, residual=None if r is None else r.to(DEV)))
    descs = w4.make_descs(layers)
    w4.w4a16_probe_reset()
    launches0 = w4.w4a16_kernel_launches()
    w4.w4a16_decode_round(descs, M)
    torch.cuda.synchronize()
    assert w4.w4a16_kernel_launches() - launches0 == 1
    assert w4.w4a16_probe_counts()[w4.RUNG_TC_SPLITK] == len(layers)
    for L, ref, (K, N, epi) in zip(layers, refs, specs):
        assert_close(L["y"], ref, f"ragged tc round K={K} N={N} epilogue={epi}")
