"""GPU parity: the CUDA library, called through its C ABI, against the oracle.

Bit-exact for pack, unpack and dequant; within the stated tolerance for y on
every rung; bit-exact for y in the integer special case; run-to-run
bit-identical per rung.  Inputs come from ``synthetic_inputs`` (the only code
the two sides share).
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic_inputs as si
from helpers import RTOL_BF16_TC, Case, assert_close, sample_rows, sampled_reference

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
CC_RUNGS = [0, 1]  # gemv, gemv_splitk
TC_RUNGS = [2, 3]  # tc, tc_splitk
MMA_RUNGS = [4, 5]  # mma, mma_splitk
ALL_RUNGS = CC_RUNGS + TC_RUNGS + MMA_RUNGS


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


def forced(w4, rung):
    class _Ctx:
        def __enter__(self):
            self.prev = w4.w4a16_set_forced_rung(rung)

        def __exit__(self, *a):
            w4.w4a16_set_forced_rung(self.prev)
    return _Ctx()


def run_linear(w4, case, poison=True):
    x, qw, s, zw = case.to(DEV)
    y = torch.full((case.M, case.N), float("nan"), dtype=torch.float16, device=DEV) if poison else None
    y = w4.w4a16_linear(x, qw, s, zw, y=y)
    torch.cuda.synchronize()
    return y


# ---------------------------------------------------------------------------
# generator: the same bits on the device as on the host
# ---------------------------------------------------------------------------
def test_synthetic_generator_device_equals_host():
    seed = si.config_seed(3, 5, 2)
    qh, sh, zh = si.layer(seed, 300, 1152)
    qd, sd, zd = si.layer(seed, 300, 1152, device=DEV)
    assert torch.equal(qd.cpu(), qh) and torch.equal(zd.cpu(), zh)
    assert torch.equal(sd.cpu().view(torch.int16), sh.view(torch.int16))


# ---------------------------------------------------------------------------
# pack / unpack / dequant: bit-exact
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("N,K", [(1, 128), (7, 384), (64, 1152), (1000, 5120), (33, 17408)])
def test_pack_unpack_bit_exact(w4, N, K):
    rng = np.random.default_rng(N * 7 + K)
    q = rng.integers(0, 16, (N, K), dtype=np.uint8)
    z = rng.integers(0, 16, (N, K // 128), dtype=np.uint8)
    qw_ref, zw_ref = oracle.pack(q, z)
    qw, zw = w4.w4a16_pack(torch.from_numpy(q).to(DEV), torch.from_numpy(z).to(DEV))
    torch.cuda.synchronize()
    assert np.array_equal(si.as_u32(qw), qw_ref)
    assert np.array_equal(si.as_u32(zw), zw_ref)
    q2, z2 = w4.w4a16_unpack(qw, zw, K)
    torch.cuda.synchronize()
    assert np.array_equal(q2.cpu().numpy(), q) and np.array_equal(z2.cpu().numpy(), z)


def test_pack_masks_high_bits(w4):
    rng = np.random.default_rng(5)
    q = rng.integers(0, 256, (9, 256), dtype=np.uint8)
    z = rng.integers(0, 256, (9, 2), dtype=np.uint8)
    qw_ref, zw_ref = oracle.pack(q & 15, z & 15)
    qw, zw = w4.w4a16_pack(torch.from_numpy(q).to(DEV), torch.from_numpy(z).to(DEV))
    torch.cuda.synchronize()
    assert np.array_equal(si.as_u32(qw), qw_ref) and np.array_equal(si.as_u32(zw), zw_ref)


@pytest.mark.parametrize("N,K", [(256, 128), (37, 1152), (515, 5120)])
def test_dequant_bit_exact(w4, N, K):
    seed = si.config_seed(50, 1, N)
    qw, s, zw = si.layer(seed, N, K)
    # include negative, subnormal and extreme scales
    sb = s.view(torch.int16).clone()
    special = torch.tensor([0x0001, 0x03FF, -0x8000 + 0x0001, 0x7BFF, -0x8000 + 0x3C00, 0x0400],
                           dtype=torch.int16)
    sb.view(-1)[: special.numel()] = special
    s = sb.view(torch.float16)
    w_exact = oracle.dequant(si.as_u32(qw), si.as_u16(s), si.as_u32(zw), K)
    w32, w16 = w4.w4a16_dequant(qw.to(DEV), s.to(DEV), zw.to(DEV), K)
    torch.cuda.synchronize()
    assert np.array_equal(w32.cpu().numpy(), w_exact.astype(np.float32))
    assert np.array_equal(w32.cpu().numpy().astype(np.float64), w_exact)  # exact in fp32
    assert np.array_equal(si.as_u16(w16), oracle.double_to_half(w_exact))


# ---------------------------------------------------------------------------
# linear: tolerance on every rung, seeded shapes spanning tiles and ragged tails
# ---------------------------------------------------------------------------
SHAPES = [(1, 1, 128), (1, 7, 256), (1, 1024, 512), (2, 1029, 1152), (3, 64, 5120),
          (4, 1000, 2048), (5, 130, 384), (6, 257, 640), (7, 96, 1024), (8, 513, 4352),
          (8, 2000, 17408), (12, 300, 1024), (20, 77, 768), (64, 200, 512)]


@pytest.mark.parametrize("rung", ALL_RUNGS + [-1])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_linear_matches_oracle(w4, rung, M, N, K):
    case = Case(si.config_seed(51, M, N % 16), M, N, K)
    if rung in (w4.RUNG_GEMV_SPLITK, w4.RUNG_TC_SPLITK, w4.RUNG_MMA_SPLITK) and K // 128 < 2:
        pytest.skip("split-K needs two groups")
    with forced(w4, rung):
        if rung >= 0:
            w4.w4a16_probe_reset()
        try:
            y = run_linear(w4, case)
        except w4.W4A16Error as e:
            if rung in (w4.RUNG_GEMV, w4.RUNG_MMA) and e.status == w4.W4A16_ERR_UNSUPPORTED:
                pytest.skip("shape needs split-K on this rung")
            raise
        if rung >= 0:
            assert w4.w4a16_probe_counts()[rung] >= 1
    assert_close(y, case.reference(), f"rung {rung} M={M} N={N} K={K}")


@pytest.mark.parametrize("rung", ALL_RUNGS)
def test_integer_case_bit_exact(w4, rung):
    # s = 1/16 and x in {-1, 0, 1}: every partial sum is an exact integer
    # multiple of 1/16 far below 2^24, so y is exact on every rung.
    M, N, K = 8, 700, 2048
    rng = np.random.default_rng(11)
    q = rng.integers(0, 16, (N, K), dtype=np.uint8)
    z = rng.integers(0, 16, (N, K // 128), dtype=np.uint8)
    X = rng.integers(-1, 2, (M, K)).astype(np.int64)
    qw, zw = oracle.pack(q, z)
    s = np.full((N, K // 128), 0x2C00, dtype=np.uint16)
    W = q.astype(np.int64) - np.repeat(z.astype(np.int64), 128, axis=1)
    want = (X @ W.T).astype(np.float64) / 16
    assert np.abs(want).max() < 2048
    x = torch.from_numpy(X.astype(np.float16)).to(DEV)
    with forced(w4, rung):
        try:
            y = w4.w4a16_linear(x, torch.from_numpy(qw.view(np.int32)).to(DEV),
                                torch.from_numpy(s.view(np.float16)).to(DEV),
                                torch.from_numpy(zw.view(np.int32)).to(DEV))
        except w4.W4A16Error as e:
            if e.status == w4.W4A16_ERR_UNSUPPORTED:
                pytest.skip("rung cannot run this shape")
            raise
    torch.cuda.synchronize()
    assert np.array_equal(y.float().cpu().numpy().astype(np.float64), want)


@pytest.mark.parametrize("rung", ALL_RUNGS)
def test_run_to_run_bit_identical(w4, rung):
    case = Case(si.config_seed(52), 4, 5120, 17408)
    with forced(w4, rung):
        try:
            a = run_linear(w4, case)
        except w4.W4A16Error:
            pytest.skip("rung cannot run this shape")
        b = run_linear(w4, case)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("M,N,K", [(4, 34816, 5120), (4, 5120, 17408), (1, 8192, 5120)])
def test_repeated_runs_bit_identical_and_sampled(w4, M, N, K):
    # A race between the kernels' shared-memory reads and the asynchronous
    # copies that refill the same buffers changes a few outputs in some runs
    # only: launch the same linear ten times back to back (no host sync in
    # between), then require every run to equal the first bit for bit, and
    # the first to match the oracle on sampled rows.
    seed = si.config_seed(54, 0, M)
    qw, s, zw = si.layer(seed, N, K, device=DEV)
    x_cpu = si.x(seed, M, K)
    x = x_cpu.to(DEV)
    outs = []
    for _ in range(10):
        y = torch.full((M, N), float("nan"), dtype=torch.float16, device=DEV)
        w4.w4a16_linear(x, qw, s, zw, y=y)
        outs.append(y)
    torch.cuda.synchronize()
    for i, y in enumerate(outs[1:], 1):
        diff = int((y.view(torch.int16) != outs[0].view(torch.int16)).sum())
        assert diff == 0, f"run {i} differs from run 0 in {diff} outputs"
    rows = sample_rows(N, 24, seed=N + K)
    ref = sampled_reference(seed, x_cpu, N, K, rows)
    assert_close(outs[0][:, torch.from_numpy(rows).to(DEV)], ref, f"M={M} N={N} K={K}")


def test_varying_sizes_back_to_back(w4):
    # Stale data between calls of different sizes shows only when sizes vary
    # (forum thread "vLLM on Hygon Z100", section 三: the all-reduce bug found
    # only by changing message sizes); launch them all, then check them all.
    rng = np.random.default_rng(12)
    cases, outs = [], []
    for i in range(24):
        M = int(rng.integers(1, 9))
        N = int(rng.integers(1, 1500))
        K = 128 * int(rng.integers(1, 40))
        c = Case(si.config_seed(53, i), M, N, K)
        x, qw, s, zw = c.to(DEV)
        y = torch.full((M, N), float("nan"), dtype=torch.float16, device=DEV)
        w4.w4a16_linear(x, qw, s, zw, y=y)
        cases.append(c)
        outs.append(y)
    torch.cuda.synchronize()
    for c, y in zip(cases, outs):
        assert_close(y, c.reference(), f"M={c.M} N={c.N} K={c.K}")


# ---------------------------------------------------------------------------
# full-size workloads, every output compared
# ---------------------------------------------------------------------------
# The weights are generated on the device by the seeded generator (equal to the
# host's, test_synthetic_generator_device_equals_host) and copied to the host
# for the oracle; the oracle's output for a workload is computed once and
# shared by every rung that runs it.
_FULL_REFS = {}


def _full_reference(key, x_cpu, qw, s, zw):
    if key not in _FULL_REFS:
        _FULL_REFS.clear()  # one workload's reference at a time
        _FULL_REFS[key] = oracle.linear(si.as_u16(x_cpu), si.as_u32(qw), si.as_u16(s),
                                        si.as_u32(zw))
    return _FULL_REFS[key]


@pytest.mark.parametrize("rung", [-1] + ALL_RUNGS)
@pytest.mark.parametrize("M,N,K,cfg", [(1, 34816, 5120, 1), (4, 5120, 17408, 2),
                                       (8, 5120, 17408, 2)])
def test_full_size_full_output(w4, M, N, K, cfg, rung):
    seed = si.config_seed(cfg, 0, M)
    qw, s, zw = si.layer(seed, N, K, device=DEV)
    x = si.x(seed, M, K)
    with forced(w4, rung):
        try:
            y = w4.w4a16_linear(x.to(DEV), qw, s, zw)
        except w4.W4A16Error as e:
            if e.status == w4.W4A16_ERR_UNSUPPORTED:
                pytest.skip("rung cannot run this shape")
            raise
    torch.cuda.synchronize()
    ref = _full_reference((cfg, M), x, qw, s, zw)
    assert_close(y, ref, f"cfg{cfg} M={M} rung {rung}")


@pytest.mark.parametrize("rung", [-1, 2, 5])
@pytest.mark.parametrize("M", [1, 2, 4, 8, 16, 32, 64])
def test_m_sweep_full_output(w4, M, rung):
    N, K = 27648, 5120
    seed = si.config_seed(4)
    qw, s, zw = si.layer(seed, N, K, device=DEV)
    x = si.x(seed, M, K)
    with forced(w4, rung):
        try:
            y = w4.w4a16_linear(x.to(DEV), qw, s, zw)
        except w4.W4A16Error as e:
            if e.status == w4.W4A16_ERR_UNSUPPORTED:
                pytest.skip("rung cannot run this shape")
            raise
    torch.cuda.synchronize()
    ref = _full_reference((4, M), x, qw, s, zw)
    assert_close(y, ref, f"sweep M={M} rung {rung}")


ROUND_SHAPES = [(5120, 8192), (6144, 5120), (5120, 34816), (17408, 5120)]  # (K, N)


def _round(w4, n_layers, M, seed_cfg=3):
    layers = []
    xs = {}
    for j, (K, N) in enumerate(ROUND_SHAPES):
        xs[j] = si.x(si.config_seed(seed_cfg, 0, 8 + j), M, K)
    for l in range(n_layers):
        for j, (K, N) in enumerate(ROUND_SHAPES):
            seed = si.config_seed(seed_cfg, l, j)
            qw, s, zw = si.layer(seed, N, K, device=DEV)
            layers.append(dict(x=xs[j].to(DEV), qweight=qw, scales=s, zeros=zw,
                               y=torch.full((M, N), float("nan"), dtype=torch.float16, device=DEV),
                               seed=seed, N=N, K=K, j=j))
    return layers, xs


def test_decode_round_eager_and_graph(w4):
    M = 4
    layers, xs = _round(w4, 2, M)
    descs = w4.make_descs(layers)
    w4.w4a16_decode_round(descs, M)
    torch.cuda.synchronize()
    eager = [L["y"].clone() for L in layers]
    for L in layers:
        L["y"].fill_(float("nan"))
    g = w4.RoundGraph(descs, M)
    g.launch()
    torch.cuda.synchronize()
    g.destroy()
    for L, e in zip(layers, eager):
        assert torch.equal(L["y"].view(torch.int16), e.view(torch.int16))
        rows = sample_rows(L["N"], 8, seed=L["seed"] & 0xFFFF)
        ref = sampled_reference(L["seed"], xs[L["j"]], L["N"], L["K"], rows)
        assert_close(L["y"][:, torch.from_numpy(rows).to(DEV)], ref, f"round layer j={L['j']}")


@pytest.mark.parametrize("graph", [False, True])
def test_decode_round_chained_waits(w4, graph):
    # Each linear reads the previous one's output (x_l = y_{l-1}), one writes
    # over an earlier one's input (write after read) and the last two write
    # the same output (write after write): the fused round must wait where
    # the results of running the linears one after another require it.
    # Every output is checked against the oracle applied to the input the GPU
    # actually used; the round runs twice (the completion counters must be
    # left zeroed for the next launch).
    M = 4
    dims = [1024, 2048, 1536, 1024, 3072, 2048]
    acts = [torch.zeros((M, d), dtype=torch.float16, device=DEV) for d in dims]
    acts[0].copy_(si.x(si.config_seed(60), M, dims[0]).to(DEV))
    layers = []
    for l in range(len(dims) - 1):
        K, N = dims[l], dims[l + 1]
        seed = si.config_seed(61, l)
        qw, s, zw = si.layer(seed, N, K, device=DEV)
        layers.append(dict(x=acts[l], qweight=qw, scales=s, zeros=zw, y=acts[l + 1], N=N, K=K,
                           seed=seed))
    # write after read: overwrite the first input once the chain has read it
    qw, s, zw = si.layer(si.config_seed(62), dims[0], dims[-1], device=DEV)
    layers.append(dict(x=acts[-1], qweight=qw, scales=s, zeros=zw, y=acts[0], N=dims[0],
                       K=dims[-1], seed=si.config_seed(62)))
    # write after write: a later linear writes the same output; only its
    # result may remain
    qw, s, zw = si.layer(si.config_seed(63), dims[0], dims[2], device=DEV)
    layers.append(dict(x=acts[2], qweight=qw, scales=s, zeros=zw, y=acts[0], N=dims[0],
                       K=dims[2], seed=si.config_seed(63)))
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
            w4.w4a16_decode_round(descs, M)
            torch.cuda.synchronize()
        assert w4.w4a16_device_status() == 0
        chain = [x0] + [acts[l + 1].clone() for l in range(len(dims) - 1)]
        # (input, output) of every linear whose output survives the round
        checks = [(l, chain[l], chain[l + 1]) for l in range(len(dims) - 1)]
        checks.append((len(layers) - 1, chain[2], acts[0].clone()))
        for l, x_used, out in checks:
            L = layers[l]
            x_cpu = x_used.cpu()
            qw_h, s_h, zw_h = si.layer(L["seed"], L["N"], L["K"])
            ref = oracle.linear(si.as_u16(x_cpu), si.as_u32(qw_h), si.as_u16(s_h), si.as_u32(zw_h))
            assert_close(out, ref, f"chained linear {l} rep {rep}")


def _round_reference(L, x_cpu):
    """The oracle's output of one round linear, from its device weights."""
    return oracle.linear(si.as_u16(x_cpu), si.as_u32(L["qweight"]), si.as_u16(L["scales"]),
                         si.as_u32(L["zeros"]))


@pytest.mark.parametrize("M", [1, 8])
def test_decode_round_m1_m8_full_output(w4, M):
    # the round at the other ends of the verify range (M = 4 runs below and
    # in the benchmark): two layers, one fused launch, every output compared
    layers, xs = _round(w4, 2, M)
    descs = w4.make_descs(layers)
    w4.w4a16_probe_reset()
    w4.w4a16_decode_round(descs, M)
    torch.cuda.synchronize()
    assert w4.w4a16_kernel_launches() == 1
    for L in layers:
        assert_close(L["y"], _round_reference(L, xs[L["j"]]), f"M={M} round linear j={L['j']}")


@pytest.mark.slow
def test_decode_round_full_64_layers_full_output(w4):
    # the whole 64-layer round at M = 4: all 256 outputs against the oracle
    M = 4
    layers, xs = _round(w4, 64, M)
    descs = w4.make_descs(layers)
    w4.w4a16_decode_round(descs, M)
    torch.cuda.synchronize()
    # the premise of copying the device weights to the host: the device
    # generator gives the host's bits (checked here on one linear's rows)
    L = layers[-1]
    rows = sample_rows(L["N"], 8, seed=5)
    qh, sh, zh = si.layer(L["seed"], L["N"], L["K"], rows=rows)
    idx = torch.from_numpy(rows).to(DEV)
    assert torch.equal(L["qweight"][idx].cpu(), qh) and torch.equal(L["zeros"][idx].cpu(), zh)
    assert torch.equal(L["scales"][idx].cpu().view(torch.int16), sh.view(torch.int16))
    for i, L in enumerate(layers):
        assert_close(L["y"], _round_reference(L, xs[L["j"]]), f"round linear {i} (j={L['j']})")
        layers[i] = None  # release the layer's weights as we go
    del layers
    torch.cuda.empty_cache()


def test_random_sweep_every_path(w4):
    # seeded random shapes across every dispatch path: M 1..64 (the mma rungs,
    # 8-token tiles and the tcgen05 rung), ragged N, K from one group to 40,
    # fp16 and bf16, each epilogue; all launched, then all checked (stale data
    # between calls of different sizes shows only this way)
    rng = np.random.default_rng(2026)
    cases = []
    for i in range(20):
        M = int(rng.integers(1, 9)) if i % 2 == 0 else int(rng.integers(9, 65))
        K = 128 * int(rng.integers(1, 41))
        epi = int(rng.integers(0, 3))
        dt = torch.bfloat16 if rng.random() < 0.4 else torch.float16
        if epi == w4.EPILOGUE_SILU_MUL:
            N = 32 * int(rng.integers(1, 60))
        else:
            N = int(rng.integers(1, 2000))
        if M > 8 and N > 1024:  # keep the oracle's share of the test short
            N = 1024  # (a multiple of 32, as SiLU-and-mul needs)
        seed = si.config_seed(54, i)
        qw, s, zw = si.layer(seed, N, K)
        x = si.x(seed, M, K).float().to(dt)
        s = s.float().to(dt) if dt == torch.bfloat16 else s
        res = si.residual(seed, M, N).float().to(dt) if epi == w4.EPILOGUE_RESIDUAL else None
        cols = N // 2 if epi == w4.EPILOGUE_SILU_MUL else N
        y = torch.full((M, cols), float("nan"), dtype=dt, device=DEV)
        w4.w4a16_linear_ex(x.to(DEV), qw.to(DEV), s.to(DEV), zw.to(DEV), epilogue=epi,
                           residual=None if res is None else res.to(DEV), y=y)
        cases.append((M, N, K, epi, dt, x, qw, s, zw, res, y))
    torch.cuda.synchronize()
    for M, N, K, epi, dt, x, qw, s, zw, res, y in cases:
        name = "bf16" if dt == torch.bfloat16 else "f16"
        bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
        ref = oracle.linear(bits(x), si.as_u32(qw), bits(s), si.as_u32(zw), dtype=name)
        if epi == w4.EPILOGUE_RESIDUAL:
            ref = oracle.add_residual(ref, bits(res), name)
        elif epi == w4.EPILOGUE_SILU_MUL:
            ref = oracle.silu_mul(ref)
        rtol = RTOL_BF16_TC if name == "bf16" and M > 8 else None  # the tcgen05 rung
        assert_close(y, ref, f"M={M} N={N} K={K} epi={epi} {name}", rtol=rtol)
