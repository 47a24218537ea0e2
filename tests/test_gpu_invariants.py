"""The method's invariants on the GPU kernels, every rung.

The oracle's pins check these invariants on the CPU.  Here they go through
the CUDA library: each forced rung of w4a16_linear (CUDA-core GEMV, warp MMA,
tcgen05, and their split-K forms), the dispatch table's choice, one fused
decode round, and w4a16_linear_ex in fp16 and bf16.
  * q = z everywhere: y = 0.  Exactly 0 on every rung when x holds small
    integers: every partial sum is then an exact multiple of the unpack's
    unit, so the warp-MMA rungs' zero-point fold (sum q x - z sum x) cancels
    exactly.  With N(0, 1) activations the fold leaves rounding noise, held
    to the acceptance rule against the oracle's exact 0.
  * One nonzero group (q = z in every other group): y = s * sum_k (q - z) x
    over that group alone.  The GPU is checked against the oracle, and the
    oracle against that closed form.
  * Linearity: y(x1 + x2) against y(x1) + y(x2) on fp16-exact grids.
    Scaling is bit-exact: y(2^p x) = 2^p y(x) wherever both outputs are
    normal fp16 values.  Every product and partial sum scales exactly, and
    the bf16 staging picks its power of two from each token's largest
    exponent.
  * Special scales (negative, subnormal 0x0001 and 0x03FF, and 65504) and
    special activations (+-65504, subnormal), against the oracle.

The method's definition: forum.sourcefind.cn thread "vLLM on Hygon Z100",
section 四 (w = (q - z) * s per group, y = x w^T).
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic_inputs as si
from helpers import RTOL_BF16_TC, assert_close

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
RUNGS = [-1, 0, 1, 2, 3, 4, 5]  # auto, gemv, gemv_splitk, tc, tc_splitk, mma, mma_splitk


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


# ---------------------------------------------------------------------------
# building cases from unpacked values (packed by the oracle's packer)
# ---------------------------------------------------------------------------
def _pack(q, z):
    qw, zw = oracle.pack(q, z)
    return torch.from_numpy(qw.view(np.int32)), torch.from_numpy(zw.view(np.int32))


def _f16(a):
    return torch.from_numpy(np.asarray(a, dtype=np.float16))


def _bits16(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _ref(x, qw, s, zw, dtype="f16"):
    return oracle.linear(_bits16(x), si.as_u32(qw), _bits16(s), si.as_u32(zw), dtype=dtype)


def _run(w4, rung, x, qw, s, zw):
    """y on a forced rung (None when the rung cannot run the shape)."""
    M, N = x.shape[0], qw.shape[0]
    y = torch.full((M, N), float("nan"), dtype=x.dtype, device=DEV)
    prev = w4.w4a16_set_forced_rung(rung)
    try:
        if rung >= 0:
            w4.w4a16_probe_reset()
        w4.w4a16_linear(x.to(DEV), qw.to(DEV), s.to(DEV), zw.to(DEV), y=y)
        if rung >= 0:
            assert w4.w4a16_probe_counts()[rung] >= 1
    except w4.W4A16Error as e:
        if e.status == w4.W4A16_ERR_UNSUPPORTED:
            return None
        raise
    finally:
        w4.w4a16_set_forced_rung(prev)
    torch.cuda.synchronize()
    return y


def _rng(tag):
    return np.random.default_rng(abs(hash(tag)) % (1 << 32))


def _scales(rng, N, G, lo=0.002, hi=0.02, signed=False):
    v = rng.uniform(lo, hi, (N, G))
    if signed:
        v *= np.where(rng.random((N, G)) < 0.5, -1.0, 1.0)
    return _f16(v)


SHAPES = [(1, 300, 1024), (4, 300, 1024), (8, 77, 2048), (16, 200, 1024)]


# ---------------------------------------------------------------------------
# q = z  =>  y = 0
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("rung", RUNGS)
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_q_equals_z_gives_zero(w4, rung, M, N, K):
    rng = np.random.default_rng(1000 + M * 7 + N + K)
    G = K // 128
    z = rng.integers(0, 16, (N, G), dtype=np.uint8)
    q = np.repeat(z, 128, axis=1)
    qw, zw = _pack(q, z)
    s = _scales(rng, N, G, signed=True)
    # small integers: every partial sum is exact, so y is exactly 0
    xi = _f16(rng.integers(-3, 4, (M, K)))
    y = _run(w4, rung, xi, qw, s, zw)
    if y is None:
        pytest.skip("the forced rung cannot run this shape")
    assert torch.count_nonzero(y.float()) == 0, f"rung {rung}: q = z left nonzero outputs"
    # N(0, 1) activations: the oracle's 0 within the acceptance rule
    xn = si.x(si.config_seed(80, M, N % 16), M, K)
    y = _run(w4, rung, xn, qw, s, zw)
    ref = _ref(xn, qw, s, zw)
    assert np.count_nonzero(ref) == 0
    assert_close(y, ref, f"q = z, N(0,1) x, rung {rung}")


# ---------------------------------------------------------------------------
# one nonzero group
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("rung", RUNGS)
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_single_nonzero_group(w4, rung, M, N, K):
    rng = np.random.default_rng(2000 + M * 7 + N + K)
    G = K // 128
    g_star = int(rng.integers(0, G))
    z = rng.integers(0, 16, (N, G), dtype=np.uint8)
    q = np.repeat(z, 128, axis=1)
    sl = slice(128 * g_star, 128 * (g_star + 1))
    q[:, sl] = rng.integers(0, 16, (N, 128), dtype=np.uint8)
    qw, zw = _pack(q, z)
    s = _scales(rng, N, G, signed=True)
    x = si.x(si.config_seed(81, M, g_star), M, K)
    ref = _ref(x, qw, s, zw)
    # the oracle against the closed form s * sum_{k in g*} (q - z) x
    d = q[:, sl].astype(np.float64) - z[:, g_star:g_star + 1].astype(np.float64)
    closed = (x.double().numpy()[:, sl] @ d.T) * s.double().numpy()[:, g_star][None, :]
    assert np.allclose(ref, closed, rtol=1e-12, atol=1e-300)
    y = _run(w4, rung, x, qw, s, zw)
    if y is None:
        pytest.skip("the forced rung cannot run this shape")
    assert_close(y, ref, f"single group {g_star}, rung {rung}")


# ---------------------------------------------------------------------------
# linearity, and exact scaling by powers of two
# ---------------------------------------------------------------------------
def _normal_mask(a, b):
    """Outputs where both values are normal, finite fp16 numbers."""
    lo = 2.0 ** -14
    return (np.abs(a) >= lo) & (np.abs(b) >= lo) & np.isfinite(a) & np.isfinite(b)


@pytest.mark.parametrize("rung", RUNGS)
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_linearity_and_exact_scaling(w4, rung, M, N, K):
    rng = np.random.default_rng(3000 + M * 7 + N + K)
    seed = si.config_seed(82, M, N % 16)
    qw, s, zw = si.layer(seed, N, K)
    # grids on which x1 + x2 is exact in fp16: multiples of 2^-6 up to 8
    x1 = _f16(rng.integers(-512, 513, (M, K)) / 64.0)
    x2 = _f16(rng.integers(-512, 513, (M, K)) / 64.0)
    x12 = _f16(x1.double().numpy() + x2.double().numpy())
    ys = [_run(w4, rung, x, qw, s, zw) for x in (x1, x2, x12)]
    if ys[0] is None:
        pytest.skip("the forced rung cannot run this shape")
    r1, r2, r12 = (_ref(x, qw, s, zw) for x in (x1, x2, x12))
    assert np.allclose(r12, r1 + r2, rtol=1e-12, atol=1e-9)  # the oracle is linear
    for y, r, what in zip(ys, (r1, r2, r12), ("x1", "x2", "x1 + x2")):
        assert_close(y, r, f"linearity {what}, rung {rung}")
    # y(x1 + x2) - y(x1) - y(x2): only the three outputs' own rounding
    a = ys[2].double().cpu().numpy()
    b = ys[0].double().cpu().numpy() + ys[1].double().cpu().numpy()
    tol = 3 * (1e-3 * np.abs(r12).max() + 1e-3)
    assert np.abs(a - b).max() <= tol
    # exact scaling: y(8 x) == 8 y(x) bit for bit where both are normal fp16
    x = si.x(seed, M, K)
    xs = _f16(x.double().numpy() * 8.0)
    y = _run(w4, rung, x, qw, s, zw).double().cpu().numpy()
    y8 = _run(w4, rung, xs, qw, s, zw).double().cpu().numpy()
    mask = _normal_mask(y * 8.0, y8) & (np.abs(y * 8.0) < 65504)
    assert mask.mean() > 0.9
    assert np.array_equal(y8[mask], 8.0 * y[mask]), f"rung {rung}: y(8x) != 8 y(x)"


# ---------------------------------------------------------------------------
# special scales and activations
# ---------------------------------------------------------------------------
def _special_scale_case(M, N, K, kind):
    rng = np.random.default_rng(4000 + M + N + K + len(kind))
    G = K // 128
    seed = si.config_seed(83, M, len(kind))
    qw, _, zw = si.layer(seed, N, K)
    x = si.x(seed, M, K).double().numpy()
    if kind == "subnormal":
        # every scale a subnormal fp16 of either sign, 0x0001 and 0x03FF among
        # them; x times 2^10 (exact) so that y is far above the absolute term
        bits = rng.integers(1, 0x400, (N, G)).astype(np.uint16)
        bits[0, 0], bits[-1, -1] = 0x0001, 0x03FF
        bits |= (rng.random((N, G)) < 0.5).astype(np.uint16) << 15
        s = torch.from_numpy(bits.view(np.float16))
        x = x * 1024.0
    else:
        # scales of both signs, with 65504 and -65504 in a few (row, group)
        # places; x times 2^-10 keeps the outputs finite
        v = rng.uniform(0.002, 0.02, (N, G)) * np.where(rng.random((N, G)) < 0.5, -1.0, 1.0)
        for r in range(0, N, max(1, N // 5)):
            v[r, int(rng.integers(0, G))] = 65504.0 if r % 2 == 0 else -65504.0
        s = _f16(v)
        x = x / 1024.0
    return _f16(x), qw, s, zw


def _special_x_case(M, N, K):
    rng = np.random.default_rng(5000 + M + N + K)
    seed = si.config_seed(84, M, 0)
    qw, s, zw = si.layer(seed, N, K)
    x = si.x(seed, M, K).view(torch.int16).numpy().copy()
    for m in range(M):
        ks = rng.choice(K, 6, replace=False)
        x[m, ks[0]] = 0x7BFF                 # 65504
        x[m, ks[1]] = np.int16(-0x0401)      # -65504 (0xFBFF)
        x[m, ks[2]] = 0x0001                 # smallest subnormal
        x[m, ks[3]] = 0x03FF                 # largest subnormal
        x[m, ks[4]] = np.int16(-0x7FFF)      # -2^-24 (0x8001)
        x[m, ks[5]] = np.int16(-0x7C01)      # -(1023 * 2^-24) (0x83FF)
    return torch.from_numpy(x).view(torch.float16), qw, s, zw


@pytest.mark.parametrize("rung", RUNGS)
@pytest.mark.parametrize("kind", ["subnormal", "large_negative", "x_extremes"])
@pytest.mark.parametrize("M,N,K", [(4, 300, 1024), (16, 200, 1024)])
def test_special_values(w4, rung, kind, M, N, K):
    if kind == "x_extremes":
        x, qw, s, zw = _special_x_case(M, N, K)
    else:
        x, qw, s, zw = _special_scale_case(M, N, K, kind)
    ref = _ref(x, qw, s, zw)
    assert np.isfinite(ref).all() and np.abs(ref).max() < 60000
    y = _run(w4, rung, x, qw, s, zw)
    if y is None:
        pytest.skip("the forced rung cannot run this shape")
    assert_close(y, ref, f"{kind}, rung {rung}")


# ---------------------------------------------------------------------------
# the same invariants through a fused decode round and w4a16_linear_ex
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("M", [1, 4, 8])
def test_invariants_in_a_fused_round(w4, M):
    N, K = 300, 1024
    rng = np.random.default_rng(6000 + M)
    G = K // 128
    z = rng.integers(0, 16, (N, G), dtype=np.uint8)
    qz, zz = _pack(np.repeat(z, 128, axis=1), z)
    cases = []
    xi = _f16(rng.integers(-3, 4, (M, K)))
    cases.append(("q = z", xi, qz, _scales(rng, N, G, signed=True), zz))
    q1 = np.repeat(z, 128, axis=1)
    q1[:, 256:384] = rng.integers(0, 16, (N, 128), dtype=np.uint8)
    qw1, zw1 = _pack(q1, z)
    cases.append(("one group", si.x(si.config_seed(85, M), M, K), qw1,
                  _scales(rng, N, G, signed=True), zw1))
    for kind in ("subnormal", "large_negative"):
        cases.append((kind,) + _special_scale_case(M, N, K, kind))
    cases.append(("x_extremes",) + _special_x_case(M, N, K))
    layers = []
    for name, x, qw, s, zw in cases:
        layers.append(dict(x=x.to(DEV), qweight=qw.to(DEV), scales=s.to(DEV), zeros=zw.to(DEV),
                           y=torch.full((M, N), float("nan"), dtype=torch.float16, device=DEV)))
    w4.w4a16_probe_reset()
    w4.w4a16_decode_round(w4.make_descs(layers), M)
    torch.cuda.synchronize()
    assert w4.w4a16_kernel_launches() == 1  # one fused launch
    for (name, x, qw, s, zw), L in zip(cases, layers):
        ref = _ref(x, qw, s, zw)
        if name == "q = z":
            assert torch.count_nonzero(L["y"].float()) == 0
        assert_close(L["y"], ref, f"fused round M={M}: {name}")


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("M", [1, 4, 8, 12])
def test_invariants_through_linear_ex(w4, dtype, M):
    N, K = 300, 1024
    name = "bf16" if dtype == torch.bfloat16 else "f16"
    rng = np.random.default_rng(7000 + M)
    G = K // 128
    z = rng.integers(0, 16, (N, G), dtype=np.uint8)
    qw0, zw0 = _pack(np.repeat(z, 128, axis=1), z)
    s = _scales(rng, N, G, signed=True).to(dtype)
    # q = z: exactly zero with small-integer x (exact in both types)
    x = torch.from_numpy(rng.integers(-3, 4, (M, K)).astype(np.float32)).to(dtype)
    y = w4.w4a16_linear_ex(x.to(DEV), qw0.to(DEV), s.to(DEV), zw0.to(DEV))
    torch.cuda.synchronize()
    assert torch.count_nonzero(y.float()) == 0
    # exact scaling by 2^3, and the oracle's linear of the same bits
    qw, s16, zw = si.layer(si.config_seed(86, M), N, K)
    s = s16.float().to(dtype)
    x = si.x(si.config_seed(86, M), M, K).float().to(dtype)
    x8 = (x.float() * 8.0).to(dtype)
    y = w4.w4a16_linear_ex(x.to(DEV), qw.to(DEV), s.to(DEV), zw.to(DEV))
    y8 = w4.w4a16_linear_ex(x8.to(DEV), qw.to(DEV), s.to(DEV), zw.to(DEV))
    torch.cuda.synchronize()
    rtol = RTOL_BF16_TC if dtype == torch.bfloat16 and M > 8 else None  # the tcgen05 rung
    assert_close(y, _ref(x, qw, s, zw, name), f"linear_ex {name} M={M}", rtol=rtol)
    a, b = y.double().cpu().numpy(), y8.double().cpu().numpy()
    lo = 2.0 ** -14 if dtype == torch.float16 else 2.0 ** -126
    mask = (np.abs(8 * a) >= lo) & (np.abs(a) >= lo) & (np.abs(8 * a) < 60000)
    assert mask.mean() > 0.9
    assert np.array_equal(b[mask], 8.0 * a[mask]), f"{name}: y(8x) != 8 y(x)"
