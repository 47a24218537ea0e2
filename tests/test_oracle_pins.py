"""Pins for the CPU oracle, against things other than the oracle itself.

Each test fixes one part of the oracle to an independent source: numpy's IEEE
binary16 conversion, closed-form packed words, exact rational arithmetic
(``fractions.Fraction``), an int64 matrix product, or an identity of the
method (w = (q - z) * s per 128-wide group along K, y = x @ w^T; forum
thread "vLLM on Hygon Z100", section 四).  A dropped term, a flipped sign, a
wrong nibble or group index, or a transposed operand in the oracle fails at
least one of them.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle

RNG = np.random.default_rng(20261202)


# ----------------------------------------------------------------------------
# binary16 conversions
# ----------------------------------------------------------------------------
def test_half_to_double_every_pattern():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = oracle.half_to_double(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # signed zeros keep their sign
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def _ties_and_edges():
    v = []
    for e in range(-24, 16):
        # exact binary16 values, midpoints (ties) and points just off them
        for m in range(0, 1024, 37):
            base = np.float64(np.float16(2.0 ** e * (1 + m / 1024.0))) if e >= -14 else None
            if base is None:
                continue
            v.append(base)
            step = 2.0 ** (max(e, -14) - 10)
            v += [base + step / 2, base - step / 2, base + step / 2 * (1 + 2 ** -40),
                  base + step / 2 * (1 - 2 ** -40)]
    for m in range(0, 1024, 7):  # subnormal range, quantum 2^-24
        b = m * 2.0 ** -24
        v += [b, b + 2.0 ** -25, b + 2.0 ** -25 * (1 + 2 ** -30), b + 2.0 ** -26]
    v += [65504.0, 65519.0, 65519.999, 65520.0, 65536.0, 1e10, 2.0 ** -25, 2.0 ** -26,
          3 * 2.0 ** -25, 5 * 2.0 ** -25, 0.0, 1e-300, 2047.5, 2048.5, 2049.0, 2051.0]
    v = np.array(v, dtype=np.float64)
    return np.concatenate([v, -v])


def test_double_to_half_round_to_nearest_even():
    vals = np.concatenate([_ties_and_edges(),
                           RNG.standard_normal(200000) * 10.0 ** RNG.integers(-8, 5, 200000),
                           np.array([np.inf, -np.inf])])
    got = oracle.double_to_half(vals)
    ref = vals.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)
    assert oracle.double_to_half(np.array([np.nan]))[0] & 0x7C00 == 0x7C00


def test_double_to_half_ties_closed_form():
    # 1 + 2^-11 lies halfway between 1 and 1 + 2^-10: ties go to the even one (1.0)
    assert oracle.double_to_half([1 + 2 ** -11])[0] == 0x3C00
    # 1 + 3*2^-11 lies halfway between 1+2^-10 (odd) and 1+2^-9 (even)
    assert oracle.double_to_half([1 + 3 * 2 ** -11])[0] == 0x3C02
    # smallest subnormal is 2^-24; half of it ties to zero, 1.5 of it to 2^-23
    assert oracle.double_to_half([2 ** -25])[0] == 0x0000
    assert oracle.double_to_half([3 * 2 ** -25])[0] == 0x0002
    assert oracle.double_to_half([65504.0])[0] == 0x7BFF
    assert oracle.double_to_half([65520.0])[0] == 0x7C00


# ----------------------------------------------------------------------------
# pack / unpack
# ----------------------------------------------------------------------------
def test_pack_closed_form_words():
    # q[n, k] = k mod 16 puts nibble j of word w at value 8w + j: little-endian
    # nibble order gives these literal words.
    K = 16
    q = np.tile(np.arange(K, dtype=np.uint8) % 16, (2, 1))
    z = np.zeros((2, 1), dtype=np.uint8)
    z[1, 0] = 9
    qw, zw = oracle.pack(q, z, group=16)
    assert qw.tolist() == [[0x76543210, 0xFEDCBA98]] * 2
    assert zw.tolist() == [[0x0], [0x9]]
    # three groups in one zeros word, pad nibbles left at zero
    q3 = np.zeros((1, 3 * 128), dtype=np.uint8)
    z3 = np.array([[1, 2, 3]], dtype=np.uint8)
    _, zw3 = oracle.pack(q3, z3, group=128)
    assert zw3.tolist() == [[0x00000321]]
    # nine groups need two words per row
    q9 = np.zeros((1, 9 * 128), dtype=np.uint8)
    z9 = np.array([[1, 2, 3, 4, 5, 6, 7, 8, 15]], dtype=np.uint8)
    _, zw9 = oracle.pack(q9, z9, group=128)
    assert zw9.tolist() == [[0x87654321, 0x0000000F]]


def test_pack_unpack_round_trip_every_nibble_everywhere():
    N, K = 16, 256
    n = np.arange(N)[:, None]
    k = np.arange(K)[None, :]
    q = ((n + k) % 16).astype(np.uint8)          # every value at every nibble position
    z = ((n + np.arange(K // 128)[None, :] * 5) % 16).astype(np.uint8)
    qw, zw = oracle.pack(q, z)
    q2, z2 = oracle.unpack(qw, zw, K)
    assert np.array_equal(q, q2) and np.array_equal(z, z2)


def test_unpack_pack_round_trip_random_words():
    N, K = 37, 1152  # G = 9: two zero words per row, 7 pad nibbles
    qw = RNG.integers(0, 1 << 32, (N, K // 8), dtype=np.uint64).astype(np.uint32)
    zw = RNG.integers(0, 1 << 32, (N, 2), dtype=np.uint64).astype(np.uint32)
    zw[:, 1] &= 0xF
    q, z = oracle.unpack(qw, zw, K)
    assert q.max() <= 15 and z.max() <= 15
    qw2, zw2 = oracle.pack(q, z)
    assert np.array_equal(qw, qw2) and np.array_equal(zw, zw2)


# ----------------------------------------------------------------------------
# dequant
# ----------------------------------------------------------------------------
SCALE_BITS = np.array([0x3C00, 0x2C00, 0x1C18, 0x0001, 0x03FF, 0x7BFF, 0xBC00,
                       0x8001, 0x2419, 0x211F], dtype=np.uint16)


def test_dequant_all_q_z_pairs_exact():
    K = 128
    qs, zs = np.meshgrid(np.arange(16), np.arange(16), indexing="ij")
    qs, zs = qs.reshape(-1), zs.reshape(-1)
    N = qs.size
    q = np.repeat(qs[:, None], K, axis=1).astype(np.uint8)
    z = zs[:, None].astype(np.uint8)
    qw, zw = oracle.pack(q, z)
    for sb in SCALE_BITS:
        s = np.full((N, 1), sb, dtype=np.uint16)
        w = oracle.dequant(qw, s, zw, K)
        s_exact = Fraction(float(np.uint16(sb).view(np.float16)))
        for i in range(N):
            want = (int(qs[i]) - int(zs[i])) * s_exact
            assert Fraction(w[i, 0]) == want
            assert np.all(w[i] == w[i, 0])


def test_dequant_group_index():
    # Distinct scale and zero per group: element k must use group k // 128.
    K, N = 512, 3
    q = RNG.integers(0, 16, (N, K)).astype(np.uint8)
    z = RNG.integers(0, 16, (N, K // 128)).astype(np.uint8)
    s = np.array([[0x3C00, 0x4000, 0x4200, 0x4400]] * N, dtype=np.uint16)  # 1, 2, 3, 4
    qw, zw = oracle.pack(q, z)
    w = oracle.dequant(qw, s, zw, K)
    g = np.arange(K) // 128
    want = (q.astype(np.int64) - z[:, g]) * (g + 1)[None, :]
    assert np.array_equal(w, want.astype(np.float64))


# ----------------------------------------------------------------------------
# linear
# ----------------------------------------------------------------------------
def _f16_bits(a):
    return np.asarray(a, dtype=np.float16).view(np.uint16)


def _brute_force_exact(xb, q, z, sb, group):
    """Exact rational y[m, n] from UNPACKED q, z (no nibble logic involved)."""
    M, K = xb.shape
    N = q.shape[0]
    xf = [[Fraction(float(v)) for v in row] for row in xb.view(np.float16)]
    sf = [[Fraction(float(v)) for v in row] for row in sb.view(np.float16)]
    y = [[Fraction(0)] * N for _ in range(M)]
    mag = [[Fraction(0)] * N for _ in range(M)]
    for m in range(M):
        for n in range(N):
            acc = Fraction(0)
            a = Fraction(0)
            for k in range(K):
                g = k // group
                t = xf[m][k] * (int(q[n, k]) - int(z[n, g])) * sf[n][g]
                acc += t
                a += abs(t)
            y[m][n] = acc
            mag[m][n] = a
    return y, mag


@pytest.mark.parametrize("M,N,K,group", [(1, 1, 128, 128), (2, 3, 256, 128),
                                         (3, 8, 256, 256), (2, 5, 384, 128)])
def test_linear_matches_exact_rationals(M, N, K, group):
    G = K // group
    q = RNG.integers(0, 16, (N, K)).astype(np.uint8)
    z = RNG.integers(0, 16, (N, G)).astype(np.uint8)
    sb = _f16_bits(RNG.uniform(0.002, 0.02, (N, G)))
    xb = _f16_bits(RNG.standard_normal((M, K)))
    qw, zw = oracle.pack(q, z, group)
    y = oracle.linear(xb, qw, sb, zw, group)
    ye, mag = _brute_force_exact(xb, q, z, sb, group)
    for m in range(M):
        for n in range(N):
            err = abs(Fraction(y[m, n]) - ye[m][n])
            assert err <= Fraction(1, 10 ** 12) * (mag[m][n] + Fraction(1, 10 ** 30))
    # sampled rows agree bit for bit with the full product
    rows = np.array([N - 1, 0] if N > 1 else [0])
    yr = oracle.linear_rows(xb, qw, sb, zw, rows, group)
    assert np.array_equal(yr, y[:, rows])


def test_q_equal_z_gives_zero():
    M, N, K = 3, 6, 512
    z = RNG.integers(0, 16, (N, K // 128)).astype(np.uint8)
    q = np.repeat(z, 128, axis=1)
    sb = _f16_bits(RNG.uniform(0.002, 0.02, (N, K // 128)))
    xb = _f16_bits(RNG.standard_normal((M, K)))
    qw, zw = oracle.pack(q, z)
    y = oracle.linear(xb, qw, sb, zw)
    assert np.array_equal(y, np.zeros((M, N)))


def test_single_nonzero_group_closed_form():
    # Every group but g* has q == z, so y[m, n] = s[n, g*] * sum_{k in g*} (q - z) x.
    M, N, K, gstar = 2, 4, 640, 3
    G = K // 128
    z = RNG.integers(0, 16, (N, G)).astype(np.uint8)
    q = np.repeat(z, 128, axis=1)
    q[:, gstar * 128:(gstar + 1) * 128] = RNG.integers(0, 16, (N, 128))
    sb = _f16_bits(RNG.uniform(0.002, 0.02, (N, G)))
    # x on a grid of small dyadic values: every partial sum is exact in binary64
    xv = RNG.integers(-64, 65, (M, K)) / 32.0
    xb = _f16_bits(xv)
    qw, zw = oracle.pack(q, z)
    y = oracle.linear(xb, qw, sb, zw)
    d = q[:, gstar * 128:(gstar + 1) * 128].astype(np.int64) - z[:, gstar:gstar + 1]
    s = sb.view(np.float16).astype(np.float64)[:, gstar]
    want = (xv[:, gstar * 128:(gstar + 1) * 128] @ d.T.astype(np.float64)) * s[None, :]
    assert np.array_equal(y, want)


def test_linearity_in_x():
    M, N, K = 2, 5, 384
    q = RNG.integers(0, 16, (N, K)).astype(np.uint8)
    z = RNG.integers(0, 16, (N, K // 128)).astype(np.uint8)
    sb = _f16_bits(RNG.uniform(0.002, 0.02, (N, K // 128)))
    qw, zw = oracle.pack(q, z)
    x1 = RNG.integers(-256, 257, (M, K)) / 64.0   # sums stay exact in binary16
    x2 = RNG.integers(-256, 257, (M, K)) / 64.0
    y1 = oracle.linear(_f16_bits(x1), qw, sb, zw)
    y2 = oracle.linear(_f16_bits(x2), qw, sb, zw)
    y12 = oracle.linear(_f16_bits(x1 + x2), qw, sb, zw)
    assert np.allclose(y12, y1 + y2, rtol=0, atol=1e-12 * np.abs(y1).max())
    # powers of two scale every product and sum exactly
    xr = RNG.standard_normal((M, K))
    yb = oracle.linear(_f16_bits(xr), qw, sb, zw)
    y8 = oracle.linear(_f16_bits(np.float16(xr).astype(np.float64) * 8), qw, sb, zw)
    assert np.array_equal(y8, 8 * yb)


@pytest.mark.parametrize("s_bits,s_val", [(0x2C00, 1 / 16), (0x3C00, 1.0)])
def test_integer_case_equals_int64_matmul(s_bits, s_val):
    # s a power of two and x in {-1, 0, 1}: y = s * (X @ (Q - Z)^T) exactly.
    M, N, K = 4, 9, 1024
    q = RNG.integers(0, 16, (N, K)).astype(np.uint8)
    z = RNG.integers(0, 16, (N, K // 128)).astype(np.uint8)
    X = RNG.integers(-1, 2, (M, K)).astype(np.int64)
    sb = np.full((N, K // 128), s_bits, dtype=np.uint16)
    qw, zw = oracle.pack(q, z)
    y = oracle.linear(_f16_bits(X), qw, sb, zw)
    W = q.astype(np.int64) - np.repeat(z.astype(np.int64), 128, axis=1)
    want = (X @ W.T).astype(np.float64) * s_val
    assert np.array_equal(y, want)


def test_hand_worked_example():
    # K = 128, one output row, one token: q = 3 on the first 64 k, 10 on the rest,
    # z = 5, s = 0.5, x = 1 on even k and -2 on odd k.
    #   sum over k<64:  (3-5)*0.5 * (32*1 + 32*(-2)) = -1 * (-32) = 32
    #   sum over k>=64: (10-5)*0.5 * (-32)           = 2.5 * (-32) = -80
    #   y = -48
    q = np.array([[3] * 64 + [10] * 64], dtype=np.uint8)
    z = np.array([[5]], dtype=np.uint8)
    s = np.array([[0x3800]], dtype=np.uint16)  # 0.5
    xb = _f16_bits([[1.0 if k % 2 == 0 else -2.0 for k in range(128)]])
    qw, zw = oracle.pack(q, z)
    assert oracle.linear(xb, qw, s, zw)[0, 0] == -48.0


def test_golden_fixture_reproduces_bit_for_bit():
    # Stored by tests/golden/make_golden.py (oracle only); pins the oracle's
    # binary64 results across host architectures.
    import json
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "oracle_linear_small.json")
    data = json.load(open(path))
    for c in data["cases"]:
        M, N, K = c["M"], c["N"], c["K"]
        G = K // 128
        x = np.array(c["x_f16_bits"], dtype=np.uint16).reshape(M, K)
        qw = np.array(c["qweight_u32"], dtype=np.uint32).reshape(N, K // 8)
        s = np.array(c["scales_f16_bits"], dtype=np.uint16).reshape(N, G)
        zw = np.array(c["zeros_u32"], dtype=np.uint32).reshape(N, (G + 7) // 8)
        y = oracle.linear(x, qw, s, zw, nthreads=2)
        want = np.array([float.fromhex(h) for h in c["y_f64_hex"]]).reshape(M, N)
        assert np.array_equal(y, want)


# ----------------------------------------------------------------------------
# epilogues: SiLU-and-mul after the fused gate+up projection (forum thread
# "vLLM on Hygon Z100", section 二) and the residual add after an output
# projection (V100 article, third round of changes)
# ----------------------------------------------------------------------------
def test_silu_mul_closed_forms():
    # silu(g) = g * sigmoid(g); sigmoid(ln 3) = 3/4, sigmoid(-ln 3) = 1/4,
    # sigmoid(0) = 1/2: closed forms that need no exponential on this side.
    import math
    l3 = math.log(3.0)
    gate = [0.0, l3, -l3, 0.0, l3]
    up = [7.0, 1.0, 1.0, -3.0, -2.0]
    got = oracle.silu_mul(np.array([gate + up]))[0]
    want = [0.0, 0.75 * l3, -0.25 * l3, 0.0, -1.5 * l3]
    assert np.allclose(got, want, rtol=4e-16, atol=0.0)
    assert got[0] == 0.0 and got[3] == 0.0


def test_silu_mul_odd_part_identity():
    # silu(g) - silu(-g) = g * (sigmoid(g) + sigmoid(-g)) = g for every g
    g = RNG.uniform(-30.0, 30.0, size=257)
    one = np.ones_like(g)
    pos = oracle.silu_mul(np.concatenate([g, one])[None, :])[0]
    neg = oracle.silu_mul(np.concatenate([-g, one])[None, :])[0]
    assert np.allclose(pos - neg, g, rtol=0.0, atol=1e-13)
    # large gates saturate: silu(g) -> g, silu(-g) -> 0
    assert np.allclose(pos[g > 25], g[g > 25], rtol=1e-10)


def test_silu_mul_column_split_and_rows():
    # gate is the first half of the columns, up the second; each output column
    # sees only its own (gate, up) pair, each row only its own row; the output
    # is linear in up
    M, I = 3, 40
    y = RNG.normal(size=(M, 2 * I))
    out = oracle.silu_mul(y)
    assert out.shape == (M, I)
    perm = RNG.permutation(I)
    yp = np.concatenate([y[:, :I][:, perm], y[:, I:][:, perm]], axis=1)
    assert np.array_equal(oracle.silu_mul(yp), out[:, perm])
    assert np.array_equal(oracle.silu_mul(y[::-1].copy()), out[::-1])
    y2 = y.copy()
    y2[:, I:] *= 2.0
    assert np.array_equal(oracle.silu_mul(y2), 2.0 * out)
    # up = 1 gives silu(gate) alone, which is positive for positive gates and
    # never below its minimum (about -0.2785)
    y1 = y.copy()
    y1[:, I:] = 1.0
    s = oracle.silu_mul(y1)
    assert np.all((s > 0) == (y[:, :I] > 0))
    assert s.min() > -0.2785


def test_add_residual_exact():
    # dyadic y and binary16 residuals: the binary64 sum is exact, so it must
    # equal the rational sum
    n = 500
    y = RNG.integers(-2 ** 20, 2 ** 20, size=n) / 1024.0
    rf = RNG.normal(size=n).astype(np.float16)
    got = oracle.add_residual(y, rf.view(np.uint16))
    want = [Fraction(float(a)) + Fraction(float(b)) for a, b in zip(y, rf)]
    assert all(Fraction(float(g)) == w for g, w in zip(got, want))
    # a residual of +0 changes nothing
    z = oracle.add_residual(y, np.zeros(n, dtype=np.uint16))
    assert np.array_equal(z, y)


# ----------------------------------------------------------------------------
# load-time repack: the nibble-level transpose of a packed 4-bit matrix
# (forum thread "vLLM on Hygon Z100", section 四: checkpoint INT4 layouts
# transposed and repacked in 8 x 8 nibble blocks)
# ----------------------------------------------------------------------------
def test_transpose_u4_hand_block():
    # A[r][c] = r: every source word of row r is r repeated (r * 0x11111111);
    # every column of A is 0, 1, ..., 7, i.e. the word 0x76543210.  And the
    # other way round for A[r][c] = c.
    rows_const = np.array([r * 0x11111111 for r in range(8)], dtype=np.uint32)
    assert np.array_equal(oracle.transpose_u4(rows_const, 8, 8)[:, 0],
                          np.full(8, 0x76543210, dtype=np.uint32))
    cols_const = np.full(8, 0x76543210, dtype=np.uint32)
    assert np.array_equal(oracle.transpose_u4(cols_const, 8, 8)[:, 0],
                          np.array([c * 0x11111111 for c in range(8)], dtype=np.uint32))


def test_transpose_u4_against_pinned_pack_unpack():
    # A [128, 256] of random nibbles: pack it along its columns (the pinned
    # packer), transpose, unpack along the new rows: A^T exactly
    A = RNG.integers(0, 16, size=(128, 256), dtype=np.uint8)
    zq = np.zeros((128, 2), dtype=np.uint8)
    src, _ = oracle.pack(A, zq)
    dst = oracle.transpose_u4(src, 128, 256)
    assert dst.shape == (256, 16)
    back, _ = oracle.unpack(dst, np.zeros((256, 1), dtype=np.uint32), 128)
    assert np.array_equal(back, A.T)
    # twice is the identity
    assert np.array_equal(oracle.transpose_u4(dst, 256, 128), src)


def test_transpose_u4_ragged_rows_pad_with_zero():
    # rows not a multiple of 8: the result equals that of the matrix padded
    # with zero rows (pad nibbles are 0)
    A = RNG.integers(0, 16, size=(128, 128), dtype=np.uint8)
    A[101:] = 0
    src, _ = oracle.pack(A, np.zeros((128, 1), dtype=np.uint8))
    full = oracle.transpose_u4(src, 128, 128)
    ragged = oracle.transpose_u4(src[:101], 101, 128)
    assert ragged.shape == (128, 13)
    assert np.array_equal(ragged, full[:, :13])


def test_transpose_u4_nibble_order():
    # one source word 0x76543210 holds the value p at position p; with order
    # P (element j at position P[j]) column j of the one-row matrix reads P[j]
    perm = [3, 7, 0, 4, 1, 5, 2, 6]
    order = sum(p << (4 * j) for j, p in enumerate(perm))
    dst = oracle.transpose_u4(np.array([0x76543210], dtype=np.uint32), 1, 8, order)
    assert dst[:, 0].tolist() == perm
    # the sequential order is the identity permutation
    dst = oracle.transpose_u4(np.array([0x76543210], dtype=np.uint32), 1, 8)
    assert dst[:, 0].tolist() == list(range(8))


def test_transpose_u16_is_numpy_transpose():
    a = RNG.integers(0, 1 << 16, size=(37, 130)).astype(np.uint16)
    assert np.array_equal(oracle.transpose_u16(a), a.T)


# ----------------------------------------------------------------------------
# bfloat16 (activations "fp16 or bf16"): conversions and the linear
# ----------------------------------------------------------------------------
def _bf16_value(bits):
    """bfloat16 is the top half of an IEEE binary32: decode with numpy's float32."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def _bf16_bits(a):
    """Inputs only: the top 16 bits of the float32 (any pattern is a valid bf16)."""
    return (np.asarray(a, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def test_bf16_to_double_every_pattern():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = oracle.bf16_to_double(bits)
    with np.errstate(invalid="ignore"):
        ref = _bf16_value(bits)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_double_to_bf16_neighbours_and_ties():
    # a and its successor b (consecutive finite positive patterns): values
    # exactly a and b map to themselves; their midpoint (exact in binary64)
    # to whichever has an even last bit; points just off the midpoint to the
    # nearer one; negative values mirror positive ones
    a = RNG.integers(1, 0x7F7F, size=20000).astype(np.uint16)
    b = (a + 1).astype(np.uint16)
    va, vb = _bf16_value(a), _bf16_value(b)
    mid = (va + vb) / 2
    assert np.array_equal(oracle.double_to_bf16(va), a)
    assert np.array_equal(oracle.double_to_bf16(vb), b)
    even = np.where(a % 2 == 0, a, b)
    assert np.array_equal(oracle.double_to_bf16(mid), even)
    eps = (vb - va) * 2.0 ** -20
    assert np.array_equal(oracle.double_to_bf16(mid - eps), a)
    assert np.array_equal(oracle.double_to_bf16(mid + eps), b)
    assert np.array_equal(oracle.double_to_bf16(-mid), even | 0x8000)


def test_double_to_bf16_closed_form():
    # 1 + 2^-8 ties between 1 and 1 + 2^-7: to even (1.0); 1 + 3 * 2^-8 ties
    # between 1 + 2^-7 (odd) and 1 + 2^-6 (even)
    assert oracle.double_to_bf16([1 + 2 ** -8])[0] == 0x3F80
    assert oracle.double_to_bf16([1 + 3 * 2 ** -8])[0] == 0x3F82
    # largest finite (2 - 2^-7) * 2^127; the midpoint to 2^128 rounds up to inf
    big = (2 - 2 ** -7) * 2.0 ** 127
    assert oracle.double_to_bf16([big])[0] == 0x7F7F
    assert oracle.double_to_bf16([(2 - 2 ** -8) * 2.0 ** 127])[0] == 0x7F80
    # subnormals: quantum 2^-133; half of it ties to zero, 1.5 of it to 2 quanta
    assert oracle.double_to_bf16([2.0 ** -134])[0] == 0x0000
    assert oracle.double_to_bf16([3 * 2.0 ** -134])[0] == 0x0002
    assert oracle.double_to_bf16([-0.0])[0] == 0x8000


def _brute_force_exact_bf16(xb, q, z, sb, group):
    M, K = xb.shape
    N = q.shape[0]
    xf = [[Fraction(float(v)) for v in row] for row in _bf16_value(xb)]
    sf = [[Fraction(float(v)) for v in row] for row in _bf16_value(sb)]
    y = [[Fraction(0)] * N for _ in range(M)]
    mag = [[Fraction(0)] * N for _ in range(M)]
    for m in range(M):
        for n in range(N):
            for k in range(K):
                t = xf[m][k] * (int(q[n, k]) - int(z[n, k // group])) * sf[n][k // group]
                y[m][n] += t
                mag[m][n] += abs(t)
    return y, mag


@pytest.mark.parametrize("M,N,K", [(1, 1, 128), (2, 3, 256)])
def test_linear_bf16_matches_exact_rationals(M, N, K):
    G = K // 128
    q = RNG.integers(0, 16, (N, K)).astype(np.uint8)
    z = RNG.integers(0, 16, (N, G)).astype(np.uint8)
    sb = _bf16_bits(RNG.uniform(0.002, 0.02, (N, G)))
    xb = _bf16_bits(RNG.standard_normal((M, K)))
    qw, zw = oracle.pack(q, z)
    y = oracle.linear(xb, qw, sb, zw, dtype="bf16")
    ye, mag = _brute_force_exact_bf16(xb, q, z, sb, 128)
    for m in range(M):
        for n in range(N):
            err = abs(Fraction(y[m, n]) - ye[m][n])
            assert err <= Fraction(1, 10 ** 12) * (mag[m][n] + Fraction(1, 10 ** 30))
    rows = np.array([N - 1, 0] if N > 1 else [0])
    assert np.array_equal(oracle.linear_rows(xb, qw, sb, zw, rows, dtype="bf16"), y[:, rows])
    # the same bits read as fp16 give a different product: the type is honoured
    assert not np.array_equal(oracle.linear(xb, qw, sb, zw), y)


def test_linear_bf16_integer_case_equals_int64_matmul():
    # x in {-1, 0, 1} (bf16 0xBF80, 0, 0x3F80), s = 2^-4 (bf16 0x3D80)
    M, N, K = 3, 7, 512
    q = RNG.integers(0, 16, (N, K)).astype(np.uint8)
    z = RNG.integers(0, 16, (N, K // 128)).astype(np.uint8)
    X = RNG.integers(-1, 2, (M, K)).astype(np.int64)
    xb = np.where(X == 1, 0x3F80, np.where(X == -1, 0xBF80, 0)).astype(np.uint16)
    sb = np.full((N, K // 128), 0x3D80, dtype=np.uint16)
    qw, zw = oracle.pack(q, z)
    W = q.astype(np.int64) - np.repeat(z.astype(np.int64), 128, axis=1)
    assert np.array_equal(oracle.linear(xb, qw, sb, zw, dtype="bf16"),
                          (X @ W.T).astype(np.float64) / 16)


def test_add_residual_bf16_exact():
    n = 300
    y = RNG.integers(-2 ** 20, 2 ** 20, size=n) / 1024.0
    rb = _bf16_bits(RNG.normal(size=n) * 4)
    got = oracle.add_residual(y, rb, dtype="bf16")
    assert all(Fraction(float(g)) == Fraction(float(a)) + Fraction(float(b))
               for g, a, b in zip(got, y, _bf16_value(rb)))


# ----------------------------------------------------------------------------
# dense 16-bit linear (weights dequantised at load time; Z100 thread, section 六)
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_dense_linear_matches_exact_rationals(dtype):
    M, N, K = 2, 3, 96
    if dtype == "f16":
        xb = _f16_bits(RNG.standard_normal((M, K)))
        wb = _f16_bits(RNG.standard_normal((N, K)) * 0.05)
        dec = lambda b: b.view(np.float16).astype(np.float64)  # noqa: E731
    else:
        xb = _bf16_bits(RNG.standard_normal((M, K)))
        wb = _bf16_bits(RNG.standard_normal((N, K)) * 0.05)
        dec = _bf16_value
    y = oracle.dense_linear(xb, wb, dtype)
    xf, wf = dec(xb), dec(wb)
    for m in range(M):
        for n in range(N):
            exact = sum(Fraction(float(a)) * Fraction(float(b)) for a, b in zip(xf[m], wf[n]))
            mag = sum(abs(Fraction(float(a)) * Fraction(float(b))) for a, b in zip(xf[m], wf[n]))
            assert abs(Fraction(y[m, n]) - exact) <= Fraction(1, 10 ** 12) * (mag + Fraction(1, 10 ** 30))
    rows = np.array([2, 0])
    assert np.array_equal(oracle.dense_linear(xb, wb, dtype, rows=rows), y[:, rows])


def test_dense_linear_equals_the_4bit_linear_on_its_dequantised_weights():
    # s a power of two: every (q - z) * s is exact in fp16, so the dense product
    # over those weights adds the same binary64 terms in the same order as the
    # (pinned) 4-bit oracle: bit-identical
    M, N, K = 3, 5, 512
    q = RNG.integers(0, 16, (N, K)).astype(np.uint8)
    z = RNG.integers(0, 16, (N, K // 128)).astype(np.uint8)
    sb = np.full((N, K // 128), 0x2C00, dtype=np.uint16)  # 1/16
    xb = _f16_bits(RNG.standard_normal((M, K)))
    qw, zw = oracle.pack(q, z)
    w = (q.astype(np.float64) - np.repeat(z, 128, axis=1)) / 16
    assert np.array_equal(oracle.dense_linear(xb, _f16_bits(w)), oracle.linear(xb, qw, sb, zw))


def test_dense_linear_integer_case_equals_int64_matmul():
    M, N, K = 4, 7, 300
    X = RNG.integers(-1, 2, (M, K)).astype(np.int64)
    W = RNG.integers(-50, 51, (N, K)).astype(np.int64)
    y = oracle.dense_linear(_f16_bits(X), _f16_bits(W))
    assert np.array_equal(y, (X @ W.T).astype(np.float64))


# ----------------------------------------------------------------------------
# mixture of experts (Z100 thread, section 七): alignment by expert, the expert
# linears, the weighted sum per token
# ----------------------------------------------------------------------------
def test_moe_align_is_a_stable_sort_by_expert():
    E = 7
    ids = RNG.integers(0, E, size=(9, 4)).astype(np.int32)
    srt, pos, off = oracle.moe_align(ids, E)
    flat = ids.reshape(-1)
    assert np.array_equal(srt, np.argsort(flat, kind="stable"))
    assert np.array_equal(pos[srt], np.arange(flat.size))
    assert np.array_equal(off, np.concatenate([[0], np.cumsum(np.bincount(flat, minlength=E))]))
    # an expert nobody chose has an empty range
    srt1, _, off1 = oracle.moe_align(np.zeros((3, 2), dtype=np.int32), 3)
    assert off1.tolist() == [0, 6, 6, 6] and srt1.tolist() == list(range(6))


def _experts(E, N, K):
    q = RNG.integers(0, 16, (E, N, K)).astype(np.uint8)
    z = RNG.integers(0, 16, (E, N, K // 128)).astype(np.uint8)
    s = _f16_bits(RNG.uniform(0.002, 0.02, (E, N, K // 128)))
    packed = [oracle.pack(q[e], z[e]) for e in range(E)]
    return np.stack([p[0] for p in packed]), s, np.stack([p[1] for p in packed])


def test_moe_linear_is_the_pinned_linear_of_each_slots_expert():
    E, N, K, T, k = 4, 6, 256, 5, 3
    qw, s, zw = _experts(E, N, K)
    ids = RNG.integers(0, E, size=(T, k)).astype(np.int32)
    x = _f16_bits(RNG.standard_normal((T, K)))
    y = oracle.moe_linear(x, qw, s, zw, ids)
    for t in range(T):
        for j in range(k):
            e = ids[t, j]
            assert np.array_equal(y[t * k + j], oracle.linear(x[t:t + 1], qw[e], s[e], zw[e])[0])
    # per-slot inputs: slot s reads row s
    xs = _f16_bits(RNG.standard_normal((T * k, K)))
    ys = oracle.moe_linear(xs, qw, s, zw, ids, per_slot=True)
    for slot in (0, 7, T * k - 1):
        e = ids.reshape(-1)[slot]
        assert np.array_equal(ys[slot], oracle.linear(xs[slot:slot + 1], qw[e], s[e], zw[e])[0])


def test_moe_sum_selects_and_is_exact():
    T, k, N = 3, 4, 5
    y = RNG.integers(-2 ** 10, 2 ** 10, size=(T * k, N)) / 64.0
    onehot = np.zeros((T, k))
    onehot[np.arange(T), [1, 3, 0]] = 1.0
    assert np.array_equal(oracle.moe_sum(y, onehot), y[[1, 7, 8]])
    w = RNG.integers(0, 64, size=(T, k)) / 64.0  # dyadic: the binary64 sum is exact
    out = oracle.moe_sum(y, w)
    for t in range(T):
        for n in range(N):
            exact = sum(Fraction(float(w[t, j])) * Fraction(float(y[t * k + j, n])) for j in range(k))
            assert Fraction(float(out[t, n])) == exact
