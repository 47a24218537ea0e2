"""GPU parity of the load-time repack (w4a16_repack_transpose,
w4a16_transpose_f16) against the oracle: bit-exact, for sequential and
permuted source nibble orders, ragged shapes and a full-size layer, and a
checkpoint stored transposed ([K, N/8] weights, [G, N/8] zeros, [G, N] scales)
that, once repacked, gives the oracle's linear.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic_inputs as si
from helpers import assert_close

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
SEQ = 0x76543210
# element j of a word at position P[j]: an interleave of even then odd elements
INTERLEAVED = sum(p << (4 * j) for j, p in enumerate([0, 2, 4, 6, 1, 3, 5, 7]))
REVERSED = sum(p << (4 * j) for j, p in enumerate([7, 6, 5, 4, 3, 2, 1, 0]))


@pytest.fixture(scope="module")
def w4():
    import __graft_entry__
    __graft_entry__.build()
    import weight_only_int4_w4a16_gb300 as w4
    w4.w4a16_init(0, 256 << 20)
    return w4


def _words(seed, rows, cols):
    return si.qweight(seed, rows, cols)  # [rows, cols/8] random words


# tile edges: one block, one tile, several tiles with ragged rows (not a
# multiple of 8) and ragged column words (not a multiple of 32)
@pytest.mark.parametrize("order", [SEQ, INTERLEAVED, REVERSED])
@pytest.mark.parametrize("rows,cols", [(8, 8), (1, 8), (256, 256), (101, 72), (1000, 264),
                                       (5120, 8192), (40, 34816)])
def test_repack_bit_exact(w4, rows, cols, order):
    src = _words(rows * 7 + cols, rows, cols)
    dst = torch.full((cols, (rows + 7) // 8), -1, dtype=torch.int32, device=DEV)
    w4.w4a16_repack_transpose(src.to(DEV), rows, cols, order, dst=dst)
    torch.cuda.synchronize()
    ref = oracle.transpose_u4(si.as_u32(src), rows, cols, order)
    assert np.array_equal(si.as_u32(dst), ref)


@pytest.mark.parametrize("rows,cols", [(1, 1), (37, 130), (40, 34816), (136, 5120)])
def test_transpose_f16_bit_exact(w4, rows, cols):
    src = si.scales(rows + cols, rows, 128 * cols)  # [rows, cols] fp16
    dst = w4.w4a16_transpose_f16(src.to(DEV))
    torch.cuda.synchronize()
    assert np.array_equal(si.as_u16(dst), oracle.transpose_u16(si.as_u16(src)))


@pytest.mark.parametrize("M,N,K", [(4, 1024, 2048), (1, 5120, 17408), (8, 264, 1408)])
def test_transposed_checkpoint_gives_the_linear(w4, M, N, K):
    # a checkpoint stored transposed: qweight [K, N/8] and zeros [G, N/8]
    # packed along N, scales [G, N]
    G = K // 128
    seed = si.config_seed(90, 0, M)
    q_ck = si.qweight(seed, K, N)
    z_ck = si.qweight(seed + 1, G, N)
    s_ck = si.scales(seed, G, 128 * N)
    qw = w4.w4a16_repack_transpose(q_ck.to(DEV), K, N)
    zw = w4.w4a16_repack_transpose(z_ck.to(DEV), G, N)
    s = w4.w4a16_transpose_f16(s_ck.to(DEV))
    x = si.x(seed, M, K)
    y = w4.w4a16_linear(x.to(DEV), qw, s, zw)
    torch.cuda.synchronize()
    q_ref = oracle.transpose_u4(si.as_u32(q_ck), K, N)
    z_ref = oracle.transpose_u4(si.as_u32(z_ck), G, N)
    s_ref = oracle.transpose_u16(si.as_u16(s_ck))
    assert np.array_equal(si.as_u32(qw), q_ref) and np.array_equal(si.as_u32(zw), z_ref)
    ref = oracle.linear(si.as_u16(x), q_ref, s_ref, z_ref)
    assert_close(y, ref, f"repacked checkpoint M={M} N={N} K={K}")
