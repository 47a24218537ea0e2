"""The allocation-free entry point (w4a16_linear_noalloc) against w4a16_linear.

Collected last.  It must pass alone in a fresh process and after every other
test: the allocation-free calls come first and need no w4a16_init; the
library is initialised only afterwards, for the comparison with
w4a16_linear (unless an earlier test already did).
"""
import pytest
import torch

import synthetic_inputs as si
from helpers import assert_close

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def w4():
    import __graft_entry__
    __graft_entry__.build()
    import weight_only_int4_w4a16_gb300 as w4
    return w4


def _linear_initialised(w4, x, qw, s, zw, y):
    try:
        return w4.w4a16_linear(x, qw, s, zw, y=y)
    except w4.W4A16Error as e:
        if e.status != w4.W4A16_ERR_NOT_INITIALIZED:
            raise
    w4.w4a16_init(0, 256 << 20)
    return w4.w4a16_linear(x, qw, s, zw, y=y)


# split K over the scratch (M=4: seven slices of K=17408), a shape without a
# split, and a ragged one (N not a multiple of 16, K of 4 groups' stages)
@pytest.mark.parametrize("M,N,K", [(4, 5120, 17408), (1, 34816, 5120), (8, 1000, 2560),
                                   (3, 777, 1408)])
def test_noalloc_two_calls_match_linear(w4, M, N, K):
    seed = si.config_seed(70, 0, M)
    qw, s, zw = si.layer(seed, N, K, device=DEV)
    x = si.x(seed, M, K).to(DEV)
    ys = [torch.full((M, N), float("nan"), dtype=torch.float16, device=DEV) for _ in range(2)]
    for y in ys:  # two calls in a row, no host synchronisation between them
        w4.w4a16_linear_noalloc(x, qw, s, zw, y)
    torch.cuda.synchronize()
    ref = torch.full((M, N), float("nan"), dtype=torch.float16, device=DEV)
    _linear_initialised(w4, x, qw, s, zw, ref)
    torch.cuda.synchronize()
    y_ref = ref.double().cpu().numpy()
    for i, y in enumerate(ys):
        assert_close(y, y_ref, f"no-alloc call {i} M={M} N={N} K={K}")
    assert torch.equal(ys[0].view(torch.int16), ys[1].view(torch.int16))


def test_noalloc_rejects_what_the_scratch_cannot_hold(w4):
    # M = 8 at K = 17408 needs at least seven K slices: 7 x 8 x 40960 fp32
    # partial sums are more than the 2 MiB scratch.  Rejected before launch.
    M, N, K = 8, 40960, 17408
    x = torch.zeros((M, K), dtype=torch.float16, device=DEV)
    qw = torch.zeros((N, K // 8), dtype=torch.int32, device=DEV)
    s = torch.zeros((N, K // 128), dtype=torch.float16, device=DEV)
    zw = torch.zeros((N, (K // 128 + 7) // 8), dtype=torch.int32, device=DEV)
    y = torch.full((M, N), float("nan"), dtype=torch.float16, device=DEV)
    with pytest.raises(w4.W4A16Error) as e:
        w4.w4a16_linear_noalloc(x, qw, s, zw, y)
    assert e.value.status == w4.W4A16_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.isnan(y).all()
    # more than 8 tokens is not this entry point's work
    x9 = torch.zeros((9, 1024), dtype=torch.float16, device=DEV)
    qw9 = torch.zeros((64, 128), dtype=torch.int32, device=DEV)
    s9 = torch.zeros((64, 8), dtype=torch.float16, device=DEV)
    zw9 = torch.zeros((64, 1), dtype=torch.int32, device=DEV)
    y9 = torch.empty((9, 64), dtype=torch.float16, device=DEV)
    with pytest.raises(w4.W4A16Error) as e:
        w4.w4a16_linear_noalloc(x9, qw9, s9, zw9, y9)
    assert e.value.status == w4.W4A16_ERR_UNSUPPORTED
