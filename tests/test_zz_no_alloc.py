"""The allocation-free entry point (w4a16_linear_noalloc).

This entry point is for callers that cannot allocate device memory: a process
whose caching allocator has reserved the whole device, or a serving loop that
must not call cudaMalloc (it synchronises the device).  Its split-K scratch is
a static device array of the library, so it needs no w4a16_init.

Its outputs are checked against the oracle and against w4a16_linear, on two
calls in a row.  The file is collected last.  It must pass alone in a fresh
process and after every other test.  The first calls need no w4a16_init; the
library is initialised only afterwards, for the comparison with w4a16_linear
(unless an earlier test already did it).
"""
import numpy as np
import pytest
import torch

import oracle
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


def _ensure_init(w4):
    if w4.w4a16_device_sm_count() == 0:
        w4.w4a16_init(0, 256 << 20)


def _oracle(x, qw, s, zw):
    return oracle.linear(si.as_u16(x), si.as_u32(qw), si.as_u16(s), si.as_u32(zw))


# split K over the scratch (M=4: four slices of K=17408), a shape without a
# split, the gate+up shape at M=8 (two slices: the largest scratch any decode
# linear of this size class needs), and ragged ones (N not a multiple of 16,
# K a few groups)
@pytest.mark.parametrize("M,N,K", [(4, 5120, 17408), (1, 34816, 5120), (8, 34816, 5120),
                                   (8, 1000, 2560), (3, 777, 1408)])
def test_noalloc_two_calls_match_oracle_and_linear(w4, M, N, K):
    seed = si.config_seed(70, 0, M)
    qw, s, zw = si.layer(seed, N, K, device=DEV)
    x = si.x(seed, M, K).to(DEV)
    ys = [torch.full((M, N), float("nan"), dtype=torch.float16, device=DEV) for _ in range(2)]
    for y in ys:  # two calls in a row, no host synchronisation between them
        w4.w4a16_linear_noalloc(x, qw, s, zw, y)
    torch.cuda.synchronize()
    assert w4.w4a16_device_status() == 0  # readable without w4a16_init
    ref = _oracle(x, qw, s, zw)
    for i, y in enumerate(ys):
        assert_close(y, ref, f"no-alloc call {i} M={M} N={N} K={K}")
    assert torch.equal(ys[0].view(torch.int16), ys[1].view(torch.int16))
    # the same result as the entry point that uses the w4a16_init workspace
    _ensure_init(w4)
    y_lin = w4.w4a16_linear(x, qw, s, zw)
    torch.cuda.synchronize()
    assert_close(ys[0], y_lin.double().cpu().numpy(), f"no-alloc vs w4a16_linear M={M}")


def test_noalloc_counts_its_launches(w4):
    M, N, K = 4, 5120, 17408  # a split-K shape
    qw, s, zw = si.layer(si.config_seed(71), N, K, device=DEV)
    x = si.x(si.config_seed(71), M, K).to(DEV)
    y = torch.empty((M, N), dtype=torch.float16, device=DEV)
    w4.w4a16_probe_reset()
    w4.w4a16_linear_noalloc(x, qw, s, zw, y)
    torch.cuda.synchronize()
    counts = w4.w4a16_probe_counts()
    assert sum(counts) == 1 and counts[w4.RUNG_MMA_SPLITK] == 1
    assert w4.w4a16_kernel_launches() == 1


def test_noalloc_rejects_what_the_scratch_cannot_hold(w4):
    # M = 8 at K = 17408 needs at least seven K slices: 7 x 8 x 40960 fp32
    # partial sums are more than the 4 MiB scratch.  Rejected before launch.
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


def test_noalloc_expired_wait_reported_and_counters_reset(w4):
    # The wait probe runs the library's bounded waits on objects that nothing
    # completes (no fault, no hang) and, for the no-alloc scratch, leaves its
    # first block counter as a split-K launch cut short would leave it.  The
    # status read must report both expiries and clear that counter: later
    # split-K calls (block 0 included) must still match the oracle, with
    # inputs that differ from call to call so stale partial sums would show.
    _ensure_init(w4)
    M, N, K = 4, 5120, 17408
    qw, s, zw = si.layer(si.config_seed(72), N, K, device=DEV)
    y = torch.empty((M, N), dtype=torch.float16, device=DEV)
    w4.w4a16_linear_noalloc(si.x(si.config_seed(72, 1), M, K).to(DEV), qw, s, zw, y)
    torch.cuda.synchronize()
    assert w4.w4a16_device_status() == 0
    w4.w4a16_wait_probe()
    assert w4.w4a16_device_status() == 4096 | 8192
    assert w4.w4a16_device_status() == 0  # cleared by the read
    for i in range(3):
        x = si.x(si.config_seed(72, 2 + i), M, K).to(DEV)
        y = torch.full((M, N), float("nan"), dtype=torch.float16, device=DEV)
        w4.w4a16_linear_noalloc(x, qw, s, zw, y)
        torch.cuda.synchronize()
        assert_close(y, _oracle(x, qw, s, zw), f"no-alloc call {i} after the probe")
    assert w4.w4a16_device_status() == 0
    assert np.isfinite(y.float().cpu().numpy()).all()
