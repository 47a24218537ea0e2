"""The expired-wait report on the GPU: the library's bounded waits (a
completion counter, an mbarrier phase) run on a counter and an mbarrier that
nothing completes; each gives up after its limit and sets its bit in the
device status word.  The context stays usable: a linear launched right after
still matches the oracle.
"""
import time

import pytest
import torch

import synthetic_inputs as si
from helpers import Case, assert_close

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def w4():
    import __graft_entry__
    __graft_entry__.build()
    import weight_only_int4_w4a16_gb300 as w4
    w4.w4a16_init(0, 256 << 20)
    return w4


def test_expired_waits_are_reported_and_the_context_survives(w4):
    assert w4.w4a16_device_status() == 0
    t0 = time.perf_counter()
    w4.w4a16_wait_probe()
    code = w4.w4a16_device_status()  # synchronises, returns and clears the word
    elapsed = time.perf_counter() - t0
    assert code == 4096 | 8192
    assert 0.3 < elapsed < 10.0  # two 200 ms limits, not a hang
    assert w4.w4a16_device_status() == 0  # cleared by the read
    c = Case(si.config_seed(77), 4, 1024, 2048)
    x, qw, s, zw = c.to(DEV)
    y = w4.w4a16_linear(x, qw, s, zw)
    torch.cuda.synchronize()
    assert_close(y, c.reference(), "linear after the probe")
    assert w4.w4a16_device_status() == 0
