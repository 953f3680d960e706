"""Failure detection on the GPU without a fault.

Every wait in the layer's kernels is bounded: when it runs out, the kernel
records a timeout in the device error word and returns, and the host reads
TERN_ETIMEOUT from tern_device_status.  Here a diagnostic kernel runs the same
wait code on a condition nothing ever meets (an mbarrier phase nobody
completes, a device counter nobody raises).  The status must come back, be
cleared by the read, and the context must still run the layer correctly.
The file runs after the parity tests (its name sorts last).
"""
import time

import pytest

import oracle
import synth
from helpers import assert_bf16_parity, to_device

pytestmark = pytest.mark.gpu

TERN_ETIMEOUT = -6
WAIT_LIMIT_S = 2.0


@pytest.fixture(scope="module")
def tl():
    import torch
    import ternary_weight_linear_gb300 as tl
    tl.build()
    tl.load()
    torch.cuda.init()
    return tl


@pytest.mark.parametrize("which", [0, 1], ids=["mbarrier", "counter"])
def test_bounded_wait_reports_timeout_and_the_context_survives(tl, which):
    import torch
    assert tl.tern_device_status() == 0
    t0 = time.monotonic()
    tl.tern_selftest_wait_timeout(which)
    status = tl.tern_device_status()
    elapsed = time.monotonic() - t0
    assert status == TERN_ETIMEOUT
    assert WAIT_LIMIT_S * 0.95 <= elapsed < 60.0
    assert tl.tern_device_status() == 0  # the read cleared the word

    c = synth.case("after_timeout", 1, K=1024, N=256, seed=which)
    W, s, x = to_device(c)
    y = tl.tern_linear(tl.tern_pack(W), s, x)
    torch.cuda.synchronize()
    assert tl.tern_device_status() == 0
    wp, _ = oracle.pack(c.W)
    y_ref, m = oracle.linear_f64(wp, c.scales, c.x, c.T, c.K, c.N)
    assert_bf16_parity(y.cpu().numpy(), y_ref, m, "a T=1 call after a timeout")
