"""Failure reporting of the bounded device waits, exercised without a fault.

Every pipeline wait in the kernels gives up after a limit of device time,
records a role/kernel code in the per-device error word and lets its kernel
return instead of hanging the GPU.  t3_selftest_wait_timeout runs that same
wait loop in one CTA on a barrier that nothing completes, with a limit of a
few milliseconds: the wait must run out, the error must reach the host as
T3_ETIMEOUT with the self-test's code, the word must be cleared by reading
it, and the device must stay usable (a product right after is bit-exact).
"""
import numpy as np
import pytest

import oracle
import t3_synth
import ternary_weight_int8_t3_gb300 as t3

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

SELFTEST_CODE = (10 << 8) | 2   # kernel 10 (the wait self-test), role 2 (a waiting converter)


def test_bounded_wait_gives_up_and_reports_timeout():
    assert torch.cuda.is_available()
    rc, _ = t3.t3_last_device_error()          # start from a clear word
    assert rc == t3.T3_OK
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    t3.t3_selftest_wait_timeout(5_000_000)      # 5 ms
    e1.record()
    rc, detail = t3.t3_last_device_error()
    assert rc == t3.T3_ETIMEOUT, t3.status_string(rc)
    assert detail == SELFTEST_CODE, hex(detail)
    ms = e0.elapsed_time(e1)
    assert 4.5 <= ms < 500.0, f"the wait gave up after {ms:.2f} ms"
    rc, detail = t3.t3_last_device_error()      # reading cleared it
    assert (rc, detail) == (t3.T3_OK, 0)


def test_device_usable_after_a_timeout():
    t3.t3_selftest_wait_timeout(2_000_000)
    rc, detail = t3.t3_last_device_error()
    assert (rc, detail) == (t3.T3_ETIMEOUT, SELFTEST_CODE)
    g = t3_synth.rng(5)
    for (M, N, K) in [(300, 272, 96), (8, 512, 1024)]:
        A = t3_synth.int8_uniform(g, (M, K))
        wp = oracle.pack(t3_synth.ternary(g, (K, N)))
        C = t3.t3_gemm_fwd(torch.from_numpy(A).cuda(), torch.from_numpy(wp).cuda(), K=K)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(C.cpu().numpy(), oracle.fwd(A, wp))
    assert t3.t3_last_device_error() == (t3.T3_OK, 0)


def test_two_timeouts_one_read():
    """Two timeouts before a read: the word holds the code once and one read
    reports and clears it."""
    t3.t3_selftest_wait_timeout(1_000_000)
    t3.t3_selftest_wait_timeout(1_000_000)
    assert t3.t3_last_device_error() == (t3.T3_ETIMEOUT, SELFTEST_CODE)
    assert t3.t3_last_device_error() == (t3.T3_OK, 0)
