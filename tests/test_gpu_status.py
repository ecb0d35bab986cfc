"""The device error word and the bounded-wait path, exercised without any
fault: a kernel waits on a barrier that nothing completes and must give up
after its budget with DPRED_E_TIMEOUT, leaving the context usable."""
import pytest
import torch

import zero_collectives_gb300 as zc

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    assert zc.device_status(clear=True) in (0, -6)
    assert zc.device_status() == 0
    zc.selftest_wait_timeout(2_000_000)   # about 1 ms of SM clocks
    torch.cuda.synchronize()
    assert zc.device_status() == -6
    assert zc.device_status(clear=True) == -6
    assert zc.device_status() == 0
    x = torch.ones(1024, device="cuda")
    assert float(x.sum().item()) == 1024.0   # the context still works


def test_selftest_rejects_bad_budget():
    with pytest.raises(zc.DpredError):
        zc.selftest_wait_timeout(-1)


def test_bounds_selftest_matches_the_build():
    """The access test on an out-of-range index records DPRED_E_BOUNDS in the
    checked build and nothing in the default build; nothing is accessed."""
    zc.device_status(clear=True)
    zc.selftest_bounds()
    torch.cuda.synchronize()
    want = -7 if zc.checked_build() else 0
    assert zc.device_status(clear=True) == want
    assert zc.device_status() == 0


def test_prediv_matches_ieee_division_on_every_fp32_input():
    """The flush pre-divides every term by the rank count.  For counts that
    are not powers of two it uses a division-free quotient (Markstein's
    correction step); for powers of two a multiply by the exact reciprocal.
    Both must equal IEEE division rounded to nearest even -- what the oracle
    computes -- on all 2^32 fp32 inputs (which include every bf16 value),
    for every rank count the library accepts."""
    for world in range(1, zc.MAX_WORLD + 1):
        n, first = zc.selftest_prediv(world)
        assert n == 0, f"world {world}: {n} inputs differ, first bit pattern {first:#010x}"
