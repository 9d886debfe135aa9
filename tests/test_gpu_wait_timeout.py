"""The error path of the bounded waits, exercised without any fault.

Every kernel's waits on its asynchronous copies give up after a time limit,
raise a device flag and let the kernel return (no trap, no hang). The
self-test entry point makes one such wait run out on purpose: one thread waits,
with the kernels' own wait routine, on a barrier that nothing ever completes.
The test checks that the wait lasted its limit, that rmsnorm_device_error
reports the flag and clears it, and that the context is still usable: a
forward and backward right after it give the same bits as before.
"""
from __future__ import annotations

import pytest
import torch

import invariant_rmsnorm_gb300 as rn
from invariant_rmsnorm_gb300 import synth
from tests.gpu_common import DEV, run_bwd, run_fwd

pytestmark = pytest.mark.gpu


def _step():
    x = synth.normal16((300, 4096), 1, DEV)
    g = synth.normal16((300, 4096), 2, DEV)
    w = synth.gamma_f32(4096, 3, DEV)
    fo = run_fwd("plain", x, w, 1e-6, False)
    bo = run_bwd("plain", g, x, w, fo["rstd"], False)
    torch.cuda.synchronize()
    return [t.clone() for t in (fo["y"], fo["rstd"], bo["dx"], bo["dgamma"])]


@pytest.mark.parametrize("limit_ns", [1_000_000, 50_000_000])
def test_wait_runs_out_and_is_reported(limit_ns):
    before = _step()
    assert rn.rmsnorm_device_error(clear=True) == 0
    waited = torch.zeros(1, dtype=torch.int64, device=DEV)
    rn.rmsnorm_selftest_wait_timeout(limit_ns, waited)
    flags = rn.rmsnorm_device_error(clear=True)
    assert flags == rn.DEVICE_ERR_WAIT_TIMEOUT
    w = int(waited.item())
    assert limit_ns <= w < limit_ns + 500_000_000, w   # gave up at its limit, not much later
    assert rn.rmsnorm_device_error(clear=False) == 0   # the flag was cleared
    after = _step()                                    # the context still works, same bits
    for a, b in zip(before, after):
        assert torch.equal(a.view(torch.int16) if a.element_size() == 2 else a.view(torch.int32),
                           b.view(torch.int16) if b.element_size() == 2 else b.view(torch.int32))
    assert rn.rmsnorm_device_error() == 0
