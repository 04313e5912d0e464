"""Failure detection on the GPU without a fault: a kernel's bounded wait runs out (an
mbarrier nobody completes, a flag nobody sets); the host reads SGEMM_ERR_TIMEOUT from the
device error word, and the context stays usable for the next product call."""
from __future__ import annotations

import time

import pytest

from gemm_case import TOL, Case, run

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.mark.parametrize("which", [0, 1], ids=["mbarrier", "flag"])
def test_bounded_wait_reports_timeout_and_context_survives(sgemm_lib, which):
    sg = sgemm_lib
    assert sg.sgemm_device_status() == sg.SGEMM_OK
    t0 = time.perf_counter()
    sg.sgemm_selftest_bounded_wait(which)
    status = sg.sgemm_device_status()
    waited = time.perf_counter() - t0
    assert status == sg.SGEMM_ERR_TIMEOUT, sg.sgemm_last_error()
    assert "bounded wait" in sg.sgemm_last_error()
    assert 1.0 < waited < 30.0
    # the word is cleared by the read, and the context still runs the product path
    assert sg.sgemm_device_status() == sg.SGEMM_OK
    err, _, _ = run(Case(256, 320, 200, 1.0, 0.5, "uniform", seed=9), sg.sgemm, torch)
    assert err <= TOL


def test_selftest_rejects_unknown_mode(sgemm_lib):
    with pytest.raises(sgemm_lib.SgemmError):
        sgemm_lib.sgemm_selftest_bounded_wait(7)
