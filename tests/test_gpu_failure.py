"""Failure detection without a GPU fault: a bounded device-side wait that
runs out is reported to the host, and the context stays usable."""
import math

import pytest
import torch

from state_summary_scan_gb300 import _capi as C

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    C.load()


def test_wait_timeout_is_reported_and_context_survives():
    scratch = torch.zeros(4, dtype=torch.int32, device="cuda")
    C.rm_cp_device_status(scratch, clear=True)          # start from a clear flag
    C.rm_cp_selftest_wait_timeout(2000)                 # a barrier nothing completes, 2 ms bound
    assert C.rm_cp_device_status(scratch, clear=True) == 7   # RM_ERR_TIMEOUT
    assert C.rm_cp_device_status(scratch, clear=True) == 0   # cleared
    # the context is still usable: a tensor-core problem runs and stays clean
    from tests_helpers import small_tc_run
    small_tc_run()
    assert C.rm_cp_device_status(scratch, clear=True) == 0


def test_normal_runs_never_time_out():
    scratch = torch.zeros(4, dtype=torch.int32, device="cuda")
    C.rm_cp_device_status(scratch, clear=True)
    from tests_helpers import small_tc_run
    for _ in range(3):
        small_tc_run()
    assert C.rm_cp_device_status(scratch, clear=True) == 0
