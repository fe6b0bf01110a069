"""Failure detection without a GPU fault: a bounded device wait on an mbarrier
that nothing completes gives up after its clock budget, records
M3_ERR_TIMEOUT in the workspace status word, and leaves the context usable
(a scan right after it still matches the oracle)."""
import numpy as np
import pytest

import oracle
import selective_state_space_mamba3_gb300 as m3
from selective_state_space_mamba3_gb300 import inputs as gen

from m3_testutil import TOL, check_close, gpu_scan, oracle_scan

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from selective_state_space_mamba3_gb300 import build
    build.build()
    oracle.build()


def test_bounded_wait_times_out_and_context_survives():
    import torch
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    m3.m3_selftest_wait_timeout(ws, 2_000_000)      # about a millisecond of SM clock
    assert m3.m3_workspace_status(ws) == m3.M3_ERR_TIMEOUT
    torch.cuda.synchronize()
    w = gen.TINY_SISO
    ins = gen.scan_inputs(w)
    for mode in (m3.M3_MATH_FP32, m3.M3_MATH_TF32):
        got = gpu_scan(w.cfg(), ins, mode)
        check_close(got, oracle_scan(w.cfg(), ins), TOL[mode])
