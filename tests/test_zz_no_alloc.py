"""m3_siso_forward_static: the SISO scan entry point for callers that cannot
allocate device memory (a host that owns every allocation, or a loop where a
cudaMalloc would synchronize the device). It must give the results of
m3_siso_forward, which takes a caller-allocated workspace, on consecutive
calls that reuse the library's fixed scratch array.

This file is collected last so that a run stopping at the first failure has
already run every other test."""
import numpy as np
import pytest

import selective_state_space_mamba3_gb300 as m3
from selective_state_space_mamba3_gb300 import inputs as gen

from m3_testutil import SCAN_KEYS, TOL, dev, gpu_scan, check_close

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("mode", [m3.M3_MATH_TF32, m3.M3_MATH_FP32])
def test_static_scratch_entry_matches_workspace_entry(mode):
    import torch
    from selective_state_space_mamba3_gb300 import build
    build.build()
    w = gen.Workload("no-alloc", 2, 200, 4, 2, 64, 128, 16, seed_index=21)
    ins = gen.scan_inputs(w)
    cfg = m3.ssm_config(w.cfg(), mode)
    ref = gpu_scan(w.cfg(), ins, mode)          # m3_siso_forward with a workspace
    d = {k: dev(ins[k]) for k in SCAN_KEYS}
    for call in range(2):
        out = torch.full((2, 200, 4, 64), float("nan"), device="cuda")
        m3.m3_siso_forward_static(cfg, *[d[k] for k in SCAN_KEYS], out)
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        assert np.all(np.isfinite(got))
        check_close(got, ref, TOL[mode], label=f"call {call}")
