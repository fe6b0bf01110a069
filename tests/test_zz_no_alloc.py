"""m3_siso_forward_static: the SISO scan entry point for callers that cannot
allocate device memory (a host that owns every allocation, or a loop where a
cudaMalloc would synchronize the device). It must give the results of
m3_siso_forward, which takes a caller-allocated workspace, on consecutive
calls that reuse the library's fixed scratch array - including a geometry
whose long sequences are split into segments, so that the summary and entry
states of the split live in that shared array - and report the status word
its bounded waits write there.

This file is collected last so that a run stopping at the first failure has
already run every other test."""
import numpy as np
import pytest

import oracle
import selective_state_space_mamba3_gb300 as m3
from selective_state_space_mamba3_gb300 import inputs as gen

from m3_testutil import SCAN_KEYS, TOL, dev, gpu_scan, check_close, oracle_scan

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from selective_state_space_mamba3_gb300 import build
    build.build()
    oracle.build()


def static_call(w, ins, mode):
    import torch
    cfg = m3.ssm_config(w.cfg(), mode)
    d = {k: dev(ins[k]) for k in SCAN_KEYS}
    out = torch.full((w.batch_size, w.sequence_length, w.num_heads, w.head_dim), float("nan"),
                     device="cuda")
    m3.m3_siso_forward_static(cfg, *[d[k] for k in SCAN_KEYS], out)
    assert m3.m3_siso_forward_static_status() == m3.M3_OK
    got = out.cpu().numpy()
    assert np.all(np.isfinite(got))
    return got


@pytest.mark.parametrize("mode", [m3.M3_MATH_TF32, m3.M3_MATH_FP32])
def test_static_scratch_entry_matches_workspace_entry(mode):
    w = gen.Workload("no-alloc", 2, 200, 4, 2, 64, 128, 16, seed_index=21)
    ins = gen.scan_inputs(w)
    ref = gpu_scan(w.cfg(), ins, mode)          # m3_siso_forward with a workspace
    for call in range(2):
        check_close(static_call(w, ins, mode), ref, TOL[mode], label=f"call {call}")


def test_static_scratch_segmented_sequences():
    """B1 H2 L1000: two sequences cannot fill the GPU, so the TF32 path splits
    each into three segments of two-chunk summary pieces; their summary states,
    angles and decays and the entry states derived from them (about 0.59 MB)
    all live in the shared array. A
    call at another geometry runs first, then two calls in a row; each is held
    to the oracle and to m3_siso_forward."""
    w = gen.Workload("no-alloc segmented", 1, 1000, 2, 1, 64, 128, 32, seed_index=22)
    mode = m3.M3_MATH_TF32
    need = m3.m3_siso_forward_workspace(m3.ssm_config(w.cfg(), mode))
    assert 256 < need <= (1 << 20), need     # segmented, and within the array
    other = gen.Workload("no-alloc other", 2, 200, 4, 2, 64, 128, 16, seed_index=21)
    static_call(other, gen.scan_inputs(other), mode)
    ins = gen.scan_inputs(w)
    ref_oracle = oracle_scan(w.cfg(), ins)
    ref_ws = gpu_scan(w.cfg(), ins, mode)
    for call in range(2):
        got = static_call(w, ins, mode)
        check_close(got, ref_oracle, TOL[mode], label=f"oracle, call {call}")
        check_close(got, ref_ws, TOL[mode], label=f"workspace entry, call {call}")
