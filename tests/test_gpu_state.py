"""GPU parity of the recurrent-state paths: m3_siso_prefill / m3_mimo_prefill
(the forward scans continued from, and handing over, the step state of
`mamba3_siso_step` / `mamba3_mimo_step`), the prefill -> step hand-off, and
the split of long sequences into segments inside the chunked tensor-core scan
(summary pass, prefix over segments, main pass), all against the CPU oracle."""
import numpy as np
import pytest

import oracle
import selective_state_space_mamba3_gb300 as m3
from selective_state_space_mamba3_gb300 import inputs as gen

from m3_testutil import SCAN_KEYS, MIMO_KEYS, TOL, dev, check_close, gpu_scan, oracle_scan

pytestmark = pytest.mark.gpu
FP32, TF32 = m3.M3_MATH_FP32, m3.M3_MATH_TF32


@pytest.fixture(scope="module", autouse=True)
def _built():
    from selective_state_space_mamba3_gb300 import build
    build.build()
    oracle.build()


def random_state(w, seed, scale=0.3):
    rng = np.random.default_rng(seed)
    B, H, P, N, A, R = w.batch_size, w.num_heads, w.head_dim, w.state_size, w.num_rope_angles, w.mimo_rank
    return dict(ssm=rng.normal(0, scale, (B, H, P, N)), angle=rng.normal(0, 2.0, (B, H, A)),
                k=rng.normal(0, 1.0, (B, H, R, N)), v=rng.normal(0, 1.0, (B, H, R, P)))


def gpu_prefill(w, ins, mode, state, mimo=False, length=None):
    """Runs the prefill entry point on tokens [0, length) from `state`
    (float64 numpy, rounded to float32); returns out and the final state."""
    import torch
    L = length or w.sequence_length
    cfg = m3.ssm_config(w.cfg(sequence_length=L), mode)
    d = {k: dev(np.ascontiguousarray(ins[k][:, :L])) for k in SCAN_KEYS[:8]}
    d.update({k: dev(ins[k]) for k in SCAN_KEYS[8:]})
    if w.num_rope_angles == 0:
        d["angle"] = None
    st = {k: dev(v.astype(np.float32)) for k, v in state.items()}
    if w.num_rope_angles == 0:
        st["angle"] = None
    B, H, P = w.batch_size, w.num_heads, w.head_dim
    out = torch.full((B, L, H, P), float("nan"), device="cuda")
    if mimo:
        for k in MIMO_KEYS:
            d[k] = dev(ins[k])
        nbytes = m3.m3_mimo_prefill_workspace(cfg)
        ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda")
        m3.m3_mimo_prefill(cfg, *[d[k] for k in SCAN_KEYS], *[d[k] for k in MIMO_KEYS],
                           st["ssm"], st["angle"], st["k"], st["v"], out, ws)
    else:
        nbytes = m3.m3_siso_prefill_workspace(cfg)
        ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda")
        m3.m3_siso_prefill(cfg, *[d[k] for k in SCAN_KEYS], st["ssm"], st["angle"], st["k"],
                           st["v"], out, ws)
    torch.cuda.synchronize()
    assert m3.m3_workspace_status(ws) == m3.M3_OK
    fin = {k: (None if v is None else v.cpu().numpy()) for k, v in st.items()}
    return out.cpu().numpy(), fin


def oracle_from_state(w, ins, state, mimo=False, length=None):
    L = length or w.sequence_length
    cfg = w.cfg(sequence_length=L)
    st = {k: np.ascontiguousarray(v.astype(np.float32).astype(np.float64)) for k, v in state.items()}
    sub = {k: (np.ascontiguousarray(v[:, :L]) if k in SCAN_KEYS[:8] else v) for k, v in ins.items()}
    extra = {k: sub[k] for k in MIMO_KEYS} if mimo else {}
    out = oracle.scan(cfg, *[sub[k] for k in SCAN_KEYS], state=st, **extra)
    return out, st


def compare_states(fin, ref, tol):
    check_close(fin["ssm"], ref["ssm"], tol, "ssm")
    check_close(fin["k"], ref["k"], 1e-5, "k")
    check_close(fin["v"], ref["v"], 1e-6, "v")
    if fin["angle"] is not None:
        check_close(fin["angle"], ref["angle"], 1e-5, "angle")


@pytest.mark.parametrize("mode", [FP32, TF32])
@pytest.mark.parametrize("mimo", [False, True], ids=["siso", "mimo"])
def test_prefill_from_state(mode, mimo):
    if mimo:
        w = gen.Workload("prefill-mimo", 2, 90, 2, 1, 32, 64, 16, mimo_rank=4, has_output_norm=1,
                         seed_index=31)
    else:
        w = gen.Workload("prefill", 2, 150, 4, 2, 32, 64, 16, seed_index=32)
    ins = gen.scan_inputs(w)
    state = random_state(w, 5)
    got, fin = gpu_prefill(w, ins, mode, state, mimo=mimo)
    ref, rst = oracle_from_state(w, ins, state, mimo=mimo)
    check_close(got, ref, TOL[mode], "out")
    compare_states(fin, rst, TOL[mode])


@pytest.mark.parametrize("mode", [FP32, TF32])
def test_prefill_then_step_equals_longer_scan(mode):
    """Prefill of 100 tokens from a zero state, then 50 single-token steps,
    against the oracle's scan of all 150 tokens."""
    import torch
    w = gen.Workload("handoff", 2, 150, 4, 2, 32, 64, 16, seed_index=33)
    ins = gen.scan_inputs(w)
    zero = oracle.zero_state(w.cfg(sequence_length=1))
    got1, fin = gpu_prefill(w, ins, mode, zero, length=100)
    st = {k: dev(v) for k, v in fin.items()}
    c1 = m3.ssm_config(w.cfg(sequence_length=1))
    par = [dev(ins[k]) for k in SCAN_KEYS[8:]]
    seq = {k: dev(ins[k]) for k in SCAN_KEYS[:8]}
    outs = []
    for t in range(100, 150):
        tok = [seq[k][:, t:t + 1].clone() for k in SCAN_KEYS[:8]]
        o = torch.empty(2, 1, 4, 32, device="cuda")
        m3.m3_siso_step(c1, *tok, *par, st["ssm"], st["angle"], st["k"], st["v"], o)
        outs.append(o)
    torch.cuda.synchronize()
    got2 = torch.cat(outs, dim=1).cpu().numpy()
    ref = oracle_scan(w.cfg(), ins)
    check_close(got1, ref[:, :100], TOL[mode], "prefill")
    check_close(got2, ref[:, 100:], TOL[mode], "steps")


@pytest.mark.parametrize("mimo", [False, True], ids=["siso", "mimo"])
def test_split_sequence_tf32(mimo):
    """Few (b, h) pairs and a long sequence: the chunked scan splits every
    sequence into segments (summary, prefix, main pass)."""
    if mimo:
        w = gen.Workload("split-mimo", 1, 600, 2, 1, 64, 64, 32, mimo_rank=4, has_output_norm=0,
                         seed_index=34)
    else:
        w = gen.Workload("split", 1, 1500, 2, 1, 64, 128, 32, seed_index=35)
    ins = gen.scan_inputs(w)
    got = gpu_scan(w.cfg(), ins, TF32, mimo=mimo)
    ref = oracle_scan(w.cfg(), ins, mimo=mimo)
    check_close(got, ref, TOL[TF32])


def test_split_prefill_from_state_tf32():
    w = gen.Workload("split-state", 1, 1200, 2, 1, 64, 128, 32, seed_index=36)
    ins = gen.scan_inputs(w)
    state = random_state(w, 9)
    got, fin = gpu_prefill(w, ins, TF32, state)
    ref, rst = oracle_from_state(w, ins, state)
    check_close(got, ref, TOL[TF32], "out")
    compare_states(fin, rst, TOL[TF32])
