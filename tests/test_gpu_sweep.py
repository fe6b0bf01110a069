"""GPU parity over a seeded sweep of geometries (oarust mamba3.rs:
`mamba3_siso`, `mamba3_mimo`, the step-state layouts of `mamba3_siso_step` /
`mamba3_mimo_step`, and `mamba3_preprocess` feeding the scans).

The fixed cases of the other files cover the workloads' own shapes; this sweep
draws odd ones within the operations' limits (P, N <= 128, A <= N / 2 and
<= 64, H % G == 0, MIMO R in {1, 2, 4, 8} with P N <= 4096): state sizes that
are not multiples of 4 or 16, heads sharing groups, sequences of one token,
ragged last chunks, and sequences long enough for few (batch, head) pairs to
be split into segments. Each case runs through the C ABI and is compared with
the oracle on the same inputs at the mode's bar (FP32-exact 1e-5, TF32 2e-3).
"""
import numpy as np
import pytest

import oracle
import selective_state_space_mamba3_gb300 as m3
from selective_state_space_mamba3_gb300 import inputs as gen

from m3_testutil import TOL, check_close, gpu_scan, oracle_scan

pytestmark = pytest.mark.gpu
FP32, TF32 = m3.M3_MATH_FP32, m3.M3_MATH_TF32
MODES = [FP32, TF32]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from selective_state_space_mamba3_gb300 import build
    build.build()
    oracle.build()


def _geometries(n, seed, mimo, max_work=1.5e8):
    """n workloads drawn by a fixed generator; the oracle's work B L H P N R is
    kept below max_work by shortening L."""
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        H = int(rng.choice([1, 2, 3, 4, 6]))
        G = int(rng.choice([g for g in (1, 2, 3, 6) if H % g == 0]))
        P = int(rng.choice([8, 16, 24, 32, 40, 64, 96, 128]))
        N = int(rng.choice([8, 12, 16, 20, 32, 48, 64, 100, 128]))
        A = int(rng.integers(0, min(64, N // 2) + 1))
        R = int(rng.choice([1, 2, 4, 8])) if mimo else 1
        if mimo and P * N > 4096:
            continue
        B = int(rng.integers(1, 3))
        L = int(rng.choice([1, 7, 64, 65, 130, 300, 700]))
        while L > 1 and B * L * H * P * N * R > max_work:
            L //= 2
        # (a MIMO draw of rank 1 always takes the output norm, so that it is
        # not the SISO operation)
        norm = int(mimo and (R == 1 or rng.random() < 0.6))
        name = f"{'mimo' if mimo else 'siso'} sweep {len(out)}"
        out.append(gen.Workload(name, B, L, H, G, P, N, A, mimo_rank=R,
                                has_z=int(rng.random() < 0.85),
                                has_d=int(rng.random() < 0.85), has_output_norm=norm,
                                seed_index=100 + len(out)))
    return out


SISO = _geometries(40, 1234, mimo=False)
MIMO = _geometries(24, 5678, mimo=True)


def _id(w):
    return (f"B{w.batch_size}L{w.sequence_length}H{w.num_heads}G{w.num_groups}"
            f"P{w.head_dim}N{w.state_size}A{w.num_rope_angles}R{w.mimo_rank}"
            f"{'n' if w.has_output_norm else ''}")


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("w", SISO, ids=_id)
def test_siso_sweep(w, mode):
    ins = gen.scan_inputs(w)
    got = gpu_scan(w.cfg(), ins, mode, mimo=False)
    ref = oracle_scan(w.cfg(), ins, mimo=False)
    check_close(got, ref, TOL[mode], _id(w))


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("w", MIMO, ids=_id)
def test_mimo_sweep(w, mode):
    ins = gen.scan_inputs(w)
    got = gpu_scan(w.cfg(), ins, mode, mimo=True)
    ref = oracle_scan(w.cfg(), ins, mimo=True)
    check_close(got, ref, TOL[mode], _id(w))


PREFILL = ([w for w in SISO if w.sequence_length > 1][:10] +
           [w for w in MIMO if w.sequence_length > 1][:6])


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("w", PREFILL, ids=_id)
def test_prefill_sweep(w, mode):
    """The scan from a random step state, and the final state it hands on."""
    from test_gpu_state import compare_states, gpu_prefill, oracle_from_state, random_state
    mimo = w in MIMO
    ins = gen.scan_inputs(w)
    state = random_state(w, 7)
    got, fin = gpu_prefill(w, ins, mode, state, mimo=mimo)
    ref, rst = oracle_from_state(w, ins, state, mimo=mimo)
    check_close(got, ref, TOL[mode], "out " + _id(w))
    compare_states(fin, rst, TOL[mode])


PACKED = SISO[:10] + MIMO[:4]


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("w", PACKED, ids=_id)
def test_packed_sweep(w, mode):
    """The packed-projection entry: the bits of preprocess + scan, and the
    oracle's preprocess -> scan chain."""
    from test_gpu_packed import oracle_chain, run_both
    p = gen.layer_projection(w)
    par = gen.scan_params(w)
    got, two_step = run_both(w, p["projected"], p["dt_bias"], par, mode, gen.PRE_DEFAULT)
    assert np.array_equal(got, two_step), np.max(np.abs(got - two_step))
    ref = oracle_chain(w, p["projected"], p["dt_bias"], par, gen.PRE_DEFAULT, slice(0, 1))
    check_close(got[0:1], ref, TOL[mode], "packed " + _id(w))


STEPS = [w.with_(sequence_length=min(w.sequence_length, 24)) for w in SISO[:12]] + \
        [w.with_(sequence_length=min(w.sequence_length, 24)) for w in MIMO[:8]]


@pytest.mark.parametrize("w", STEPS, ids=_id)
def test_step_sweep(w):
    """Single-token steps from zero states over up to 24 tokens against the
    oracle's scan of the same tokens (FP32-exact bar)."""
    from test_gpu_parity import run_gpu_steps
    mimo = w.name.startswith("mimo")
    ins = gen.scan_inputs(w)
    got, _ = run_gpu_steps(w, ins, w.sequence_length, mimo=mimo)
    ref = oracle_scan(w.cfg(), ins, mimo=mimo)
    check_close(got, ref, TOL[FP32], "step " + _id(w))


BWD_SISO = [w.with_(sequence_length=min(w.sequence_length, 300)) for w in SISO[:16]]
BWD_MIMO = [w.with_(sequence_length=min(w.sequence_length, 130)) for w in MIMO[:10]]


@pytest.mark.parametrize("w", BWD_SISO, ids=_id)
def test_siso_backward_sweep(w):
    """m3_siso_backward on the drawn SISO geometries (up to 300 tokens) against
    the oracle's adjoints (FP32 bar, per-token floor for vanishing gradients)."""
    from test_gpu_backward import compare, gpu_backward
    ins = gen.scan_inputs(w)
    dout = gen.output_gradient(w)
    got = gpu_backward(w.cfg(), ins, dout)
    ref = oracle.siso_backward(w.cfg(), dout, *[ins[k] for k in oracle.GRAD_NAMES])
    compare(got, ref, "backward " + _id(w))


@pytest.mark.parametrize("w", BWD_MIMO, ids=_id)
def test_mimo_backward_sweep(w):
    """m3_mimo_backward on the drawn MIMO geometries (up to 130 tokens)."""
    from test_gpu_backward import gpu_mimo_backward, mimo_compare
    ins = gen.scan_inputs(w)
    dout = gen.output_gradient(w)
    got = gpu_mimo_backward(w.cfg(), ins, dout)
    ref = oracle.mimo_backward(w.cfg(), dout, *[ins[k] for k in oracle.MIMO_GRAD_NAMES])
    mimo_compare(got, ref, "mimo backward " + _id(w))
