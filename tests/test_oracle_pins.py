"""Pins for the CPU oracle: checks against what the source pages and plain
mathematics fix, never against the oracle itself or the CUDA path.

Source: oarust 0.8.6 `src/rs/ml/matrix/mamba3.rs` (operand layouts, limits,
state semantics of `mamba3_siso_step`, `num_groups == 0` rule, MIMO shapes and
the 1.0e-5 output-norm epsilon) and the `oa::ml::matrix` API reference
(`softplus` is overflow-safe; `rope` is split-half).
"""
import math

import numpy as np
import pytest

import oracle
from oracle.closed_form import closed_form_scan
from selective_state_space_mamba3_gb300 import inputs as gen

SCAN_KEYS = ("c", "b", "x", "z", "adt", "dt", "trap", "angle", "c_bias", "b_bias", "d")
MIMO_KEYS = ("mimo_x", "mimo_z", "mimo_o", "norm_weight")


def small(B=2, L=12, H=4, G=2, P=5, N=8, A=3, R=1, has_z=1, has_d=1, norm=0, seed=7):
    w = gen.Workload("pin", B, L, H, G, P, N, A, mimo_rank=R, has_z=has_z, has_d=has_d,
                     has_output_norm=norm, seed_index=seed)
    return w, gen.scan_inputs(w)


def run_scan(w, ins, **cfg_over):
    cfg = w.cfg(**cfg_over)
    mimo = {k: ins[k] for k in MIMO_KEYS if k in ins} if cfg["mimo_rank"] > 1 or cfg["has_output_norm"] else {}
    return oracle.scan(cfg, *[ins[k] for k in SCAN_KEYS], **mimo)


def rel(a, b):
    return np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300)


# --- pin 3: the token loop equals the materialised O(L^2) unrolled sum -------

@pytest.mark.parametrize("shape", [
    dict(),
    dict(B=1, L=9, H=2, G=0, P=3, N=6, A=3),        # 2A == N, num_groups 0
    dict(B=1, L=7, H=3, G=1, P=4, N=5, A=0),        # no rotation, odd N
    dict(B=1, L=10, H=2, G=2, P=2, N=4, A=1, has_z=0, has_d=0),
])
def test_siso_scan_equals_closed_form(shape):
    w, ins = small(**shape)
    got = run_scan(w, ins)
    cfg = w.cfg()
    ref = closed_form_scan(cfg["batch_size"], cfg["sequence_length"], cfg["num_heads"],
                           cfg["num_groups"], cfg["head_dim"], cfg["state_size"],
                           cfg["num_rope_angles"], 1, cfg["has_z"], cfg["has_d"], 0,
                           *[ins[k] for k in SCAN_KEYS])
    assert rel(got, ref) < 1e-12


@pytest.mark.parametrize("norm", [0, 1])
def test_mimo_scan_equals_closed_form(norm):
    w, ins = small(B=1, L=8, H=2, G=1, P=4, N=6, A=2, R=3, norm=norm)
    got = run_scan(w, ins)
    cfg = w.cfg()
    ref = closed_form_scan(cfg["batch_size"], cfg["sequence_length"], cfg["num_heads"],
                           cfg["num_groups"], cfg["head_dim"], cfg["state_size"],
                           cfg["num_rope_angles"], 3, 1, 1, norm,
                           *[ins[k] for k in SCAN_KEYS], *[ins[k] for k in MIMO_KEYS])
    assert rel(got, ref) < 1e-12


# --- hand-worked two-token example (brute force on the smallest case) --------

def test_two_token_hand_example():
    # B=1, L=2, H=1, G=1, P=1, N=2, A=1: one rotary pair, no gate, D=0.
    w = gen.Workload("hand", 1, 2, 1, 1, 1, 2, 1, has_z=0, has_d=0)
    c = np.array([1.0, 0.0, 0.5, 0.5], np.float32).reshape(1, 2, 1, 2)
    b = np.array([0.0, 1.0, 1.0, 0.0], np.float32).reshape(1, 2, 1, 2)
    x = np.array([2.0, -1.0], np.float32).reshape(1, 2, 1, 1)
    z = np.zeros((1, 2, 1, 1), np.float32)
    dt = np.array([0.5, 0.25], np.float32).reshape(1, 2, 1)
    adt = np.array([-0.5, -1.0], np.float32).reshape(1, 2, 1)
    trap = np.array([0.0, 0.0], np.float32).reshape(1, 2, 1)   # lambda = 1/2
    angle = np.array([math.pi / 2, 0.0], np.float32).reshape(1, 2, 1)
    zero_bias = np.zeros((1, 2), np.float32)
    d = np.zeros((1,), np.float32)
    got = oracle.scan(w.cfg(), c, b, x, z, adt, dt, trap, angle, zero_bias, zero_bias, d)
    # By hand, in float64 from the float32 inputs:
    # t=0: theta = 0.5*(pi/2 as float32); k0 = Rot(theta)(0,1) = (-sin, cos),
    #      q0 = Rot(theta)(1,0) = (cos, sin); h0 = gamma0*x0*k0, gamma0 = 0.25.
    #      y0 = h0.q0 = 0.25*2*(k0.q0) = 0 (orthogonal).
    th = 0.5 * float(np.float32(math.pi / 2))
    k0 = np.array([-math.sin(th), math.cos(th)])
    g0 = 0.25
    h0 = g0 * 2.0 * k0
    assert abs(got[0, 0, 0, 0] - h0 @ np.array([math.cos(th), math.sin(th)])) < 1e-15
    # t=1: theta unchanged (angle 0); k1 = Rot(th)(1,0), q1 = Rot(th)(.5,.5);
    #      h1 = e^{-1} h0 + s1 e^{-1} x0 k0 + gamma1 x1 k1, s1 = gamma1 = 0.125.
    k1 = np.array([math.cos(th), math.sin(th)])
    q1 = np.array([0.5 * math.cos(th) - 0.5 * math.sin(th), 0.5 * math.sin(th) + 0.5 * math.cos(th)])
    a1 = math.exp(-1.0)
    h1 = a1 * h0 + 0.125 * a1 * 2.0 * k0 + 0.125 * (-1.0) * k1
    assert abs(got[0, 1, 0, 0] - h1 @ q1) < 1e-15


# --- pin 2: Euler limit with zero angles is the plain diagonal selective scan

def textbook_selective_scan(x, B_, C_, adt, dt, D, z):
    """Discretised diagonal SSM (Mamba-2 / SSD form), zero-order-hold in A,
    Euler in B: h_t = exp(adt_t) h_{t-1} + dt_t x_t B_t^T, y_t = h_t C_t + D x_t,
    gated by silu(z). Shapes for one (b, h): x [L,P], B_/C_ [L,N]."""
    L, P = x.shape
    N = B_.shape[1]
    h = np.zeros((P, N))
    ys = []
    for t in range(L):
        h = math.exp(adt[t]) * h + dt[t] * np.outer(x[t], B_[t])
        y = h @ C_[t] + D * x[t]
        ys.append(y * z[t] / (1.0 + np.exp(-z[t])))
    return np.array(ys)


def test_euler_zero_angle_is_plain_selective_scan():
    w, ins = small(B=2, L=16, H=2, G=1, P=3, N=6, A=3)
    ins["trap"][:] = 40.0          # sigmoid(40) = 1 - 4e-18: pure current-token weight
    ins["angle"][:] = 0.0
    got = run_scan(w, ins)
    f = lambda a: a.astype(np.float64)
    for bb in range(2):
        for h in range(2):
            Bk = f(ins["b"][bb, :, 0]) + f(ins["b_bias"][h])
            Cq = f(ins["c"][bb, :, 0]) + f(ins["c_bias"][h])
            ref = textbook_selective_scan(f(ins["x"][bb, :, h]), Bk, Cq, f(ins["adt"][bb, :, h]),
                                          f(ins["dt"][bb, :, h]), float(ins["d"][h]),
                                          f(ins["z"][bb, :, h]))
            assert rel(got[bb, :, h], ref) < 1e-12


# --- pin 1: the step applied token by token equals the full scan ------------

@pytest.mark.parametrize("R", [1, 3])
def test_step_equals_scan(R):
    w, ins = small(B=2, L=10, H=2, G=1, P=4, N=6, A=2, R=R, norm=1 if R > 1 else 0)
    full = run_scan(w, ins)
    cfg1 = w.cfg(sequence_length=1)
    state = oracle.zero_state(cfg1)
    mimo = {k: ins[k] for k in MIMO_KEYS} if R > 1 else {}
    for t in range(w.sequence_length):
        tok = [np.ascontiguousarray(ins[k][:, t:t + 1]) for k in SCAN_KEYS[:8]]
        out = oracle.step(cfg1, *tok, ins["c_bias"], ins["b_bias"], ins["d"], state=state, **mimo)
        assert np.array_equal(out[:, 0], full[:, t])


@pytest.mark.parametrize("R", [1, 4])
def test_split_scan_with_state_equals_whole(R):
    """Scanning a sequence in two pieces, the second from the ssm / angle / k / v
    state the first returns, reproduces the one-piece scan exactly (the
    prefill -> prefill and prefill -> decode hand-off of the state API)."""
    w, ins = small(B=2, L=20, H=2, G=1, P=4, N=6, A=2, R=R, norm=1 if R > 1 else 0)
    full = run_scan(w, ins)
    mimo = {k: ins[k] for k in MIMO_KEYS} if R > 1 else {}
    state = oracle.zero_state(w.cfg(sequence_length=1))
    outs = []
    for t0, t1 in ((0, 7), (7, 20)):
        part = [np.ascontiguousarray(ins[k][:, t0:t1]) for k in SCAN_KEYS[:8]]
        outs.append(oracle.scan(w.cfg(sequence_length=t1 - t0), *part, ins["c_bias"],
                                ins["b_bias"], ins["d"], state=state, **mimo))
    assert np.array_equal(np.concatenate(outs, axis=1), full)


# --- pin 6: rotation only enters through angle differences ------------------

def test_angle_state_offset_invariance():
    w, ins = small(B=1, L=8, H=2, G=1, P=3, N=8, A=4)
    cfg1 = w.cfg(sequence_length=1)
    s0 = oracle.zero_state(cfg1)
    s1 = oracle.zero_state(cfg1)
    s1["angle"][:] = 1.234
    for t in range(8):
        tok = [np.ascontiguousarray(ins[k][:, t:t + 1]) for k in SCAN_KEYS[:8]]
        o0 = oracle.step(cfg1, *tok, ins["c_bias"], ins["b_bias"], ins["d"], state=s0)
        o1 = oracle.step(cfg1, *tok, ins["c_bias"], ins["b_bias"], ins["d"], state=s1)
        assert rel(o1, o0) < 1e-12


def test_full_turn_rotation_is_identity():
    # dt * angle = 2*pi per token: every rotation is a whole number of turns,
    # so the result equals the rotation-free scan with the same operands.
    w, ins = small(B=1, L=10, H=1, G=1, P=3, N=6, A=3)
    ins["angle"] = (2 * math.pi / ins["dt"][:, :, 0:1].astype(np.float64)).repeat(3, axis=2)
    got = run_scan(w, ins)
    ref = run_scan(w, dict(ins, angle=np.zeros_like(ins["angle"])))
    # float32(2*pi/dt) misses a whole turn by ~1e-7 rad per token; a broken
    # rotation or angle cumsum is off by O(1).
    assert rel(got, ref) < 1e-6


# --- pin 4: num_groups == 0 is one group per head; G < H shares rows --------

def test_groups_zero_equals_per_head():
    w, ins = small(B=1, L=6, H=3, G=0, P=2, N=4, A=1)
    a = run_scan(w, ins)
    b = run_scan(w.with_(num_groups=3), ins)
    assert np.array_equal(a, b)


def test_shared_groups_equal_duplicated_rows():
    w, ins = small(B=2, L=6, H=4, G=2, P=3, N=4, A=2)
    a = run_scan(w, ins)
    dup = dict(ins)
    dup["c"] = np.repeat(ins["c"], 2, axis=2)   # head h reads group h // 2
    dup["b"] = np.repeat(ins["b"], 2, axis=2)
    b = run_scan(w.with_(num_groups=4), dup)
    assert np.array_equal(a, b)


# --- pin 5: MIMO of rank 1 with unit projections and no norm is SISO --------

def test_mimo_rank1_is_siso():
    w, ins = small(B=1, L=9, H=2, G=1, P=4, N=6, A=2)
    siso = run_scan(w, ins)
    ones = np.ones((2, 1, 4), np.float32)
    mimo = oracle.scan(w.cfg(), *[ins[k] for k in SCAN_KEYS], mimo_x=ones, mimo_z=ones,
                       mimo_o=ones, norm_weight=np.ones((2, 4), np.float32))
    assert rel(mimo, siso) < 1e-14


# --- pin 7: output norm -----------------------------------------------------

def test_output_norm_rms():
    w, ins = small(B=1, L=7, H=2, G=1, P=6, N=4, A=1, R=2, norm=1)
    ins["norm_weight"][:] = 1.0
    normed = run_scan(w, ins)
    plain = run_scan(w, ins, has_output_norm=0)
    m = np.mean(plain ** 2, axis=-1)
    rms = np.sqrt(np.mean(normed ** 2, axis=-1))
    # RMS of v / sqrt(mean v^2 + eps) is sqrt(m / (m + eps)); direction unchanged.
    assert np.allclose(rms, np.sqrt(m / (m + 1e-5)), rtol=1e-12, atol=0)
    cos = np.sum(normed * plain, -1) / (np.linalg.norm(normed, axis=-1) * np.linalg.norm(plain, axis=-1))
    assert np.allclose(cos, 1.0, atol=1e-12)


# --- pin 9: degenerate cases --------------------------------------------------

def test_zero_keys_give_skip_only():
    w, ins = small(B=1, L=5, H=2, G=1, P=3, N=4, A=1)
    for k in ("c", "b", "c_bias", "b_bias"):
        ins[k] = np.zeros_like(ins[k])
    got = run_scan(w, ins)
    x = ins["x"].astype(np.float64)
    z = ins["z"].astype(np.float64)
    ref = ins["d"].astype(np.float64)[None, None, :, None] * x * z / (1 + np.exp(-z))
    assert rel(got, ref) < 1e-15


def test_linear_in_x_without_gate():
    w, ins = small(B=1, L=8, H=2, G=1, P=3, N=4, A=2, has_z=0, has_d=1)
    a = run_scan(w, ins)
    b = run_scan(w, dict(ins, x=ins["x"] * 2))
    assert rel(b, 2 * a) < 1e-14


# --- pin 8: preprocess -------------------------------------------------------

def test_preprocess_closed_forms():
    w = gen.TINY_SISO
    p = gen.tiny_projection(w)
    proj, dtb = p["projected"], p["dt_bias"]
    # make the extremes of the dt clamp and the A floor occur
    o = 2 * 32 + 2 * 16
    proj[0, o:o + 2] = [-30.0, 30.0]        # dt_raw: below dt_min, above dt_max
    proj[1, o + 2:o + 4] = [-40.0, 0.0]     # a_raw: softplus(-40) < a_floor
    kw = dict(inner_size=32, state_size=16, num_heads=2, num_rope_angles=8, num_groups=1,
              mimo_rank=1, **gen.TINY_PRE)
    out = oracle.preprocess(proj, dtb, **kw)
    f = proj.astype(np.float64)
    assert np.array_equal(out["z"], f[:, 0:32]) and np.array_equal(out["x"], f[:, 32:64])
    for key, off in (("bh", 64), ("ch", 80)):
        raw = f[:, off:off + 16]
        ms_raw = np.mean(raw ** 2, axis=1)
        ms_out = np.mean(out[key] ** 2, axis=1)
        # mean square of v / sqrt(m + eps) is m / (m + eps), direction kept
        assert np.allclose(ms_out, ms_raw / (ms_raw + np.float64(np.float32(1e-6))), rtol=1e-13)
        assert np.allclose(out[key] * np.sqrt(ms_raw + np.float64(np.float32(1e-6)))[:, None], raw,
                           rtol=1e-12, atol=1e-14)
    dt = out["dt"]
    lo, hi = float(np.float32(1e-3)), float(np.float32(0.1))
    assert np.all(dt >= lo) and np.all(dt <= hi)
    assert dt[0, 0] == lo and dt[0, 1] == hi
    sp = np.logaddexp(0.0, f[:, o:o + 2] + dtb.astype(np.float64)[None])   # library softplus
    inside = (sp > lo) & (sp < hi)
    assert np.allclose(dt[inside], sp[inside], rtol=1e-14)
    floor = float(np.float32(1e-4))
    a_mag = np.maximum(np.logaddexp(0.0, f[:, o + 2:o + 4]), floor)
    assert np.allclose(out["adt"], -a_mag * dt, rtol=1e-14)
    assert np.all(out["adt"] <= -floor * dt)
    assert out["adt"][1, 0] == -floor * dt[1, 0]
    assert np.array_equal(out["trap"], f[:, o + 4:o + 6])
    assert np.array_equal(out["angle"], f[:, o + 6:o + 14])


def test_preprocess_softplus_overflow_safe():
    kw = dict(inner_size=4, state_size=4, num_heads=1, num_rope_angles=0, num_groups=1,
              mimo_rank=1, epsilon=1e-6, dt_min=1e-3, dt_max=1e30, a_floor=1e-4)
    proj = np.zeros((2, 4 + 4 + 8 + 3), np.float32)
    proj[:, 16] = [80.0, 1e30]      # dt_raw huge: softplus(v) = v, no overflow
    out = oracle.preprocess(proj, np.zeros((1,), np.float32), **kw)
    assert out["dt"][0, 0] == 80.0 and out["dt"][1, 0] == float(np.float32(1e30))
    assert np.all(np.isfinite(out["adt"]))


# --- regression fixture: the tiny workload's chained output (tests/golden) ---

def test_tiny_golden_fixture():
    """The oracle still reproduces tests/golden/tiny_siso_chain.txt, its own
    output for the tiny SISO workload (preprocess chained into the scan),
    frozen by tests/golden/make_golden.py: a change to the oracle's arithmetic
    shows up here and must be justified before the fixture is rewritten."""
    import importlib.util
    import os
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "make_golden.py")
    spec = importlib.util.spec_from_file_location("make_golden", path)
    mg = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mg)
    ref = np.loadtxt(mg.FIXTURE)
    got = np.asarray(mg.tiny_chain_output(), np.float64).ravel()
    assert ref.shape == got.shape == (2048,)
    assert np.max(np.abs(got - ref)) <= 1e-12 * np.max(np.abs(ref))
