"""GPU parity of m3_siso_backward (oarust mamba3.rs `mamba3_siso_backward`, the
eleven adjoints of `SsmBackward`) against the oracle's reverse-mode adjoints
(`m3o_siso_backward`, itself pinned to central differences of the forward
oracle), on the same seeded inputs and output gradient.

Bar: the FP32 bar of the forward, 1e-5 normwise (max|gpu - oracle| / max|oracle|
per gradient), for all eleven gradients. The two gradients that vanish in
exact arithmetic with a single token from a zero state (the angle adjoint:
q_t . k_t does not depend on theta_t; d adt: the state then holds no decayed
term) are compared against a floor of 1e-2 times the call's largest
per-token gradient instead of their own rounding residue: the kernels form
them as differences of terms of that size, whose rounding is absolute. Outputs start as NaN, so an
element the kernels never write fails the comparison.
"""
import numpy as np
import pytest

import oracle
import selective_state_space_mamba3_gb300 as m3
from selective_state_space_mamba3_gb300 import inputs as gen

from m3_testutil import check_close, dev, normwise

pytestmark = pytest.mark.gpu

KEYS = oracle.GRAD_NAMES  # c, b, x, z, adt, dt, trap, angle, c_bias, b_bias, d
# FP32 sweeps against the FP64 oracle: the state and adjoint-state sums are
# those of the FP32 forward (a few 1e-7 of the largest element); d adt, d dt
# and d angle add running sums over the later tokens (measured at most 1.7e-6
# at L = 2048).
BWD_TOL = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _built():
    from selective_state_space_mamba3_gb300 import build
    build.build()
    oracle.build()


def grad_shapes(cfg):
    B, L, H = cfg["batch_size"], cfg["sequence_length"], cfg["num_heads"]
    P, N, A = cfg["head_dim"], cfg["state_size"], cfg["num_rope_angles"]
    G = cfg["num_groups"] or H
    return dict(c=(B, L, G, N), b=(B, L, G, N), x=(B, L, H, P), z=(B, L, H, P), adt=(B, L, H),
                dt=(B, L, H), trap=(B, L, H), angle=(B, L, A), c_bias=(H, N), b_bias=(H, N),
                d=(H,))


def gpu_backward(cfg, ins, dout, calls=1):
    """m3_siso_backward through the C ABI; returns {name: float32 array} (and,
    with calls > 1, asserts that every call gives the same bits)."""
    import torch
    c = m3.ssm_config(cfg, m3.M3_MATH_FP32)
    d = {k: dev(ins[k]) for k in KEYS}
    if cfg["num_rope_angles"] == 0:
        d["angle"] = None
    go = dev(dout)
    wsb = m3.m3_siso_backward_workspace(c)
    assert wsb > 0
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    first = None
    for _ in range(calls):
        g = {k: torch.full(s, float("nan"), device="cuda") for k, s in grad_shapes(cfg).items()}
        if cfg["num_rope_angles"] == 0:
            g["angle"] = None
        m3.m3_siso_backward(c, go, *[d[k] for k in KEYS], *[g[k] for k in KEYS], ws)
        torch.cuda.synchronize()
        got = {k: (np.zeros(grad_shapes(cfg)[k], np.float32) if g[k] is None else g[k].cpu().numpy())
               for k in KEYS}
        if first is None:
            first = got
        else:
            for k in KEYS:
                assert np.array_equal(first[k], got[k]), f"call-to-call difference in {k}"
    return first


# the per-token gradients, whose scale sets the floor for a gradient that
# vanishes (the parameter gradients sum over all tokens and are larger)
PER_TOKEN = ("c", "b", "x", "z", "adt", "dt", "trap")


# gradients that vanish in exact arithmetic when every sequence has one token
VANISH_AT_L1 = ("adt", "angle")


def compare(got, ref, label, tol=BWD_TOL):
    floor = 1e-2 * max(float(np.max(np.abs(ref[k]))) for k in PER_TOKEN)
    one_token = ref["x"].shape[1] == 1
    for k in KEYS:
        if ref[k].size == 0:
            continue
        assert np.all(np.isfinite(got[k])), f"{label} {k}: unwritten or non-finite elements"
        if one_token and k in VANISH_AT_L1:
            err = float(np.max(np.abs(got[k].astype(np.float64) - ref[k]))) / floor
            assert err <= tol, (label, k, "against the floor", err)
        else:
            check_close(got[k], ref[k], tol, f"{label} grad {k}")


def case(B, L, H, G, P, N, A, has_z=1, has_d=1, seed=70):
    w = gen.Workload("bwd", B, L, H, G, P, N, A, has_z=has_z, has_d=has_d, seed_index=seed)
    ins = gen.scan_inputs(w)
    ins["d"] = np.linspace(0.5, 1.5, H, dtype=np.float32)  # a skip weight per head
    return w.cfg(), ins, gen.output_gradient(w)


CASES = {
    # the tiny workload's shape
    "tiny": dict(B=1, L=64, H=2, G=1, P=16, N=16, A=8),
    # heads sharing a group; a ragged last tile (100 = 6 x 16 + 4)
    "groups_ragged": dict(B=2, L=100, H=4, G=2, P=32, N=64, A=16),
    # one group per head (num_groups 0), every dim rotated, no gate
    "g0_full_rotation": dict(B=1, L=33, H=3, G=0, P=24, N=48, A=24, has_z=0),
    # no rotation, no skip, sizes that are not multiples of 4
    "plain_odd": dict(B=2, L=17, H=2, G=1, P=8, N=12, A=0, has_d=0),
    # a single token per sequence
    "one_token": dict(B=3, L=1, H=2, G=2, P=64, N=128, A=32),
    # the largest state, P = N = 128
    "p128_n128": dict(B=1, L=40, H=2, G=1, P=128, N=128, A=64),
    # one head (its angle gradient is written directly), P = N = 100
    "one_head_p100": dict(B=1, L=20, H=1, G=1, P=100, N=100, A=50),
    # the 1B-layer head shape on a shorter sequence
    "layer_short": dict(B=2, L=256, H=8, G=1, P=64, N=128, A=32),
    # the long-context head shape (G = 4, A = 64) on a shorter sequence
    "long_short": dict(B=1, L=300, H=8, G=4, P=64, N=128, A=64),
}


@pytest.mark.parametrize("name", list(CASES))
def test_siso_backward_matches_oracle(name):
    cfg, ins, dout = case(**CASES[name])
    got = gpu_backward(cfg, ins, dout, calls=2)
    ref = oracle.siso_backward(cfg, dout, *[ins[k] for k in KEYS])
    compare(got, ref, name)


def test_siso_backward_1b_layer_sampled():
    """The SISO 1B-layer workload (B8 L2048 H32 G1 P64 N128 A32), in the
    launch configuration the benchmark times: every gradient of batch row 0
    against the oracle run on that row (the rows are independent up to the
    bias and D sums), and the batch sums checked by properties that hold at
    any size: sum_h d c_bias[h] = sum over all (b, t) of d C (both sum the
    same per-head terms), and d D[h] = sum_{b,t,p} dout silu(z) x."""
    w = gen.SISO_1B
    cfg, ins = w.cfg(), gen.scan_inputs(w)
    dout = gen.output_gradient(w)
    got = gpu_backward(cfg, ins, dout)
    row = slice(0, 1)
    cfg1 = dict(cfg, batch_size=1)
    ins1 = {k: (v[row] if k in KEYS[:8] else v) for k, v in ins.items()}
    ref = oracle.siso_backward(cfg1, dout[row], *[ins1[k] for k in KEYS])
    for k in KEYS[:8]:
        assert np.all(np.isfinite(got[k])), k
        check_close(got[k][row], ref[k], BWD_TOL, f"1b row 0 grad {k}")
    for k, src in (("c_bias", "c"), ("b_bias", "b")):
        lhs = got[k].astype(np.float64).sum(axis=0)
        rhs = got[src].astype(np.float64).sum(axis=(0, 1, 2))
        assert normwise(lhs, rhs) < 1e-5, k
    z = ins["z"].astype(np.float64)
    dd = np.sum(dout * z / (1 + np.exp(-z)) * ins["x"], axis=(0, 1, 3))
    check_close(got["d"], dd, BWD_TOL, "1b grad d (closed form)")


def test_siso_backward_rejects_bad_calls():
    """Host checks: MIMO rank, output norm, a short workspace and a NULL
    gradient are refused before anything is enqueued."""
    import ctypes
    import torch
    cfg, ins, dout = case(**CASES["tiny"])
    lib = m3.load_library()
    good = m3.ssm_config(cfg, m3.M3_MATH_FP32)
    n = ctypes.c_size_t(0)
    for bad in (dict(mimo_rank=2), dict(has_output_norm=1), dict(head_dim=129)):
        c = m3.ssm_config(dict(cfg, **bad), m3.M3_MATH_FP32)
        assert lib.m3_siso_backward_workspace(ctypes.byref(c), ctypes.byref(n)) == \
            m3.M3_ERR_INVALID_ARGUMENT
    wsb = m3.m3_siso_backward_workspace(good)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    d = {k: dev(ins[k]) for k in KEYS}
    g = {k: torch.zeros(s, device="cuda") for k, s in grad_shapes(cfg).items()}
    args = [d[k] for k in KEYS] + [g[k] for k in KEYS]
    with pytest.raises(m3.M3Error) as e:
        m3.m3_siso_backward(good, dev(dout), *args, ws[: wsb - 256])
    assert e.value.status == m3.M3_ERR_WORKSPACE
    args[KEYS.index("x") + len(KEYS)] = None
    with pytest.raises(m3.M3Error) as e:
        m3.m3_siso_backward(good, dev(dout), *args, ws)
    assert e.value.status == m3.M3_ERR_INVALID_ARGUMENT


# --- MIMO adjoints (`mamba3_mimo_backward`, the fifteen of `Mamba3MimoBackward`)

MKEYS = oracle.MIMO_GRAD_NAMES


def mimo_grad_shapes(cfg):
    B, L, H = cfg["batch_size"], cfg["sequence_length"], cfg["num_heads"]
    P, N, A, R = cfg["head_dim"], cfg["state_size"], cfg["num_rope_angles"], cfg["mimo_rank"]
    G = cfg["num_groups"] or H
    return dict(c=(B, L, R * G, N), b=(B, L, R * G, N), x=(B, L, H, P), z=(B, L, H, P),
                adt=(B, L, H), dt=(B, L, H), trap=(B, L, H), angle=(B, L, A), c_bias=(H, R, N),
                b_bias=(H, R, N), d=(H,), mimo_x=(H, R, P), mimo_z=(H, R, P), mimo_o=(H, R, P),
                norm_weight=(H, P))


def gpu_mimo_backward(cfg, ins, dout, calls=1):
    import torch
    c = m3.ssm_config(cfg, m3.M3_MATH_FP32)
    d = {k: dev(ins[k]) for k in MKEYS}
    if cfg["num_rope_angles"] == 0:
        d["angle"] = None
    go = dev(dout)
    ws = torch.empty(m3.m3_mimo_backward_workspace(c), dtype=torch.uint8, device="cuda")
    first = None
    for _ in range(calls):
        g = {k: torch.full(s, float("nan"), device="cuda") for k, s in mimo_grad_shapes(cfg).items()}
        if cfg["num_rope_angles"] == 0:
            g["angle"] = None
        m3.m3_mimo_backward(c, go, *[d[k] for k in MKEYS], *[g[k] for k in MKEYS], ws)
        torch.cuda.synchronize()
        got = {k: (np.zeros(mimo_grad_shapes(cfg)[k], np.float32) if g[k] is None
                   else g[k].cpu().numpy()) for k in MKEYS}
        if first is None:
            first = got
        else:
            for k in MKEYS:
                assert np.array_equal(first[k], got[k]), f"call-to-call difference in {k}"
    return first


def mimo_compare(got, ref, label, tol=BWD_TOL):
    floor = 1e-2 * max(float(np.max(np.abs(ref[k]))) for k in PER_TOKEN)
    one_token = ref["x"].shape[1] == 1
    for k in MKEYS:
        if ref[k].size == 0:
            continue
        assert np.all(np.isfinite(got[k])), f"{label} {k}: unwritten or non-finite elements"
        if one_token and k in VANISH_AT_L1:
            err = float(np.max(np.abs(got[k].astype(np.float64) - ref[k]))) / floor
            assert err <= tol, (label, k, "against the floor", err)
        else:
            check_close(got[k], ref[k], tol, f"{label} grad {k}")


def mimo_case(B, L, H, G, P, N, A, R, norm, has_z=1, has_d=1, seed=80):
    w = gen.Workload("mbwd", B, L, H, G, P, N, A, mimo_rank=R, has_z=has_z, has_d=has_d,
                     has_output_norm=norm, seed_index=seed)
    ins = gen.scan_inputs(w)
    ins["d"] = np.linspace(0.5, 1.5, H, dtype=np.float32)
    return w.cfg(), ins, gen.output_gradient(w)


MIMO_CASES = {
    # the MIMO R4 workload's head shape with the norm, on a shorter sequence
    "r4_norm": dict(B=1, L=40, H=2, G=1, P=64, N=64, A=32, R=4, norm=1),
    # rank 2 without the norm, heads sharing groups, a ragged last tile
    "r2_groups": dict(B=2, L=33, H=4, G=2, P=32, N=32, A=8, R=2, norm=0),
    # rank 3 (the rank-4 instance with three ranks), no gate, odd sizes
    "r3_odd": dict(B=1, L=21, H=2, G=1, P=24, N=20, A=5, R=3, norm=1, has_z=0),
    # rank 8
    "r8": dict(B=1, L=17, H=1, G=1, P=16, N=16, A=4, R=8, norm=1),
    # rank 1 with the norm and N = 128
    "r1_norm_n128": dict(B=1, L=30, H=2, G=2, P=16, N=128, A=32, R=1, norm=1),
    # rank 5, P N = 4000, no skip, A = 0
    "r5_p40_n100": dict(B=1, L=12, H=2, G=1, P=40, N=100, A=0, R=5, norm=0, has_d=0),
}


@pytest.mark.parametrize("name", list(MIMO_CASES))
def test_mimo_backward_matches_oracle(name):
    cfg, ins, dout = mimo_case(**MIMO_CASES[name])
    got = gpu_mimo_backward(cfg, ins, dout, calls=2)
    ref = oracle.mimo_backward(cfg, dout, *[ins[k] for k in MKEYS])
    mimo_compare(got, ref, name)


def test_mimo_backward_r4_workload():
    """The MIMO R4 workload (B4 L4096 H32 G1 P64 N64 A32 R4 with the output
    norm) whole: every one of the fifteen gradients against the oracle."""
    w = gen.MIMO_R4
    cfg, ins = w.cfg(), gen.scan_inputs(w)
    dout = gen.output_gradient(w)
    got = gpu_mimo_backward(cfg, ins, dout)
    ref = oracle.mimo_backward(cfg, dout, *[ins[k] for k in MKEYS])
    mimo_compare(got, ref, "mimo r4 workload")


def test_siso_backward_long_context_heads():
    """The long-context head shape (G4 P64 N128 A64) over 4,096 tokens of 8
    heads: one 512-thread sweep block per sequence (fewer sequences than SMs),
    256 tiles carried in order, every gradient against the oracle."""
    cfg, ins, dout = case(B=1, L=4096, H=8, G=4, P=64, N=128, A=64, seed=73)
    got = gpu_backward(cfg, ins, dout)
    ref = oracle.siso_backward(cfg, dout, *[ins[k] for k in KEYS], threads=8)
    compare(got, ref, "long-context heads")


@pytest.mark.parametrize("mimo", [False, True], ids=["siso", "mimo"])
def test_autograd_binding(mimo):
    """selective_state_space_mamba3_gb300.autograd: loss = sum(out * W) through
    torch.autograd; the .grad of every operand equals the oracle's adjoints for
    grad_out = W, and the forward equals the oracle's scan."""
    import torch
    from selective_state_space_mamba3_gb300 import autograd as m3ag
    if mimo:
        cfg, ins, dout = mimo_case(B=1, L=40, H=2, G=1, P=32, N=32, A=8, R=2, norm=1)
        keys = MKEYS
    else:
        cfg, ins, dout = case(B=2, L=50, H=4, G=2, P=16, N=32, A=8)
        keys = KEYS
    t = {k: dev(ins[k]).requires_grad_(True) for k in keys}
    fn = m3ag.mimo_scan if mimo else m3ag.siso_scan
    out = fn(cfg, *[t[k] for k in keys])
    (out * dev(dout)).sum().backward()
    torch.cuda.synchronize()
    if mimo:
        ref = oracle.mimo_backward(cfg, dout, *[ins[k] for k in keys])
        ref_out = oracle.scan(cfg, *[ins[k] for k in KEYS], **{k: ins[k] for k in MKEYS[11:]})
    else:
        ref = oracle.siso_backward(cfg, dout, *[ins[k] for k in keys])
        ref_out = oracle.scan(cfg, *[ins[k] for k in KEYS])
    check_close(out.detach().cpu().numpy(), ref_out, BWD_TOL, "autograd forward")
    for k in keys:
        check_close(t[k].grad.cpu().numpy(), ref[k], BWD_TOL, f"autograd grad {k}")


def test_autograd_preprocess_into_scan():
    """The tiny workload trained end to end through the autograd binding:
    preprocess -> SISO scan -> sum(out * W). The projection and dt_bias
    gradients equal the oracle's chain (the scan adjoints of the oracle's
    preprocess outputs, fed to the oracle's preprocess adjoint)."""
    import torch
    from selective_state_space_mamba3_gb300 import autograd as m3ag
    w = gen.TINY_SISO
    p = gen.tiny_projection(w)
    pkw = dict(inner_size=32, state_size=16, num_heads=2, num_rope_angles=8, num_groups=1,
               mimo_rank=1, **gen.TINY_PRE)
    cfg = w.cfg()
    dout = gen.output_gradient(w)
    proj = dev(p["projected"]).requires_grad_(True)
    dtb = dev(p["dt_bias"]).requires_grad_(True)
    x, z, bh, ch, dt, adt, trap, angle = m3ag.preprocess(pkw, proj, dtb)
    shp = lambda t, *s: t.reshape(*s)
    out = m3ag.siso_scan(cfg, shp(ch, 1, 64, 1, 16), shp(bh, 1, 64, 1, 16), shp(x, 1, 64, 2, 16),
                         shp(z, 1, 64, 2, 16), shp(adt, 1, 64, 2), shp(dt, 1, 64, 2),
                         shp(trap, 1, 64, 2), shp(angle, 1, 64, 8), dev(p["c_bias"]),
                         dev(p["b_bias"]), dev(p["d"]))
    (out * dev(dout)).sum().backward()
    torch.cuda.synchronize()
    pre = oracle.preprocess(p["projected"], p["dt_bias"], **pkw)
    f = lambda k, *s: pre[k].astype(np.float32).reshape(s)
    sc = dict(c=f("ch", 1, 64, 1, 16), b=f("bh", 1, 64, 1, 16), x=f("x", 1, 64, 2, 16),
              z=f("z", 1, 64, 2, 16), adt=f("adt", 1, 64, 2), dt=f("dt", 1, 64, 2),
              trap=f("trap", 1, 64, 2), angle=f("angle", 1, 64, 8), c_bias=p["c_bias"],
              b_bias=p["b_bias"], d=p["d"])
    g = oracle.siso_backward(cfg, dout, *[sc[k] for k in KEYS])
    pg = {"x": g["x"].reshape(64, 32), "z": g["z"].reshape(64, 32), "bh": g["b"].reshape(64, 16),
          "ch": g["c"].reshape(64, 16), "dt": g["dt"].reshape(64, 2), "adt": g["adt"].reshape(64, 2),
          "trap": g["trap"].reshape(64, 2), "angle": g["angle"].reshape(64, 8)}
    ref = oracle.preprocess_backward(p["projected"], p["dt_bias"], pg, **pkw)
    check_close(proj.grad.cpu().numpy(), ref["projected"], BWD_TOL, "autograd d projected")
    check_close(dtb.grad.cpu().numpy(), ref["dt_bias"], BWD_TOL, "autograd d dt_bias")
