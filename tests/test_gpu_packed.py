"""GPU parity of m3_siso_forward_packed / m3_mimo_forward_packed: the scans of a
packed input projection (oarust mamba3.rs `mamba3_preprocess` feeding
`mamba3_siso` / `mamba3_mimo`).

Where the chunked kernel reads the packed rows itself (SISO P = 64, N = 128,
A = 32 or 64, W a multiple of 4), its output must have the bits of
m3_preprocess followed by the scan in the same math mode; every other SISO
shape, and every MIMO shape, goes through the preprocess kernel and a
workspace, with the same result. Both are also held to the oracle's preprocess -> scan chain at the
mode's bar (FP32-exact 1e-5, TF32 2e-3), on the first and last batch rows."""
import numpy as np
import pytest

import oracle
import selective_state_space_mamba3_gb300 as m3
from selective_state_space_mamba3_gb300 import inputs as gen

from m3_testutil import TOL, dev, check_close

pytestmark = pytest.mark.gpu
FP32, TF32 = m3.M3_MATH_FP32, m3.M3_MATH_TF32


@pytest.fixture(scope="module", autouse=True)
def _built():
    from selective_state_space_mamba3_gb300 import build
    build.build()
    oracle.build()


MIMO_PAR = ("mimo_x", "mimo_z", "mimo_o", "norm_weight")


def pre_kw(w, pre):
    G = w.num_heads if w.num_groups == 0 else w.num_groups
    return dict(inner_size=w.num_heads * w.head_dim, state_size=w.state_size,
                num_heads=w.num_heads, num_rope_angles=w.num_rope_angles, num_groups=G,
                mimo_rank=w.mimo_rank, **pre)


def is_mimo(w):
    return w.mimo_rank > 1 or w.has_output_norm


def run_both(w, proj, dt_bias, par, mode, pre):
    """(packed entry output, m3_preprocess + scan output)."""
    import torch
    B, L, H, P, N, A, R = (w.batch_size, w.sequence_length, w.num_heads, w.head_dim,
                           w.state_size, w.num_rope_angles, w.mimo_rank)
    G = H if w.num_groups == 0 else w.num_groups
    mimo = is_mimo(w)
    cfg = m3.ssm_config(w.cfg(), mode)
    pcfg = m3.preprocess_config(**pre_kw(w, pre))
    dp, db = dev(proj), dev(dt_bias)
    cb, bb, d = dev(par["c_bias"]), dev(par["b_bias"]), dev(par["d"])
    mp = [dev(par[k]) for k in MIMO_PAR] if mimo else []
    out = torch.full((B, L, H, P), float("nan"), device="cuda")
    if mimo:
        nws = m3.m3_mimo_forward_packed_workspace(cfg, pcfg)
        ws = torch.empty(max(nws, 16), dtype=torch.uint8, device="cuda")
        m3.m3_mimo_forward_packed(cfg, pcfg, dp, db, cb, bb, d, *mp, out, ws)
    else:
        nws = m3.m3_siso_forward_packed_workspace(cfg, pcfg)
        ws = torch.empty(max(nws, 16), dtype=torch.uint8, device="cuda")
        m3.m3_siso_forward_packed(cfg, pcfg, dp, db, cb, bb, d, out, ws)
    e = lambda *s: torch.empty(*s, device="cuda")
    x, z = e(B, L, H, P), e(B, L, H, P)
    bh, ch = e(B, L, G * R, N), e(B, L, G * R, N)
    dt, adt, trap = e(B, L, H), e(B, L, H), e(B, L, H)
    ang = e(B, L, A) if A else None
    m3.m3_preprocess(pcfg, B * L, dp, db, x, z, bh, ch, dt, adt, trap, ang)
    out2 = torch.full_like(out, float("nan"))
    if mimo:
        nws2 = m3.m3_mimo_forward_workspace(cfg)
        ws2 = torch.empty(max(nws2, 16), dtype=torch.uint8, device="cuda")
        m3.m3_mimo_forward(cfg, ch, bh, x, z, adt, dt, trap, ang, cb, bb, d, *mp, out2, ws2)
    else:
        nws2 = m3.m3_siso_forward_workspace(cfg)
        ws2 = torch.empty(max(nws2, 16), dtype=torch.uint8, device="cuda")
        m3.m3_siso_forward(cfg, ch, bh, x, z, adt, dt, trap, ang, cb, bb, d, out2, ws2)
    torch.cuda.synchronize()
    assert m3.m3_workspace_status(ws) == m3.M3_OK
    return out.cpu().numpy(), out2.cpu().numpy()


def oracle_chain(w, proj, dt_bias, par, pre, bsl):
    """The oracle's preprocess of batch rows `bsl`, then its scan."""
    L, H, P, N, A, R = (w.sequence_length, w.num_heads, w.head_dim, w.state_size,
                        w.num_rope_angles, w.mimo_rank)
    G = H if w.num_groups == 0 else w.num_groups
    nb = bsl.stop - bsl.start
    rows = proj.reshape(w.batch_size, L, -1)[bsl].reshape(nb * L, -1)
    o = oracle.preprocess(rows, dt_bias, **pre_kw(w, pre))
    f = lambda k, *s: o[k].astype(np.float32).reshape(nb, L, *s)
    extra = {k: par[k] for k in MIMO_PAR} if is_mimo(w) else {}
    return oracle.scan(w.cfg(batch_size=nb), f("ch", G * R, N), f("bh", G * R, N), f("x", H, P),
                       f("z", H, P), f("adt", H), f("dt", H), f("trap", H),
                       f("angle", A) if A else np.zeros((nb, L, 0), np.float32),
                       par["c_bias"], par["b_bias"], par["d"], **extra)


CASES = {
    # fused: the 1B-layer shape with two batch rows (W = 4480)
    "fused_siso_layer": (gen.SISO_1B.with_(batch_size=2), gen.PRE_DEFAULT),
    # fused, long sequences split into segments (A = 64, G = 4; W = 5280)
    "fused_long_segments": (gen.SISO_LONG.with_(batch_size=1, sequence_length=4096),
                            gen.PRE_DEFAULT),
    # fused, a ragged last chunk and two heads per group
    "fused_ragged": (gen.Workload("packed ragged", 2, 1000, 4, 2, 64, 128, 32, seed_index=51),
                     dict(epsilon=1e-5, dt_min=2e-3, dt_max=0.2, a_floor=0.5)),
    # preprocess + scan through the workspace: W = 110 is not a multiple of 4
    "workspace_tiny": (gen.TINY_SISO, gen.TINY_PRE),
    # MIMO: the R4 workload's shape with two batch rows and 1,000 tokens
    "mimo_r4": (gen.MIMO_R4.with_(batch_size=2, sequence_length=1000), gen.PRE_DEFAULT),
    # MIMO: rank 2, no compile-time instance of the scan
    "mimo_r2": (gen.Workload("packed MIMO R2", 1, 300, 4, 2, 32, 32, 8, mimo_rank=2,
                                       has_output_norm=1, seed_index=52), gen.PRE_DEFAULT),
}


@pytest.mark.parametrize("mode", [FP32, TF32])
@pytest.mark.parametrize("case", list(CASES))
def test_packed_scan(case, mode):
    w, pre = CASES[case]
    if case == "workspace_tiny":
        p = gen.tiny_projection(w)
        proj, dt_bias = p["projected"], p["dt_bias"]
        par = {k: p[k] for k in ("c_bias", "b_bias", "d")}
    else:
        p = gen.layer_projection(w)
        proj, dt_bias = p["projected"], p["dt_bias"]
        par = gen.scan_params(w)
    got, two_step = run_both(w, proj, dt_bias, par, mode, pre)
    assert np.all(np.isfinite(got))
    assert np.array_equal(got, two_step), np.max(np.abs(got - two_step))
    for bsl in (slice(0, 1), slice(w.batch_size - 1, w.batch_size)):
        ref = oracle_chain(w, proj, dt_bias, par, pre, bsl)
        check_close(got[bsl], ref, TOL[mode], label=f"{case} batch {bsl.start}")
