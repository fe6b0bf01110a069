"""GPU parity: every entry point of libm3, called through its C ABI, against
the CPU oracle on the same seeded inputs (oarust mamba3.rs operations:
`mamba3_preprocess`, `mamba3_siso`, `mamba3_mimo`, `mamba3_siso_step`,
`mamba3_mimo_step`).

Bars: preprocess outputs elementwise (slices bit-exact, transforms within a
few float32 ulps); scans normwise max-relative error <= 1e-5 in FP32-exact
mode and <= 2e-3 in TF32 mode. Full-size workloads run entirely on the GPU
and are compared on the batch rows the oracle recomputes.
"""
import numpy as np
import pytest

import oracle
import selective_state_space_mamba3_gb300 as m3
from selective_state_space_mamba3_gb300 import inputs as gen

from m3_testutil import (SCAN_KEYS, MIMO_KEYS, TOL, dev, normwise, gpu_scan, oracle_scan,
                         check_close)

pytestmark = pytest.mark.gpu
FP32, TF32 = m3.M3_MATH_FP32, m3.M3_MATH_TF32


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    from selective_state_space_mamba3_gb300 import build
    build.build()
    oracle.build()
    assert torch.cuda.is_available()


# ---------------------------------------------------------------- preprocess

def gpu_preprocess(proj, dt_bias, **kw):
    import torch
    rows = proj.shape[0]
    I, N, H, A = kw["inner_size"], kw["state_size"], kw["num_heads"], kw["num_rope_angles"]
    GRN = kw["num_groups"] * kw["mimo_rank"] * N
    shapes = dict(x=(rows, I), z=(rows, I), bh=(rows, GRN), ch=(rows, GRN), dt=(rows, H),
                  adt=(rows, H), trap=(rows, H), angle=(rows, A))
    outs = {k: torch.full(s, float("nan"), device="cuda") for k, s in shapes.items()}
    m3.m3_preprocess(m3.preprocess_config(**kw), rows, dev(proj), dev(dt_bias),
                     *[outs[k] for k in ("x", "z", "bh", "ch", "dt", "adt", "trap", "angle")])
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in outs.items()}


def check_preprocess(got, ref):
    for k in ("x", "z", "trap", "angle"):
        assert np.array_equal(got[k].astype(np.float64), ref[k]), k
    for k in ("bh", "ch", "dt", "adt"):
        err = np.max(np.abs(got[k] - ref[k]) / (np.abs(ref[k]) + 1e-30))
        assert err < 2e-6, (k, err)


def test_preprocess_tiny_unaligned_width():
    w = gen.TINY_SISO
    p = gen.tiny_projection(w)
    kw = dict(inner_size=32, state_size=16, num_heads=2, num_rope_angles=8, num_groups=1,
              mimo_rank=1, **gen.TINY_PRE)
    assert p["projected"].shape[1] == 110      # W not a multiple of 4: scalar path
    check_preprocess(gpu_preprocess(p["projected"], p["dt_bias"], **kw),
                     oracle.preprocess(p["projected"], p["dt_bias"], **kw))


@pytest.mark.parametrize("w", [gen.SISO_1B, gen.MIMO_R4, gen.SISO_LONG],
                         ids=["siso_layer", "mimo_layer", "long_context_layer"])
def test_preprocess_layer_shape(w):
    p = gen.layer_projection(w)
    kw = dict(inner_size=w.num_heads * w.head_dim, state_size=w.state_size,
              num_heads=w.num_heads, num_rope_angles=w.num_rope_angles,
              num_groups=w.num_groups, mimo_rank=w.mimo_rank, **gen.PRE_DEFAULT)
    check_preprocess(gpu_preprocess(p["projected"], p["dt_bias"], **kw),
                     oracle.preprocess(p["projected"], p["dt_bias"], **kw))


def test_preprocess_odd_state_and_groups():
    rng = np.random.default_rng(5)
    kw = dict(inner_size=24, state_size=17, num_heads=3, num_rope_angles=5, num_groups=3,
              mimo_rank=2, epsilon=1e-5, dt_min=1e-2, dt_max=0.5, a_floor=0.5)
    W = 2 * 24 + 2 * 3 * 2 * 17 + 9 + 5
    proj = (rng.standard_normal((37, W)) * 3).astype(np.float32)
    dtb = rng.uniform(-2, 2, size=3).astype(np.float32)
    check_preprocess(gpu_preprocess(proj, dtb, **kw), oracle.preprocess(proj, dtb, **kw))


# --------------------------------------------------------------- SISO scans

def tiny_chain():
    """Tiny workload end to end: preprocess -> SISO scan on both sides."""
    w = gen.TINY_SISO
    p = gen.tiny_projection(w)
    kw = dict(inner_size=32, state_size=16, num_heads=2, num_rope_angles=8, num_groups=1,
              mimo_rank=1, **gen.TINY_PRE)
    shape = dict(x=(1, 64, 2, 16), z=(1, 64, 2, 16), bh=(1, 64, 1, 16), ch=(1, 64, 1, 16),
                 dt=(1, 64, 2), adt=(1, 64, 2), trap=(1, 64, 2), angle=(1, 64, 8))
    g = gpu_preprocess(p["projected"], p["dt_bias"], **kw)
    o = oracle.preprocess(p["projected"], p["dt_bias"], **kw)
    def scan_ins(pre):
        ins = {k: pre[k].astype(np.float32).reshape(shape[k]) for k in shape}
        ins["c"], ins["b"] = ins.pop("ch"), ins.pop("bh")
        ins.update(c_bias=p["c_bias"], b_bias=p["b_bias"], d=p["d"])
        return ins
    return w, scan_ins(g), scan_ins(o)


@pytest.mark.parametrize("mode", [FP32, TF32])
def test_tiny_chain(mode):
    """Tiny workload, preprocess chained into the scan on both sides; the GPU
    output is also held to the frozen oracle output in tests/golden."""
    import os
    w, gins, oins = tiny_chain()
    got = gpu_scan(w.cfg(), gins, mode)
    ref = oracle_scan(w.cfg(), oins)
    check_close(got, ref, TOL[mode])
    golden = np.loadtxt(os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                                     "tiny_siso_chain.txt")).reshape(got.shape)
    check_close(got, golden, TOL[mode], label="golden")


EDGE = [
    dict(B=2, L=100, H=4, G=2, P=64, N=128, A=32),
    dict(B=1, L=70, H=2, G=1, P=16, N=16, A=0),             # no rotation
    dict(B=1, L=65, H=2, G=2, P=32, N=64, A=32),            # 2A == N
    dict(B=1, L=40, H=1, G=1, P=1, N=1, A=0),               # P = N = 1
    dict(B=2, L=33, H=3, G=3, P=17, N=17, A=8),             # odd sizes, G = H
    dict(B=1, L=130, H=2, G=0, P=128, N=128, A=64),         # maxima, num_groups 0
    dict(B=3, L=1, H=2, G=1, P=8, N=8, A=2),                # single token
    dict(B=1, L=63, H=2, G=1, P=64, N=128, A=16),
    dict(B=1, L=64, H=2, G=1, P=64, N=128, A=16),
    dict(B=1, L=129, H=4, G=2, P=64, N=128, A=16, has_z=0),
    dict(B=1, L=200, H=2, G=1, P=64, N=128, A=16, has_d=0),
    dict(B=1, L=300, H=2, G=1, P=48, N=96, A=20),
    # compile-time instances (P64 N128 A32 / A64): ragged lengths, gate and D skip off,
    # a single token
    dict(B=1, L=65, H=2, G=1, P=64, N=128, A=32, has_z=0),
    dict(B=1, L=127, H=2, G=1, P=64, N=128, A=32, has_d=0),
    dict(B=2, L=1, H=2, G=1, P=64, N=128, A=32),
    dict(B=1, L=90, H=2, G=1, P=64, N=128, A=64),
]


def edge_case(B, L, H, G, P, N, A, has_z=1, has_d=1, R=1, norm=0, seed=11):
    w = gen.Workload("edge", B, L, H, G, P, N, A, mimo_rank=R, has_z=has_z, has_d=has_d,
                     has_output_norm=norm, seed_index=seed)
    return w, gen.scan_inputs(w)


@pytest.mark.parametrize("mode", [FP32, TF32])
@pytest.mark.parametrize("shape", EDGE, ids=[str(i) for i in range(len(EDGE))])
def test_siso_edge_shapes(shape, mode):
    w, ins = edge_case(**shape)
    got = gpu_scan(w.cfg(), ins, mode)
    ref = oracle_scan(w.cfg(), ins)
    check_close(got, ref, TOL[mode])


@pytest.mark.parametrize("mode", [FP32, TF32])
@pytest.mark.parametrize("w", [gen.SISO_1B, gen.SISO_LONG], ids=["siso_1b", "siso_long"])
def test_siso_full_size(w, mode):
    """Full workload on the GPU; the oracle recomputes the first and last
    batch rows (the recurrence is independent per batch row)."""
    ins = gen.scan_inputs(w)
    got = gpu_scan(w.cfg(), ins, mode)
    assert np.all(np.isfinite(got))
    for bsl in (slice(0, 1), slice(w.batch_size - 1, w.batch_size)):
        ref = oracle_scan(w.cfg(), ins, batch=bsl)
        check_close(got[bsl], ref, TOL[mode])


@pytest.mark.parametrize("mode", [FP32, TF32])
@pytest.mark.parametrize("mimo", [False, True], ids=["siso", "mimo"])
def test_strong_decay_chunks(mimo, mode):
    """The log decay adt scaled up along the sequence (x1 at the start, x15 for
    SISO / x60 for MIMO at the end), so that the chunks' summed |adt| runs from
    about 3-12 to about 170: the chunked kernel's factored decay mask (SISO,
    sum <= 85) and its exact-exponential mask both run, and so do its lazy and
    its rescaling state updates (compile-time P64 N128 A32 and R4 P64 N64 A32)."""
    shape = (dict(B=1, L=640, H=2, G=1, P=64, N=64, A=32, R=4, norm=1) if mimo
             else dict(B=1, L=640, H=2, G=1, P=64, N=128, A=32))
    w, ins = edge_case(**shape, seed=12)
    top = 60.0 if mimo else 15.0
    ramp = 1.0 + (top - 1.0) * np.arange(w.sequence_length) / w.sequence_length
    ins["adt"] = (ins["adt"] * ramp[None, :, None]).astype(np.float32)
    got = gpu_scan(w.cfg(), ins, mode, mimo=mimo)
    ref = oracle_scan(w.cfg(), ins, mimo=mimo)
    check_close(got, ref, TOL[mode])


# --------------------------------------------------------------- MIMO scans

MIMO_EDGE = [
    dict(B=1, L=50, H=2, G=1, P=16, N=16, A=4, R=2, norm=1),
    dict(B=2, L=70, H=2, G=2, P=64, N=64, A=32, R=4, norm=1),
    dict(B=1, L=33, H=3, G=1, P=32, N=128, A=64, R=8, norm=0),
    dict(B=1, L=40, H=2, G=1, P=128, N=32, A=3, R=3, norm=1, has_z=0),
    dict(B=1, L=20, H=2, G=0, P=8, N=8, A=0, R=1, norm=1),
]


@pytest.mark.parametrize("mode", [FP32, TF32])
@pytest.mark.parametrize("shape", MIMO_EDGE, ids=[str(i) for i in range(len(MIMO_EDGE))])
def test_mimo_edge_shapes(shape, mode):
    w, ins = edge_case(**shape)
    cfg = w.cfg()
    got = gpu_scan(cfg, ins, mode, mimo=True)
    ref = oracle_scan(cfg, ins, mimo=True)
    check_close(got, ref, TOL[mode])


@pytest.mark.parametrize("mode", [FP32, TF32])
def test_mimo_full_size(mode):
    """MIMO R4 workload with the output norm, both modes at their own bars
    (TF32 runs the split-operand flavour here: the norm makes each token's own
    relative error the normwise error). The oracle recomputes the first and
    the last batch rows."""
    w = gen.MIMO_R4
    ins = gen.scan_inputs(w)
    got = gpu_scan(w.cfg(), ins, mode, mimo=True)
    assert np.all(np.isfinite(got))
    for bsl in (slice(0, 1), slice(w.batch_size - 1, w.batch_size)):
        ref = oracle_scan(w.cfg(), ins, mimo=True, batch=bsl)
        check_close(got[bsl], ref, TOL[mode], label=f"batch {bsl.start}")


def test_mimo_full_size_tf32_without_norm():
    """The same workload without the output norm (single-pass TF32 operands)."""
    w = gen.MIMO_R4.with_(has_output_norm=0)
    ins = gen.scan_inputs(gen.MIMO_R4)
    got = gpu_scan(w.cfg(), ins, TF32, mimo=True)
    ref = oracle_scan(w.cfg(), ins, mimo=True, batch=slice(0, 1))
    check_close(got[0:1], ref, TOL[TF32])


# --------------------------------------------------------------------- step

def run_gpu_steps(w, ins, steps, mimo=False):
    """Calls the step entry point once per token; returns outputs [B, steps, H, P]
    and the final states (numpy)."""
    import torch
    cfg = w.cfg(sequence_length=1)
    c = m3.ssm_config(cfg)
    B, H, P, N, A, R = w.batch_size, w.num_heads, w.head_dim, w.state_size, w.num_rope_angles, w.mimo_rank
    st = dict(ssm=torch.zeros(B, H, P, N, device="cuda"), angle=torch.zeros(B, H, A, device="cuda"),
              k=torch.zeros(B, H, R, N, device="cuda"), v=torch.zeros(B, H, R, P, device="cuda"))
    if A == 0:
        st["angle"] = None
    seq = {k: dev(ins[k]) for k in SCAN_KEYS[:8]}
    par = {k: dev(ins[k]) for k in SCAN_KEYS[8:]}
    if mimo:
        par.update({k: dev(ins[k]) for k in MIMO_KEYS})
    outs = torch.empty(steps, B, 1, H, P, device="cuda")
    for t in range(steps):
        tok = [seq[k][:, t:t + 1].clone() for k in SCAN_KEYS[:8]]   # fresh, 16-byte aligned
        if A == 0:
            tok[7] = None
        if mimo:
            m3.m3_mimo_step(c, *tok, par["c_bias"], par["b_bias"], par["d"],
                            *[par[k] for k in MIMO_KEYS], st["ssm"], st["angle"], st["k"],
                            st["v"], outs[t])
        else:
            m3.m3_siso_step(c, *tok, par["c_bias"], par["b_bias"], par["d"], st["ssm"],
                            st["angle"], st["k"], st["v"], outs[t])
    torch.cuda.synchronize()
    out = outs[:, :, 0].permute(1, 0, 2, 3).cpu().numpy()
    return out, {k: (None if v is None else v.cpu().numpy()) for k, v in st.items()}


def test_decode_step_512_tokens():
    """Decode workload: 512 single-token calls at B=256; every call's output and
    the final states against the oracle's full 512-token scan of the same
    tokens. The first 3 and the last 3 batch rows are recomputed: the first and
    the last blocks of the grid (the last, partial wave)."""
    import numpy as np
    w = gen.DECODE_STEP
    ins = gen.decode_inputs(w)
    got, st = run_gpu_steps(w, ins, w.steps)
    bsl = np.r_[0:3, w.batch_size - 3:w.batch_size]
    cfg = w.cfg(sequence_length=w.steps, batch_size=len(bsl))
    ostate = oracle.zero_state(cfg)
    sub = {k: (v[bsl] if k in SCAN_KEYS[:8] else v) for k, v in ins.items()}
    ref = oracle.scan(cfg, *[sub[k] for k in SCAN_KEYS], state=ostate)
    check_close(got[bsl], ref, 1e-5)
    check_close(st["ssm"][bsl], ostate["ssm"], 1e-5)
    check_close(st["k"][bsl], ostate["k"], 1e-5)
    check_close(st["v"][bsl], ostate["v"], 1e-6)
    check_close(st["angle"][bsl], ostate["angle"], 1e-5)


@pytest.mark.parametrize("shape", [dict(B=2, L=24, H=4, G=2, P=17, N=17, A=8),
                                   dict(B=1, L=10, H=2, G=1, P=8, N=6, A=0)])
def test_siso_step_odd_shapes(shape):
    w, ins = edge_case(**shape)
    got, _ = run_gpu_steps(w, ins, w.sequence_length)
    ref = oracle_scan(w.cfg(), ins)
    check_close(got, ref, 1e-5)


@pytest.mark.parametrize("shape", [dict(B=2, L=16, H=2, G=1, P=64, N=64, A=32, R=4, norm=1),
                                   dict(B=1, L=12, H=3, G=3, P=16, N=12, A=5, R=3, norm=0)])
def test_mimo_step(shape):
    w, ins = edge_case(**shape)
    got, _ = run_gpu_steps(w, ins, w.sequence_length, mimo=True)
    ref = oracle_scan(w.cfg(), ins, mimo=True)
    check_close(got, ref, 1e-5)


def test_rejected_step_leaves_state_untouched():
    import torch
    w, ins = edge_case(B=1, L=1, H=2, G=1, P=8, N=8, A=2)
    cfg = m3.ssm_config(w.cfg(sequence_length=2))           # L != 1: rejected
    st = [torch.randn(s, device="cuda") for s in ((1, 2, 8, 8), (1, 2, 2), (1, 2, 1, 8), (1, 2, 1, 8))]
    before = [s.clone() for s in st]
    d = {k: dev(ins[k]) for k in SCAN_KEYS}
    out = torch.zeros(1, 1, 2, 8, device="cuda")
    with pytest.raises(m3.M3Error) as e:
        m3.m3_siso_step(cfg, *[d[k] for k in SCAN_KEYS], *st, out)
    assert e.value.status == m3.M3_ERR_INVALID_ARGUMENT
    torch.cuda.synchronize()
    for a, b in zip(st, before):
        assert torch.equal(a, b)
