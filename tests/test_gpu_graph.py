"""The entry points inside CUDA graphs: each call is captured on the current
stream with torch.cuda.graph, replayed, and its results compared bit for bit
with the same call run eagerly. This covers the launches that depend on one
another programmatically (the packed step's row pass and scan, the
preprocess adjoint's three kernels), a decode loop of single-token steps
replayed from reset states, and the SISO backward's ordered reductions.
"""
import numpy as np
import pytest

import selective_state_space_mamba3_gb300 as m3
from selective_state_space_mamba3_gb300 import inputs as gen

from m3_testutil import dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    from selective_state_space_mamba3_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def captured(fn):
    """fn captured into a CUDA graph (after one run on a side stream)."""
    import torch
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="relaxed"):
        fn()
    return g


def replay(g, *buffers):
    """Poisons the result buffers, replays g, returns them (numpy)."""
    import torch
    for b in buffers:
        b.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    return [b.cpu().numpy() for b in buffers]


def test_packed_step_in_a_graph():
    """m3_siso_forward_packed (TF32: the row pass, then the packed scan as its
    programmatic dependent) at the 1B-layer head shape, 1,024 tokens."""
    import torch
    w = gen.SISO_1B.with_(name="graph packed step", batch_size=1, sequence_length=1024)
    B, L, H, P, N, A = (w.batch_size, w.sequence_length, w.num_heads, w.head_dim, w.state_size,
                        w.num_rope_angles)
    p = gen.layer_projection(w)
    sp = gen.scan_params(w)
    cfg = m3.ssm_config(w.cfg(), m3.M3_MATH_TF32)
    pcfg = m3.preprocess_config(inner_size=H * P, state_size=N, num_heads=H, num_rope_angles=A,
                                num_groups=w.num_groups, mimo_rank=1, **gen.PRE_DEFAULT)
    proj, dtb = dev(p["projected"]), dev(p["dt_bias"])
    cb, bb, d = dev(sp["c_bias"]), dev(sp["b_bias"]), dev(sp["d"])
    out = torch.empty(B, L, H, P, device="cuda")
    ws = torch.empty(max(m3.m3_siso_forward_packed_workspace(cfg, pcfg), 16), dtype=torch.uint8,
                     device="cuda")
    fn = lambda: m3.m3_siso_forward_packed(cfg, pcfg, proj, dtb, cb, bb, d, out, ws)
    fn()
    torch.cuda.synchronize()
    eager = out.cpu().numpy()
    assert np.all(np.isfinite(eager))
    (got,) = replay(captured(fn), out)
    assert np.array_equal(got, eager)
    assert m3.m3_workspace_status(ws) == m3.M3_OK


def test_preprocess_backward_in_a_graph():
    """m3_preprocess_backward: the row kernel and its two programmatic
    dependents (the dt_bias partials and their sum)."""
    import torch
    rng = np.random.default_rng(21)
    kw = dict(inner_size=160, state_size=16, num_heads=40, num_rope_angles=4, num_groups=2,
              mimo_rank=1, epsilon=1e-6, dt_min=1e-3, dt_max=0.1, a_floor=1e-4)
    rows, I, H, A, bc = 300, 160, 40, 4, 2 * 16
    W = 2 * I + 2 * bc + 3 * H + A
    proj = dev(rng.standard_normal((rows, W)).astype(np.float32) * 2)
    dtb = dev(rng.uniform(-2, 2, size=H).astype(np.float32))
    shapes = dict(x=(rows, I), z=(rows, I), bh=(rows, bc), ch=(rows, bc), dt=(rows, H),
                  adt=(rows, H), trap=(rows, H), angle=(rows, A))
    grads = {k: dev(v) for k, v in gen.preprocess_output_gradient(gen.TINY_SISO, shapes).items()}
    cfg = m3.preprocess_config(**kw)
    gp = torch.empty(rows, W, device="cuda")
    gb = torch.empty(H, device="cuda")
    ws = torch.empty(max(m3.m3_preprocess_backward_workspace(cfg, rows), 16), dtype=torch.uint8,
                     device="cuda")
    fn = lambda: m3.m3_preprocess_backward(cfg, rows, proj, dtb,
                                           *[grads[k] for k in gen.PRE_OUTPUTS], gp, gb, ws)
    fn()
    torch.cuda.synchronize()
    eager = (gp.cpu().numpy(), gb.cpu().numpy())
    got = replay(captured(fn), gp, gb)
    assert np.array_equal(got[0], eager[0]) and np.array_equal(got[1], eager[1])


def test_decode_loop_in_a_graph():
    """Eight m3_siso_step calls captured as one graph and replayed from zeroed
    states: the same outputs and states as the eager loop."""
    import torch
    w = gen.DECODE_STEP.with_(name="graph decode", batch_size=4, num_heads=4)
    steps = 8
    ins = gen.decode_inputs(w, steps=steps)
    B, H, P, N, A = w.batch_size, w.num_heads, w.head_dim, w.state_size, w.num_rope_angles
    keys = ("c", "b", "x", "z", "adt", "dt", "trap", "angle")
    toks = [[dev(ins[k][:, t:t + 1]) for k in keys] for t in range(steps)]
    par = [dev(ins[k]) for k in ("c_bias", "b_bias", "d")]
    st = [torch.zeros(s, device="cuda") for s in ((B, H, P, N), (B, H, A), (B, H, N), (B, H, P))]
    outs = torch.empty(steps, B, 1, H, P, device="cuda")
    cfg = m3.ssm_config(w.cfg(sequence_length=1))

    def loop():
        for t in range(steps):
            m3.m3_siso_step(cfg, *toks[t], *par, *st, outs[t])

    loop()
    torch.cuda.synchronize()
    eager = [outs.cpu().numpy()] + [s.cpu().numpy() for s in st]
    for s in st:
        s.zero_()
    g = captured(loop)   # its side-stream run advanced the states: reset them
    for s in st:
        s.zero_()
    outs.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    got = [outs.cpu().numpy()] + [s.cpu().numpy() for s in st]
    for a, b in zip(got, eager):
        assert np.array_equal(a, b)


def test_siso_backward_in_a_graph():
    """m3_siso_backward (the two sweeps and the ordered finish) on a grouped
    shape with rotary angles."""
    import torch
    w = gen.Workload("graph backward", 2, 96, 4, 2, 32, 64, 16, seed_index=71)
    ins = gen.scan_inputs(w)
    dout = dev(gen.output_gradient(w))
    keys = ("c", "b", "x", "z", "adt", "dt", "trap", "angle", "c_bias", "b_bias", "d")
    d = {k: dev(ins[k]) for k in keys}
    g = {k: torch.empty_like(d[k]) for k in keys}
    cfg = m3.ssm_config(w.cfg())
    ws = torch.empty(m3.m3_siso_backward_workspace(cfg), dtype=torch.uint8, device="cuda")
    fn = lambda: m3.m3_siso_backward(cfg, dout, *[d[k] for k in keys], *[g[k] for k in keys], ws)
    fn()
    torch.cuda.synchronize()
    eager = [g[k].cpu().numpy() for k in keys]
    got = replay(captured(fn), *[g[k] for k in keys])
    for k, a, b in zip(keys, got, eager):
        assert np.array_equal(a, b), k
