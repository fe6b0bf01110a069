"""GPU parity of m3_preprocess_backward (oarust mamba3.rs
`mamba3_preprocess_backward`, the gradients of `Mamba3PreprocessBackward`)
against the oracle's FP64 adjoint, called through the C ABI on the same seeded
inputs.

Bars, derived from the float32 arithmetic of the kernel:
  - z, x, trap and angle columns: bit-exact (copies of the output gradients);
  - B / C columns: per N-row u with output gradient g, max |error| <= 4e-6 x
    (s max|g| + s^3 max|u| sum|g u| / N), the sizes of the two terms whose
    difference the row is (they cancel in some short rows). The inverse RMS
    and sum g u are float32 sums, four terms a lane and a five-step butterfly
    (at N <= 128), so about ten roundings of that size;
  - dt_raw and a_raw columns: exact zeros where the oracle's clamp or floor
    stops the gradient, elsewhere normwise over the column block <= 4e-6;
  - dt_bias: |error| <= 1e-5 x sum over rows |d dt_raw|. The fixed-order float32
    sum takes each term through at most chunk / 8 + 8 + per + 32 roundings
    (chunk rows per partial, per partials per warp of the final sum): 60 at
    16,384 rows (128-row chunks), a worst case of 3.6e-6; 90 in the
    140,000-row case (256-row chunks).
The clamp and floor decisions are taken by the kernel in float32 and by the
oracle in float64. Where softplus lies within a relative 1e-5 of a bound the
two may decide differently, so the test gives those (row, head) elements a
zero output gradient for dt and adt. Both readings then agree, and the
decisions elsewhere are compared exactly.
"""
import numpy as np
import pytest

import oracle
import selective_state_space_mamba3_gb300 as m3
from selective_state_space_mamba3_gb300 import inputs as gen

from m3_testutil import dev

pytestmark = pytest.mark.gpu
NAMES = gen.PRE_OUTPUTS


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    from selective_state_space_mamba3_gb300 import build
    build.build()
    oracle.build()
    assert torch.cuda.is_available()


def _shapes(rows, kw):
    I, N, H, A = kw["inner_size"], kw["state_size"], kw["num_heads"], kw["num_rope_angles"]
    bc = kw["num_groups"] * kw["mimo_rank"] * N
    return dict(x=(rows, I), z=(rows, I), bh=(rows, bc), ch=(rows, bc), dt=(rows, H),
                adt=(rows, H), trap=(rows, H), angle=(rows, A))


def _mask_ties(proj, dtb, grads, kw):
    """Zero the dt / adt output gradients where a clamp or floor decision is
    within float32 resolution of its bound; returns the count zeroed."""
    I, N, H = kw["inner_size"], kw["state_size"], kw["num_heads"]
    o_s = 2 * I + 2 * kw["num_groups"] * kw["mimo_rank"] * N
    sp = np.logaddexp(0.0, proj[:, o_s:o_s + H].astype(np.float64) + dtb.astype(np.float64))
    sa = np.logaddexp(0.0, proj[:, o_s + H:o_s + 2 * H].astype(np.float64))
    lo, hi, fl = (float(np.float32(kw[k])) for k in ("dt_min", "dt_max", "a_floor"))
    near = (np.abs(sp - lo) <= 1e-5 * lo) | (np.abs(sp - hi) <= 1e-5 * hi)
    near_a = np.abs(sa - fl) <= 1e-5 * fl
    grads["dt"][near] = 0
    grads["adt"][near | near_a] = 0
    return int(near.sum() + near_a.sum())


def gpu_preprocess_backward(proj, dtb, grads, kw):
    import torch
    rows, W = proj.shape
    cfg = m3.preprocess_config(**kw)
    gp = torch.full((rows, W), float("nan"), device="cuda")
    gb = torch.full((kw["num_heads"],), float("nan"), device="cuda")
    ws = torch.empty(max(m3.m3_preprocess_backward_workspace(cfg, rows), 16), dtype=torch.uint8,
                     device="cuda")
    m3.m3_preprocess_backward(cfg, rows, dev(proj), dev(dtb), *[dev(grads[k]) for k in NAMES],
                              gp, gb, ws)
    torch.cuda.synchronize()
    return gp.cpu().numpy(), gb.cpu().numpy()


def check(proj, dtb, grads, kw):
    rows = proj.shape[0]
    I, N, H = kw["inner_size"], kw["state_size"], kw["num_heads"]
    bc = kw["num_groups"] * kw["mimo_rank"] * N
    o_s = 2 * I + 2 * bc
    got, got_b = gpu_preprocess_backward(proj, dtb, grads, kw)
    ref = oracle.preprocess_backward(proj, dtb, grads, **kw)
    want, want_b = ref["projected"], ref["dt_bias"]
    assert np.all(np.isfinite(got)) and np.all(np.isfinite(got_b))
    for lo_c, hi_c in ((0, 2 * I), (o_s + 2 * H, want.shape[1])):
        assert np.array_equal(got[:, lo_c:hi_c].astype(np.float64), want[:, lo_c:hi_c])
    nrow = 2 * bc // N
    g_bc = got[:, 2 * I:o_s].reshape(rows, nrow, N).astype(np.float64)
    w_bc = want[:, 2 * I:o_s].reshape(rows, nrow, N)
    u = proj[:, 2 * I:o_s].reshape(rows, nrow, N).astype(np.float64)
    gin = np.concatenate([grads["bh"], grads["ch"]], axis=1).reshape(rows, nrow, N).astype(np.float64)
    s = 1.0 / np.sqrt(np.mean(u * u, axis=-1) + float(np.float32(kw["epsilon"])))
    scale = (s * np.max(np.abs(gin), axis=-1) +
             s ** 3 * np.max(np.abs(u), axis=-1) * np.sum(np.abs(gin * u), axis=-1) / N)
    err = np.max(np.abs(g_bc - w_bc), axis=-1) / np.maximum(scale, 1e-30)
    assert np.max(err) <= 4e-6, np.max(err)
    for c0 in (o_s, o_s + H):
        g, w = got[:, c0:c0 + H].astype(np.float64), want[:, c0:c0 + H]
        assert np.array_equal(g == 0, w == 0), c0
        e = np.max(np.abs(g - w)) / max(np.max(np.abs(w)), 1e-30)
        assert e <= 4e-6, (c0, e)
    bound = 1e-5 * np.sum(np.abs(want[:, o_s:o_s + H]), axis=0) + 1e-30
    assert np.all(np.abs(got_b - want_b) <= bound), np.max(np.abs(got_b - want_b) / bound)
    return got, got_b


def _random_case(rows, kw, seed, raw_sigma=3.0):
    rng = np.random.default_rng(seed)
    I, N, H, A = kw["inner_size"], kw["state_size"], kw["num_heads"], kw["num_rope_angles"]
    W = 2 * I + 2 * kw["num_groups"] * kw["mimo_rank"] * N + 3 * H + A
    proj = (rng.standard_normal((rows, W)) * raw_sigma).astype(np.float32)
    dtb = rng.uniform(-2, 2, size=H).astype(np.float32)
    grads = gen.preprocess_output_gradient(gen.TINY_SISO, _shapes(rows, kw), salt=seed)
    return proj, dtb, grads


def test_tiny_unaligned_width():
    """The tiny workload's projection (W = 110, not a multiple of 4: the scalar
    path of the kernel)."""
    w = gen.TINY_SISO
    p = gen.tiny_projection(w)
    kw = dict(inner_size=32, state_size=16, num_heads=2, num_rope_angles=8, num_groups=1,
              mimo_rank=1, **gen.TINY_PRE)
    rows = p["projected"].shape[0]
    grads = gen.preprocess_output_gradient(w, _shapes(rows, kw))
    _mask_ties(p["projected"], p["dt_bias"], grads, kw)
    check(p["projected"], p["dt_bias"], grads, kw)


def test_odd_state_both_clamps_and_floor():
    """N = 17 (scalar B / C rows), R = 2, G = 3; dt bounds [1e-2, 0.5] and a
    floor of 0.5 with raw columns ~ N(0, 9): many elements clamped on both sides
    and floored, so the zero pattern is exercised."""
    kw = dict(inner_size=24, state_size=17, num_heads=3, num_rope_angles=5, num_groups=3,
              mimo_rank=2, epsilon=1e-5, dt_min=1e-2, dt_max=0.5, a_floor=0.5)
    proj, dtb, grads = _random_case(37, kw, seed=5)
    _mask_ties(proj, dtb, grads, kw)
    got, _ = check(proj, dtb, grads, kw)
    o_s = 2 * 24 + 2 * 3 * 2 * 17
    assert np.sum(got[:, o_s:o_s + 3] == 0) > 5 and np.sum(got[:, o_s + 3:o_s + 6] == 0) > 5


def test_many_heads_ragged_rows():
    """H = 40 (two 32-head blocks of the dt_bias sums), 300 rows (chunks of 128
    with a ragged last one), W a multiple of 4 (the vector path)."""
    kw = dict(inner_size=160, state_size=16, num_heads=40, num_rope_angles=4, num_groups=2,
              mimo_rank=1, epsilon=1e-6, dt_min=1e-3, dt_max=0.1, a_floor=1e-4)
    proj, dtb, grads = _random_case(300, kw, seed=9)
    assert proj.shape[1] % 4 == 0
    _mask_ties(proj, dtb, grads, kw)
    check(proj, dtb, grads, kw)


def test_many_rows():
    """140,000 rows: more than 1024 chunks of 128, so the dt_bias partials take
    chunks of 256 rows."""
    kw = dict(inner_size=4, state_size=4, num_heads=2, num_rope_angles=0, num_groups=1,
              mimo_rank=1, epsilon=1e-6, dt_min=1e-3, dt_max=0.1, a_floor=1e-4)
    proj, dtb, grads = _random_case(140000, kw, seed=13, raw_sigma=2.0)
    _mask_ties(proj, dtb, grads, kw)
    check(proj, dtb, grads, kw)


def test_many_heads():
    """H = 1100: the scalar columns take five passes of the block's threads,
    the dt_bias sums 35 blocks of 32 heads (the last one partial)."""
    kw = dict(inner_size=4, state_size=4, num_heads=1100, num_rope_angles=2, num_groups=1,
              mimo_rank=1, epsilon=1e-6, dt_min=1e-2, dt_max=0.5, a_floor=0.5)
    proj, dtb, grads = _random_case(150, kw, seed=17)
    _mask_ties(proj, dtb, grads, kw)
    check(proj, dtb, grads, kw)


@pytest.mark.parametrize("w", [gen.SISO_1B, gen.MIMO_R4, gen.SISO_LONG],
                         ids=["siso_layer", "mimo_layer", "long_context_layer"])
def test_layer_shape(w):
    """The layer's packed projection (the distributions of the preprocess parity
    tests) at full size, every element compared, and a second call bit-identical."""
    p = gen.layer_projection(w)
    kw = dict(inner_size=w.num_heads * w.head_dim, state_size=w.state_size,
              num_heads=w.num_heads, num_rope_angles=w.num_rope_angles,
              num_groups=w.num_groups, mimo_rank=w.mimo_rank, **gen.PRE_DEFAULT)
    rows = p["projected"].shape[0]
    grads = gen.preprocess_output_gradient(w, _shapes(rows, kw))
    masked = _mask_ties(p["projected"], p["dt_bias"], grads, kw)
    assert masked < 1e-3 * rows * w.num_heads
    got, got_b = check(p["projected"], p["dt_bias"], grads, kw)
    again, again_b = gpu_preprocess_backward(p["projected"], p["dt_bias"], grads, kw)
    assert np.array_equal(got, again) and np.array_equal(got_b, again_b)


@pytest.mark.parametrize("rows, heads, angles", [(1, 3, 2), (7, 1, 4), (129, 2, 0)],
                         ids=["one_row", "one_head", "no_angles_null_pointer"])
def test_degenerate_sizes(rows, heads, angles):
    """One row (one block, one dt_bias partial), one head, and A = 0 with the
    angle gradient passed as a NULL pointer (129 rows: two partial chunks)."""
    import torch
    kw = dict(inner_size=8, state_size=8, num_heads=heads, num_rope_angles=angles, num_groups=1,
              mimo_rank=2, epsilon=1e-5, dt_min=1e-2, dt_max=0.5, a_floor=0.5)
    proj, dtb, grads = _random_case(rows, kw, seed=23)
    _mask_ties(proj, dtb, grads, kw)
    if angles:
        check(proj, dtb, grads, kw)
        return
    cfg = m3.preprocess_config(**kw)
    gp = torch.full(proj.shape, float("nan"), device="cuda")
    gb = torch.full((heads,), float("nan"), device="cuda")
    ws = torch.empty(max(m3.m3_preprocess_backward_workspace(cfg, rows), 16), dtype=torch.uint8,
                     device="cuda")
    g = [None if k == "angle" else dev(grads[k]) for k in NAMES]
    m3.m3_preprocess_backward(cfg, rows, dev(proj), dev(dtb), *g, gp, gb, ws)
    torch.cuda.synchronize()
    ref = oracle.preprocess_backward(proj, dtb, grads, **kw)
    assert np.all(np.isfinite(gp.cpu().numpy()))
    err = np.max(np.abs(gp.cpu().numpy() - ref["projected"])) / np.max(np.abs(ref["projected"]))
    assert err <= 4e-6, err
    bound = 1e-5 * np.sum(np.abs(ref["projected"][:, -3 * heads:-2 * heads]), axis=0) + 1e-30
    assert np.all(np.abs(gb.cpu().numpy() - ref["dt_bias"]) <= bound)
