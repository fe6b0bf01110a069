"""Pins for the oracle's preprocess adjoint (`m3o_preprocess_backward`, the
gradients of `Mamba3PreprocessBackward` / `mamba3_preprocess_backward` in
oarust mamba3.rs): against central differences of the oracle's own forward
preprocess (the definition of the derivative), against the directional
derivative of the B / C RMS normalisation along its own row (a closed form),
and against the structure of the map (identity slices, clamped elements).

Central differences: the loss is sum_k sum(out_k * g_k) over the eight
preprocess outputs. Inputs are rounded to multiples of 2^-20 (all below 8 in
magnitude, so float32 holds v +- eps exactly) and each is moved by
eps = 2^-16. Every (row, head) keeps softplus(dt_raw + dt_bias) and
softplus(a_raw) at least 0.02 away from the clamp bounds, so that no
difference straddles a kink; elements on either side of each bound are
present, so the clamps' zero gradients are pinned as well.
"""
import numpy as np
import pytest

import oracle

EPS = 2.0 ** -16
KW = dict(inner_size=3, state_size=5, num_heads=3, num_rope_angles=2, num_groups=1, mimo_rank=2,
          epsilon=2.0 ** -7, dt_min=0.05, dt_max=0.8, a_floor=0.3)
ROWS = 8
NAMES = oracle.PRE_GRAD_NAMES


def _softplus(v):
    return np.logaddexp(0.0, v)


def _setup(seed=7):
    rng = np.random.default_rng(seed)
    I, N, H, A = KW["inner_size"], KW["state_size"], KW["num_heads"], KW["num_rope_angles"]
    bc = KW["num_groups"] * KW["mimo_rank"] * N
    W = 2 * I + 2 * bc + 3 * H + A
    o_s = 2 * I + 2 * bc
    proj = rng.normal(0.0, 2.0, size=(ROWS, W))
    dtb = rng.uniform(-2.0, 2.0, size=H)
    q = 2.0 ** 20
    proj = np.round(np.clip(proj, -7.5, 7.5) * q) / q
    dtb = np.round(dtb * q) / q
    # one element on each side of every bound, whatever the draw
    proj[0, o_s + 0] = -6.0 - dtb[0]   # softplus ~ 2.5e-3 < dt_min
    proj[1, o_s + 1] = 3.0 - dtb[1]    # softplus ~ 3.05 > dt_max
    proj[2, o_s + 2] = -1.0 - dtb[2]   # softplus ~ 0.31, inside
    proj[0, o_s + H] = -3.0            # softplus ~ 0.049 < a_floor
    proj[1, o_s + H] = 1.0             # softplus ~ 1.31 > a_floor
    lo, hi, fl = KW["dt_min"], KW["dt_max"], KW["a_floor"]
    # keep every softplus at least 0.02 away from the bounds it meets
    for _ in range(64):
        sp = _softplus(proj[:, o_s:o_s + H] + dtb)
        near = (np.abs(sp - lo) < 0.02) | (np.abs(sp - hi) < 0.02)
        sa = _softplus(proj[:, o_s + H:o_s + 2 * H])
        near_a = np.abs(sa - fl) < 0.02
        if not near.any() and not near_a.any():
            break
        proj[:, o_s:o_s + H][near] += 0.125
        proj[:, o_s + H:o_s + 2 * H][near_a] += 0.125
    sp = _softplus(proj[:, o_s:o_s + H] + dtb)
    sa = _softplus(proj[:, o_s + H:o_s + 2 * H])
    assert (sp < lo).any() and (sp > hi).any() and ((sp > lo) & (sp < hi)).any()
    assert (sa < fl).any() and (sa > fl).any()
    assert np.all(np.abs(proj) < 8)
    proj = proj.astype(np.float32)
    dtb = dtb.astype(np.float32)
    shapes = dict(x=(ROWS, I), z=(ROWS, I), bh=(ROWS, bc), ch=(ROWS, bc), dt=(ROWS, H),
                  adt=(ROWS, H), trap=(ROWS, H), angle=(ROWS, A))
    grads = {k: rng.standard_normal(size=shapes[k]).astype(np.float32) for k in NAMES}
    return proj, dtb, grads


def _loss(proj, dtb, grads):
    out = oracle.preprocess(proj, dtb, threads=1, **KW)
    return float(sum(np.sum(out[k] * grads[k].astype(np.float64)) for k in NAMES))


def test_preprocess_adjoint_equals_central_differences():
    proj, dtb, grads = _setup()
    ref = oracle.preprocess_backward(proj, dtb, grads, threads=1, **KW)
    for name, base in (("projected", proj), ("dt_bias", dtb)):
        fd = np.zeros(base.shape)
        for i in np.ndindex(base.shape):
            v = base[i]
            up, dn = np.float32(v + np.float32(EPS)), np.float32(v - np.float32(EPS))
            assert float(up) - float(v) == EPS and float(v) - float(dn) == EPS
            moved = base.copy()
            moved[i] = up
            lp = _loss(moved, dtb, grads) if name == "projected" else _loss(proj, moved, grads)
            moved[i] = dn
            lm = _loss(moved, dtb, grads) if name == "projected" else _loss(proj, moved, grads)
            fd[i] = (lp - lm) / (2 * EPS)
        g = ref[name]
        assert g.shape == fd.shape
        scale = max(np.max(np.abs(fd)), 1e-3)
        err = np.max(np.abs(g - fd)) / scale
        assert err < 2e-7, (name, err)


def test_clamped_elements_have_zero_gradient_and_slices_are_identity():
    proj, dtb, grads = _setup(seed=11)
    I, N, H, A = KW["inner_size"], KW["state_size"], KW["num_heads"], KW["num_rope_angles"]
    bc = KW["num_groups"] * KW["mimo_rank"] * N
    o_s = 2 * I + 2 * bc
    g = oracle.preprocess_backward(proj, dtb, grads, threads=1, **KW)["projected"]
    assert np.array_equal(g[:, :I], grads["z"].astype(np.float64))
    assert np.array_equal(g[:, I:2 * I], grads["x"].astype(np.float64))
    assert np.array_equal(g[:, o_s + 2 * H:o_s + 3 * H], grads["trap"].astype(np.float64))
    assert np.array_equal(g[:, o_s + 3 * H:], grads["angle"].astype(np.float64))
    sp = _softplus(proj[:, o_s:o_s + H].astype(np.float64) + dtb)
    clamped = (sp < KW["dt_min"]) | (sp > KW["dt_max"])
    assert clamped.any() and np.all(g[:, o_s:o_s + H][clamped] == 0)
    assert np.all(g[:, o_s:o_s + H][~clamped] != 0)
    floored = _softplus(proj[:, o_s + H:o_s + 2 * H].astype(np.float64)) < KW["a_floor"]
    assert floored.any() and np.all(g[:, o_s + H:o_s + 2 * H][floored] == 0)


@pytest.mark.parametrize("eps", [2.0 ** -7, 1.0, 2.0 ** -20])
def test_rms_adjoint_along_its_own_row(eps):
    """Scaling a B / C row u by c moves the normalised row along
    d/dc [c u / sqrt(c^2 ms + eps)] at c = 1, = u s eps / (ms + eps) with
    s = 1 / sqrt(ms + eps), ms = mean(u^2). So the adjoint's component along
    u must be sum_n du_n u_n = s eps / (ms + eps) * sum_n g_n u_n: a dropped
    s^3 term, a wrong 1/N or a missing eps breaks it (and for small eps the
    adjoint is orthogonal to u, the norm's scale invariance)."""
    kw = dict(KW, epsilon=eps)
    proj, dtb, grads = _setup(seed=3)
    I, N = kw["inner_size"], kw["state_size"]
    rows_bc = kw["num_groups"] * kw["mimo_rank"]
    g = oracle.preprocess_backward(proj, dtb, grads, threads=1, **kw)["projected"]
    e = float(np.float32(eps))
    for which, gk in ((0, "bh"), (1, "ch")):
        off = 2 * I + which * rows_bc * N
        for r in range(ROWS):
            for j in range(rows_bc):
                u = proj[r, off + j * N:off + (j + 1) * N].astype(np.float64)
                gu = grads[gk][r, j * N:(j + 1) * N].astype(np.float64)
                du = g[r, off + j * N:off + (j + 1) * N]
                ms = np.mean(u * u)
                s = 1.0 / np.sqrt(ms + e)
                want = s * e / (ms + e) * np.dot(gu, u)
                got = np.dot(du, u)
                assert abs(got - want) <= 1e-12 * (s * np.linalg.norm(gu) * np.linalg.norm(u) + 1e-300)


def test_preprocess_adjoint_is_linear_in_the_output_gradients():
    """Exact split of every output gradient into its even and odd rows:
    adjoint(g) = adjoint(g_even) + adjoint(g_odd)."""
    proj, dtb, grads = _setup(seed=5)
    even = {k: v.copy() for k, v in grads.items()}
    for v in even.values():
        v[1::2] = 0
    odd = {k: (grads[k] - even[k]).astype(np.float32) for k in NAMES}
    a = oracle.preprocess_backward(proj, dtb, grads, threads=1, **KW)
    b = oracle.preprocess_backward(proj, dtb, even, threads=1, **KW)
    c = oracle.preprocess_backward(proj, dtb, odd, threads=1, **KW)
    for k in ("projected", "dt_bias"):
        ref = b[k] + c[k]
        assert np.max(np.abs(a[k] - ref)) <= 1e-12 * max(1.0, np.max(np.abs(ref))), k
