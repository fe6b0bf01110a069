"""Pins for the oracle's adjoints (`m3o_siso_backward`, the eleven gradients of
`SsmBackward` / `mamba3_siso_backward`, and `m3o_mimo_backward`, the fifteen of
`Mamba3MimoBackward` / `mamba3_mimo_backward` in oarust mamba3.rs): every
gradient element is checked against the central difference of the oracle's
own forward scan, the definition of the derivative, on tiny inputs.

The loss is sum(out * dout). The inputs are rounded to multiples of 2^-20
(all below 8 in magnitude, so float32 holds them and v +- eps exactly) and
each is moved by +-eps with eps = 2^-16, so that the two forward calls see
exactly v +- eps. The central difference is then exact up to eps^2 / 6 times
the third derivative (below 1e-9 here, also where the output norm curves
sharply at the first tokens, whose small dt makes o small) plus the forward
oracle's double rounding (about 1e-11 after the division by 2 eps); a
dropped term, a wrong sign or a transposed rotation in the adjoint moves its
gradient by far more.
"""
import numpy as np
import pytest

import oracle
from selective_state_space_mamba3_gb300 import inputs as gen

KEYS = ("c", "b", "x", "z", "adt", "dt", "trap", "angle", "c_bias", "b_bias", "d")
MIMO_KEYS = KEYS + ("mimo_x", "mimo_z", "mimo_o", "norm_weight")
EPS = 2.0 ** -16

SHAPES = {
    # heads sharing a group (the c / b gradients sum over the group's heads),
    # rotary pairs plus plain dims
    "groups": dict(B=2, L=5, H=2, G=1, P=3, N=6, A=2),
    # one group per head (num_groups 0), every dim rotated (2A == N)
    "g0_full_rotation": dict(B=1, L=6, H=2, G=0, P=2, N=4, A=2),
    # no gate, no skip, no rotation, odd sizes
    "plain": dict(B=1, L=4, H=3, G=3, P=3, N=5, A=0, has_z=0, has_d=0),
    # a single token (no previous-token term)
    "one_token": dict(B=2, L=1, H=2, G=2, P=2, N=4, A=1),
}


def _setup(B, L, H, G, P, N, A, has_z=1, has_d=1):
    w = gen.Workload("backward pin", B, L, H, G, P, N, A, has_z=has_z, has_d=has_d,
                     seed_index=61)
    ins = gen.scan_inputs(w)
    rng = np.random.default_rng(17)
    ins["d"] = rng.uniform(0.5, 1.5, size=(H,)).astype(np.float32)  # a non-trivial skip
    q = 2.0 ** 20
    for k in KEYS:
        assert np.all(np.abs(ins[k]) < 8)
        ins[k] = (np.round(ins[k].astype(np.float64) * q) / q).astype(np.float32)
    return w.cfg(), ins, gen.output_gradient(w)


def _loss(cfg, ins, dout):
    return float(np.sum(oracle.scan(cfg, *[ins[k] for k in KEYS]) * dout))


@pytest.mark.parametrize("name", list(SHAPES))
def test_siso_adjoints_equal_central_differences(name):
    cfg, ins, dout = _setup(**SHAPES[name])
    grads = oracle.siso_backward(cfg, dout, *[ins[k] for k in KEYS])
    for key in KEYS:
        base = ins[key]
        fd = np.zeros(base.shape)
        for i in np.ndindex(base.shape):
            v = base[i]
            up, dn = np.float32(v + np.float32(EPS)), np.float32(v - np.float32(EPS))
            assert float(up) - float(v) == EPS and float(v) - float(dn) == EPS
            moved = dict(ins)
            moved[key] = base.copy()
            moved[key][i] = up
            lp = _loss(cfg, moved, dout)
            moved[key][i] = dn
            lm = _loss(cfg, moved, dout)
            fd[i] = (lp - lm) / (2 * EPS)
        g = grads[key]
        assert g.shape == fd.shape, key
        if g.size == 0:
            continue
        if key == "z" and not cfg["has_z"] or key == "d" and not cfg["has_d"]:
            assert np.all(g == 0) and np.all(fd == 0), key
            continue
        scale = max(np.max(np.abs(fd)), 1e-3)
        err = np.max(np.abs(g - fd)) / scale
        assert err < 2e-6, (name, key, err)


def test_backward_is_linear_in_the_output_gradient():
    """The adjoints are linear in dout: with dout split exactly into two parts
    (the even and the odd tokens), grads(dout) = grads(part 1) + grads(part 2)."""
    cfg, ins, d = _setup(**SHAPES["groups"])
    d1 = d.copy()
    d1[:, 1::2] = 0
    d2 = (d - d1).astype(np.float32)
    g = oracle.siso_backward(cfg, d, *[ins[k] for k in KEYS])
    g1 = oracle.siso_backward(cfg, d1, *[ins[k] for k in KEYS])
    g2 = oracle.siso_backward(cfg, d2, *[ins[k] for k in KEYS])
    for key in KEYS:
        ref = g1[key] + g2[key]
        assert np.max(np.abs(g[key] - ref)) <= 1e-12 * max(1.0, np.max(np.abs(ref))), key


MIMO_SHAPES = {
    # rank 2 with the output norm, two heads sharing a group
    "mimo_norm": dict(B=1, L=4, H=2, G=1, P=3, N=4, A=1, R=2, norm=1),
    # rank 3 without the norm, a group per head, two batch rows
    "mimo_r3": dict(B=2, L=3, H=2, G=2, P=2, N=6, A=2, R=3, norm=0),
    # no gate, no skip, with the norm
    "mimo_plain_norm": dict(B=1, L=3, H=1, G=1, P=4, N=4, A=2, R=2, norm=1, has_z=0, has_d=0),
}


def _mimo_setup(B, L, H, G, P, N, A, R, norm, has_z=1, has_d=1):
    w = gen.Workload("mimo backward pin", B, L, H, G, P, N, A, mimo_rank=R, has_z=has_z,
                     has_d=has_d, has_output_norm=norm, seed_index=62)
    ins = gen.scan_inputs(w)
    rng = np.random.default_rng(19)
    ins["d"] = rng.uniform(0.5, 1.5, size=(H,)).astype(np.float32)
    q = 2.0 ** 20
    for k in MIMO_KEYS:
        assert np.all(np.abs(ins[k]) < 8)
        ins[k] = (np.round(ins[k].astype(np.float64) * q) / q).astype(np.float32)
    return w.cfg(), ins, gen.output_gradient(w)


def _mimo_loss(cfg, ins, dout):
    out = oracle.scan(cfg, *[ins[k] for k in KEYS], **{k: ins[k] for k in MIMO_KEYS[11:]})
    return float(np.sum(out * dout))


@pytest.mark.parametrize("name", list(MIMO_SHAPES))
def test_mimo_adjoints_equal_central_differences(name):
    cfg, ins, dout = _mimo_setup(**MIMO_SHAPES[name])
    grads = oracle.mimo_backward(cfg, dout, *[ins[k] for k in MIMO_KEYS])
    for key in MIMO_KEYS:
        base = ins[key]
        fd = np.zeros(base.shape)
        for i in np.ndindex(base.shape):
            v = base[i]
            up, dn = np.float32(v + np.float32(EPS)), np.float32(v - np.float32(EPS))
            assert float(up) - float(v) == EPS and float(v) - float(dn) == EPS
            moved = dict(ins)
            moved[key] = base.copy()
            moved[key][i] = up
            lp = _mimo_loss(cfg, moved, dout)
            moved[key][i] = dn
            lm = _mimo_loss(cfg, moved, dout)
            fd[i] = (lp - lm) / (2 * EPS)
        g = grads[key]
        assert g.shape == fd.shape, key
        if g.size == 0:
            continue
        unused = (key in ("z", "mimo_z") and not cfg["has_z"] or key == "d" and not cfg["has_d"]
                  or key == "norm_weight" and not cfg["has_output_norm"])
        if unused:
            assert np.all(g == 0) and np.all(fd == 0), key
            continue
        scale = max(np.max(np.abs(fd)), 1e-3)
        err = np.max(np.abs(g - fd)) / scale
        assert err < 2e-6, (name, key, err)


def test_mimo_rank1_adjoints_equal_siso():
    """Rank 1 with unit projections and no norm is the SISO operation; its
    MIMO adjoints equal the SISO ones (and the unit projections' gradients
    are the sums the SISO adjoints imply)."""
    cfg, ins, dout = _setup(**SHAPES["groups"])
    H, P = cfg["num_heads"], cfg["head_dim"]
    ones = np.ones((H, 1, P), np.float32)
    mcfg = dict(cfg, mimo_rank=1, has_output_norm=0)
    gm = oracle.mimo_backward(mcfg, dout, *[ins[k] for k in KEYS], ones, ones, ones,
                              np.ones((H, P), np.float32))
    gs = oracle.siso_backward(cfg, dout, *[ins[k] for k in KEYS])
    for k in KEYS:
        ref = gs[k]
        got = gm[k].reshape(ref.shape)
        assert np.max(np.abs(got - ref)) <= 1e-12 * max(1.0, np.max(np.abs(ref))), k
