"""Pins for the oracle's SISO adjoints (`m3o_siso_backward`, the eleven
gradients of `SsmBackward` / `mamba3_siso_backward` in oarust mamba3.rs):
every gradient element is checked against the central difference of the
oracle's own forward scan, the definition of the derivative, on tiny inputs.

The loss is sum(out * dout). The inputs are rounded to multiples of 2^-20
(all below 8 in magnitude, so float32 holds them and v +- eps exactly) and
each is moved by +-eps with eps = 2^-12, so that the two forward calls see
exactly v +- eps. The central
difference is then exact up to eps^2 / 6 * f''' (about 1e-8 here) plus the
forward oracle's double rounding; a dropped term, a wrong sign or a
transposed rotation in the adjoint moves its gradient by far more.
"""
import numpy as np
import pytest

import oracle
from selective_state_space_mamba3_gb300 import inputs as gen

KEYS = ("c", "b", "x", "z", "adt", "dt", "trap", "angle", "c_bias", "b_bias", "d")
EPS = 2.0 ** -12

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
