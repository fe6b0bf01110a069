"""Materialised O(L^2) kernel form of the Mamba-3 scan (numpy, float64).

TEST INFRASTRUCTURE ONLY: a second, independent statement of the recurrence
that the oracle's token loop (`m3_oracle.cpp`) implements, used to pin it.
It is written as the unrolled sum rather than a recurrence, and handles the
rotary pairs as complex numbers instead of 2x2 rotations, so that an index,
sign or decay-placement slip in either one shows up as a mismatch.

Source: oarust 0.8.6 `src/rs/ml/matrix/mamba3.rs`, `mamba3_siso` and
`mamba3_mimo` operand docs. Unrolling the exponential-trapezoidal update
    h_t = a_t h_{t-1} + s_t a_t X_{t-1} + g_t X_t,   X_t = sum_r x_{t,r} k_{t,r}^T
gives
    h_t = sum_{s<=t} exp(sum_{s<i<=t} adt_i) * (g_s + s_{s+1} [s<t]) * X_s,
so y_{t,r} = sum_{s<=t} Lmask(t,s) * sum_r' (q_{t,r} . k_{s,r'}) x_{s,r'} + D x_{t,r}.
Only tiny shapes are meant (cost B*H*L^2*R^2*(N+P)).
"""
from __future__ import annotations

import numpy as np


def _sig(v):
    return 1.0 / (1.0 + np.exp(-v))


def closed_form_scan(B, L, H, num_groups, P, N, A, R, has_z, has_d, has_norm,
                     c, b, x, z, adt, dt, trap, angle, c_bias, b_bias, d,
                     mimo_x=None, mimo_z=None, mimo_o=None, norm_weight=None):
    """Returns out [B, L, H, P] in float64. Inputs are numpy arrays in the
    mamba3.rs layouts (C/B [B,L,R*G,N], biases [H,R,N] or [H,N] when R == 1)."""
    G = H if num_groups == 0 else num_groups
    f = lambda a: np.asarray(a, dtype=np.float64)
    c = f(c).reshape(B, L, G, R, N)
    b = f(b).reshape(B, L, G, R, N)
    x = f(x).reshape(B, L, H, P)
    z = f(z).reshape(B, L, H, P)
    adt = f(adt).reshape(B, L, H)
    dt = f(dt).reshape(B, L, H)
    trap = f(trap).reshape(B, L, H)
    angle = f(angle).reshape(B, L, A)
    c_bias = f(c_bias).reshape(H, R, N)
    b_bias = f(b_bias).reshape(H, R, N)
    d = f(d).reshape(H)
    mimo = mimo_o is not None
    out = np.zeros((B, L, H, P))
    lam = _sig(trap)
    gam = lam * dt
    scl = (1.0 - lam) * dt
    # theta [B, L, H, A]: running sum of dt * angle over tokens.
    theta = np.cumsum(dt[:, :, :, None] * angle[:, :, None, :], axis=1)
    rot = np.exp(1j * theta)
    hpg = H // G
    for bb in range(B):
        for h in range(H):
            g = h // hpg
            qh = c[bb, :, g] + c_bias[h][None]          # [L, R, N]
            kh = b[bb, :, g] + b_bias[h][None]
            # complex rotary part (pair a <-> a + A) and the untouched tail
            qz = (qh[..., :A] + 1j * qh[..., A:2 * A]) * rot[bb, :, h][:, None, :]
            kz = (kh[..., :A] + 1j * kh[..., A:2 * A]) * rot[bb, :, h][:, None, :]
            # dot[t, r, s, r'] = q_{t,r} . k_{s,r'}
            dot = np.real(np.einsum('tra,sqa->trsq', qz, np.conj(kz)))
            dot = dot + np.einsum('trn,sqn->trsq', qh[..., 2 * A:], kh[..., 2 * A:])
            xs = x[bb, :, h]                            # [L, P]
            if mimo:
                xr = xs[:, None, :] * f(mimo_x).reshape(H, R, P)[h][None]   # [L, R, P]
            else:
                xr = xs[:, None, :]
            cum = np.cumsum(adt[bb, :, h])
            y = np.zeros((L, R, P))
            for t in range(L):
                for s in range(t + 1):
                    decay = np.exp(cum[t] - cum[s])
                    coef = gam[bb, s, h] + (scl[bb, s + 1, h] if s < t else 0.0)
                    y[t] += decay * coef * np.einsum('rq,qp->rp', dot[t, :, s, :], xr[s])
            if has_d:
                y += d[h] * xr
            if not mimo:
                yo = y[:, 0, :]
                if has_z:
                    yo = yo * (z[bb, :, h] * _sig(z[bb, :, h]))
                out[bb, :, h] = yo
            else:
                mz = f(mimo_z).reshape(H, R, P)[h]
                mo = f(mimo_o).reshape(H, R, P)[h]
                if has_z:
                    zr = z[bb, :, h][:, None, :] * mz[None]
                    y = y * (zr * _sig(zr))
                o = np.einsum('trp,rp->tp', y, mo)
                if has_norm:
                    nw = f(norm_weight).reshape(H, P)[h]
                    o = o / np.sqrt(np.mean(o * o, axis=1, keepdims=True) + 1e-5) * nw[None]
                out[bb, :, h] = o
    return out
