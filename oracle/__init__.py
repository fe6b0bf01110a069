"""CPU oracle for the Mamba-3 selective-state scan (FP64).

TEST INFRASTRUCTURE ONLY. Only the test suite, the smoke check and the
benchmark's CPU-baseline leg may import this package; the library's product
path never does and must fail loudly instead of falling back to it.

`m3_oracle.cpp` (plain C++, double precision, std::thread over (batch, head))
holds the token-by-token recurrence and the preprocess; `closed_form.py` holds
the independent O(L^2) unrolled form used to pin it. The readings taken where
the source pages are silent are listed at the top of `m3_oracle.cpp`.

Pinned functions (see tests/test_oracle_pins.py): preprocess, SISO scan, SISO
step (as the scan with explicit state), MIMO scan, MIMO step; SISO and MIMO
adjoints (tests/test_oracle_backward_pins.py: central differences of the scans);
the preprocess adjoint (tests/test_oracle_preprocess_backward_pins.py: central
differences of the preprocess, the RMS norm's scale invariance, the clamps).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "m3_oracle.cpp")
_LIB_PATH = os.path.join(_HERE, "libm3_oracle.so")
_lock = threading.Lock()
_lib = None

_i64 = ctypes.c_int64
_f64 = ctypes.c_double
_ptr = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compiles m3_oracle.cpp into libm3_oracle.so beside it (g++, -O2)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-pthread",
                               "-o", tmp, _SRC])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.m3o_preprocess.restype = ctypes.c_int
            lib.m3o_preprocess.argtypes = [_i64] * 7 + [_f64] * 4 + [_ptr] * 10 + [ctypes.c_int]
            lib.m3o_preprocess_backward.restype = ctypes.c_int
            lib.m3o_preprocess_backward.argtypes = ([_i64] * 7 + [_f64] * 4 + [_ptr] * 12 +
                                                    [ctypes.c_int])
            lib.m3o_scan.restype = ctypes.c_int
            lib.m3o_scan.argtypes = [_i64] * 8 + [ctypes.c_int] * 3 + [_ptr] * 20 + [ctypes.c_int]
            lib.m3o_siso_backward.restype = ctypes.c_int
            lib.m3o_siso_backward.argtypes = ([_i64] * 7 + [ctypes.c_int] * 2 + [_ptr] * 23 +
                                              [ctypes.c_int])
            lib.m3o_mimo_backward.restype = ctypes.c_int
            lib.m3o_mimo_backward.argtypes = ([_i64] * 8 + [ctypes.c_int] * 3 + [_ptr] * 31 +
                                              [ctypes.c_int])
            _lib = lib
    return _lib


def default_threads() -> int:
    return int(os.environ.get("M3_ORACLE_THREADS", os.cpu_count() or 1))


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def preprocess(projected, dt_bias, *, inner_size, state_size, num_heads, num_rope_angles,
               num_groups, mimo_rank, epsilon, dt_min, dt_max, a_floor, threads=None):
    """Fused projection preprocess. Returns dict of float64 arrays
    x, z [rows, I]; bh, ch [rows, G*R*N]; dt, adt, trap [rows, H]; angle [rows, A]."""
    projected = _f32(projected)
    dt_bias = _f32(dt_bias)
    rows = projected.shape[0]
    I, N, H, A, G, R = inner_size, state_size, num_heads, num_rope_angles, num_groups, mimo_rank
    outs = dict(x=np.zeros((rows, I)), z=np.zeros((rows, I)), bh=np.zeros((rows, G * R * N)),
                ch=np.zeros((rows, G * R * N)), dt=np.zeros((rows, H)), adt=np.zeros((rows, H)),
                trap=np.zeros((rows, H)), angle=np.zeros((rows, A)))
    # epsilon and the bounds are float32 config fields; the oracle sees the same values.
    st = _load().m3o_preprocess(rows, I, N, H, A, G, R, float(np.float32(epsilon)),
                                float(np.float32(dt_min)), float(np.float32(dt_max)),
                                float(np.float32(a_floor)), _p(projected), _p(dt_bias),
                                *[_p(outs[k]) for k in ("x", "z", "bh", "ch", "dt", "adt", "trap", "angle")],
                                threads or default_threads())
    if st != 0:
        raise ValueError("oracle preprocess: invalid geometry")
    return outs


PRE_GRAD_NAMES = ("x", "z", "bh", "ch", "dt", "adt", "trap", "angle")


def preprocess_backward(projected, dt_bias, grads, *, inner_size, state_size, num_heads,
                        num_rope_angles, num_groups, mimo_rank, epsilon, dt_min, dt_max, a_floor,
                        threads=None):
    """Adjoint of the fused projection preprocess. grads: dict of the eight
    output gradients (PRE_GRAD_NAMES, the shapes `preprocess` returns, read as
    float32). Returns dict of float64 arrays projected [rows, W], dt_bias [H]."""
    projected = _f32(projected)
    dt_bias = _f32(dt_bias)
    rows, W = projected.shape
    I, N, H, A, G, R = inner_size, state_size, num_heads, num_rope_angles, num_groups, mimo_rank
    g = {k: _f32(grads[k]) for k in PRE_GRAD_NAMES}
    out = dict(projected=np.zeros((rows, W)), dt_bias=np.zeros((H,)))
    st = _load().m3o_preprocess_backward(rows, I, N, H, A, G, R, float(np.float32(epsilon)),
                                         float(np.float32(dt_min)), float(np.float32(dt_max)),
                                         float(np.float32(a_floor)), _p(projected), _p(dt_bias),
                                         *[_p(g[k]) for k in PRE_GRAD_NAMES],
                                         _p(out["projected"]), _p(out["dt_bias"]),
                                         threads or default_threads())
    if st != 0:
        raise ValueError("oracle preprocess_backward: invalid geometry")
    return out


def scan(cfg, c, b, x, z, adt, dt, trap, angle, c_bias, b_bias, d, mimo_x=None, mimo_z=None,
         mimo_o=None, norm_weight=None, state=None, threads=None):
    """SISO (mimo_o is None) or MIMO token-by-token scan.

    cfg: dict with batch_size, sequence_length, num_heads, num_groups, head_dim,
    state_size, num_rope_angles, mimo_rank, has_z, has_d, has_output_norm.
    state: optional dict of float64 arrays ssm [B,H,P,N], angle [B,H,A],
    k [B,H,R,N], v [B,H,R,P]; read, then overwritten in place.
    Returns out [B, L, H, P] float64."""
    B, L, H = cfg["batch_size"], cfg["sequence_length"], cfg["num_heads"]
    P, N, A, R = cfg["head_dim"], cfg["state_size"], cfg["num_rope_angles"], cfg["mimo_rank"]
    arrs = [_f32(a) for a in (c, b, x, z, adt, dt, trap, angle, c_bias, b_bias, d)]
    mimo = [None if a is None else _f32(a) for a in (mimo_x, mimo_z, mimo_o, norm_weight)]
    out = np.zeros((B, L, H, P))
    st_ptrs = [None] * 4
    if state is not None:
        for key in ("ssm", "angle", "k", "v"):
            arr = state[key]
            if arr.dtype != np.float64 or not arr.flags["C_CONTIGUOUS"]:
                raise TypeError("oracle state arrays must be contiguous float64")
        st_ptrs = [_p(state[k]) for k in ("ssm", "angle", "k", "v")]
    rc = _load().m3o_scan(B, L, H, cfg["num_groups"], P, N, A, R, int(cfg["has_z"]),
                          int(cfg["has_d"]), int(cfg.get("has_output_norm", 0)),
                          *[_p(a) for a in arrs], *[_p(a) for a in mimo], _p(out), *st_ptrs,
                          threads or default_threads())
    if rc != 0:
        raise ValueError("oracle scan: invalid geometry")
    return out


def zero_state(cfg):
    """Zero recurrent state in the step layouts (float64)."""
    B, H = cfg["batch_size"], cfg["num_heads"]
    P, N, A, R = cfg["head_dim"], cfg["state_size"], cfg["num_rope_angles"], cfg["mimo_rank"]
    return dict(ssm=np.zeros((B, H, P, N)), angle=np.zeros((B, H, A)),
                k=np.zeros((B, H, R, N)), v=np.zeros((B, H, R, P)))


def step(cfg, *args, state, **kw):
    """One token (sequence_length must be 1) with explicit state, SISO or MIMO:
    the `mamba3_siso_step` / `mamba3_mimo_step` semantics."""
    if cfg["sequence_length"] != 1:
        raise ValueError("step requires sequence_length == 1")
    return scan(cfg, *args, state=state, **kw)


GRAD_NAMES = ("c", "b", "x", "z", "adt", "dt", "trap", "angle", "c_bias", "b_bias", "d")


def siso_backward(cfg, dout, c, b, x, z, adt, dt, trap, angle, c_bias, b_bias, d, threads=None):
    """The eleven SISO adjoints (`mamba3_siso_backward`) of the scan from a zero
    state, given dout [B,L,H,P], the gradient of its output. Returns a dict of
    float64 arrays keyed by GRAD_NAMES, each in its forward operand's layout:
    c/b [B,L,G,N], x/z [B,L,H,P], adt/dt/trap [B,L,H], angle [B,L,A],
    c_bias/b_bias [H,N], d [H]."""
    B, L, H = cfg["batch_size"], cfg["sequence_length"], cfg["num_heads"]
    P, N, A = cfg["head_dim"], cfg["state_size"], cfg["num_rope_angles"]
    G = cfg["num_groups"] or H
    if cfg.get("mimo_rank", 1) != 1 or cfg.get("has_output_norm", 0):
        raise ValueError("oracle siso_backward: SISO only")
    arrs = [_f32(a) for a in (dout, c, b, x, z, adt, dt, trap, angle, c_bias, b_bias, d)]
    shapes = dict(c=(B, L, G, N), b=(B, L, G, N), x=(B, L, H, P), z=(B, L, H, P),
                  adt=(B, L, H), dt=(B, L, H), trap=(B, L, H), angle=(B, L, A),
                  c_bias=(H, N), b_bias=(H, N), d=(H,))
    g = {k: np.zeros(shapes[k]) for k in GRAD_NAMES}
    rc = _load().m3o_siso_backward(B, L, H, cfg["num_groups"], P, N, A, int(cfg["has_z"]),
                                   int(cfg["has_d"]), *[_p(a) for a in arrs],
                                   *[_p(g[k]) for k in GRAD_NAMES], threads or default_threads())
    if rc != 0:
        raise ValueError("oracle siso_backward: invalid geometry")
    return g


MIMO_GRAD_NAMES = GRAD_NAMES + ("mimo_x", "mimo_z", "mimo_o", "norm_weight")


def mimo_backward(cfg, dout, c, b, x, z, adt, dt, trap, angle, c_bias, b_bias, d, mimo_x, mimo_z,
                  mimo_o, norm_weight, threads=None):
    """The fifteen MIMO adjoints (`mamba3_mimo_backward`) of the scan from a
    zero state, given dout [B,L,H,P]. Returns a dict of float64 arrays keyed by
    MIMO_GRAD_NAMES in the forward operands' layouts: c/b [B,L,R*G,N], x/z
    [B,L,H,P], adt/dt/trap [B,L,H], angle [B,L,A], c_bias/b_bias [H,R,N],
    d [H], mimo_x/z/o [H,R,P], norm_weight [H,P]."""
    B, L, H = cfg["batch_size"], cfg["sequence_length"], cfg["num_heads"]
    P, N, A, R = cfg["head_dim"], cfg["state_size"], cfg["num_rope_angles"], cfg["mimo_rank"]
    G = cfg["num_groups"] or H
    arrs = [_f32(a) for a in (dout, c, b, x, z, adt, dt, trap, angle, c_bias, b_bias, d, mimo_x,
                               mimo_z, mimo_o, norm_weight)]
    shapes = dict(c=(B, L, R * G, N), b=(B, L, R * G, N), x=(B, L, H, P), z=(B, L, H, P),
                  adt=(B, L, H), dt=(B, L, H), trap=(B, L, H), angle=(B, L, A),
                  c_bias=(H, R, N), b_bias=(H, R, N), d=(H,), mimo_x=(H, R, P),
                  mimo_z=(H, R, P), mimo_o=(H, R, P), norm_weight=(H, P))
    g = {k: np.zeros(shapes[k]) for k in MIMO_GRAD_NAMES}
    rc = _load().m3o_mimo_backward(B, L, H, cfg["num_groups"], P, N, A, R, int(cfg["has_z"]),
                                   int(cfg["has_d"]), int(cfg.get("has_output_norm", 0)),
                                   *[_p(a) for a in arrs], *[_p(g[k]) for k in MIMO_GRAD_NAMES],
                                   threads or default_threads())
    if rc != 0:
        raise ValueError("oracle mimo_backward: invalid geometry")
    return g
