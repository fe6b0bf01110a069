"""Seeded synthetic inputs for the Mamba-3 scan workloads.

This module only draws random numbers with the shapes and value distributions
of the workloads below; it holds none of the method's arithmetic, so both the
CUDA path and the CPU oracle can be fed from it. Every array is float32,
C-contiguous, in the operand layouts of oarust's `mamba3_siso` / `mamba3_mimo`
(C/B [B,L,R*G,N], x/z [B,L,H,P], adt/dt/trap [B,L,H], angle [B,L,A],
biases [H,R,N] ([H,N] when R == 1), D [H], mimo_* [H,R,P], norm_weight [H,P]).

Generator: numpy PCG64 seeded with 0x4D330000 + workload index.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, asdict, replace

import numpy as np

SEED_BASE = 0x4D330000


@dataclass(frozen=True)
class Workload:
    name: str
    batch_size: int
    sequence_length: int
    num_heads: int
    num_groups: int
    head_dim: int
    state_size: int
    num_rope_angles: int
    mimo_rank: int = 1
    has_z: int = 1
    has_d: int = 1
    has_output_norm: int = 0
    seed_index: int = 0
    steps: int = 0          # decode workloads: number of single-token calls

    def cfg(self, **override):
        d = {k: v for k, v in asdict(self).items() if k not in ("name", "seed_index", "steps")}
        d.update(override)
        return d

    def with_(self, **kw):
        return replace(self, **kw)

    @property
    def tokens(self):
        return self.batch_size * self.sequence_length


# The five workloads. Sizes and distributions are those of the benchmark
# configurations; each is named by what it is.
TINY_SISO = Workload("tiny SISO B1 L64 H2 G1 P16 N16 A8", 1, 64, 2, 1, 16, 16, 8, seed_index=1)
SISO_1B = Workload("SISO 1B-layer B8 L2048 H32 G1 P64 N128 A32", 8, 2048, 32, 1, 64, 128, 32,
                   seed_index=2)
SISO_LONG = Workload("long-context SISO B2 L16384 H32 G4 P64 N128 A64", 2, 16384, 32, 4, 64, 128,
                     64, seed_index=3)
MIMO_R4 = Workload("MIMO R4 B4 L4096 H32 G1 P64 N64 A32 norm", 4, 4096, 32, 1, 64, 64, 32,
                   mimo_rank=4, has_output_norm=1, seed_index=4)
DECODE_STEP = Workload("decode step B256 H32 G1 P64 N128 A32 x512", 256, 1, 32, 1, 64, 128, 32,
                       seed_index=5, steps=512)

WORKLOADS = [TINY_SISO, SISO_1B, SISO_LONG, MIMO_R4, DECODE_STEP]

# Preprocess settings of the tiny workload.
TINY_PRE = dict(epsilon=1e-6, dt_min=1e-3, dt_max=0.1, a_floor=1e-4)


def rng_for(w: Workload, salt: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(SEED_BASE + w.seed_index + 1000 * salt))


def packed_width(inner, state, heads, angles, groups, rank):
    return 2 * inner + 2 * groups * rank * state + 3 * heads + angles


def _normal(rng, shape, sigma=1.0):
    a = rng.standard_normal(size=shape, dtype=np.float32)
    if sigma != 1.0:
        a *= np.float32(sigma)
    return a


def _unit_rms_rows(rng, shape):
    """Rows drawn uniformly on the sphere of radius sqrt(n): a standard normal
    vector scaled to unit root-mean-square (the distribution of an
    RMS-normalised Gaussian row)."""
    a = rng.standard_normal(size=shape, dtype=np.float32)
    n = shape[-1]
    norm = np.sqrt(np.sum(a.astype(np.float64) ** 2, axis=-1, keepdims=True) / n)
    norm[norm == 0] = 1.0
    return (a / norm).astype(np.float32)


def scan_inputs(w: Workload, salt: int = 0, *, length=None):
    """Scan operands for workload w: x, z ~ N(0,1); B, C rows unit-RMS Gaussian;
    dt log-uniform on [1e-3, 0.1]; adt = -A*dt with A ~ U(1,16) per (b,t,h);
    trap ~ N(0,1); angle ~ N(0, 0.5^2); c_bias, b_bias ~ N(0, 0.1^2); D = 1.
    MIMO adds mimo_x/z/o ~ N(0, 1/R) and norm_weight = 1 + N(0, 0.02^2)."""
    rng = rng_for(w, salt)
    B, L, H, P = w.batch_size, length or w.sequence_length, w.num_heads, w.head_dim
    G = H if w.num_groups == 0 else w.num_groups
    N, A, R = w.state_size, w.num_rope_angles, w.mimo_rank
    out = {}
    out["c"] = _unit_rms_rows(rng, (B, L, R * G, N))
    out["b"] = _unit_rms_rows(rng, (B, L, R * G, N))
    out["x"] = _normal(rng, (B, L, H, P))
    out["z"] = _normal(rng, (B, L, H, P))
    dt = np.exp(rng.uniform(math.log(1e-3), math.log(0.1), size=(B, L, H))).astype(np.float32)
    a_mag = rng.uniform(1.0, 16.0, size=(B, L, H)).astype(np.float32)
    out["dt"] = dt
    out["adt"] = (-a_mag * dt).astype(np.float32)
    out["trap"] = _normal(rng, (B, L, H))
    out["angle"] = _normal(rng, (B, L, A), 0.5)
    bias_shape = (H, N) if R == 1 else (H, R, N)
    out["c_bias"] = _normal(rng, bias_shape, 0.1)
    out["b_bias"] = _normal(rng, bias_shape, 0.1)
    out["d"] = np.ones((H,), dtype=np.float32)
    if R > 1 or w.has_output_norm:
        s = 1.0 / math.sqrt(R)
        out["mimo_x"] = _normal(rng, (H, R, P), s)
        out["mimo_z"] = _normal(rng, (H, R, P), s)
        out["mimo_o"] = _normal(rng, (H, R, P), s)
        out["norm_weight"] = (1.0 + _normal(rng, (H, P), 0.02)).astype(np.float32)
    return out


def tiny_projection(w: Workload = TINY_SISO, salt: int = 0):
    """Packed projection for the tiny workload: projected ~ N(0,1) over all
    columns, dt_bias ~ U(-4,-2); plus scan biases ~ N(0, 0.1^2) and D = 1."""
    rng = rng_for(w, 100 + salt)
    G = w.num_groups
    W = packed_width(w.num_heads * w.head_dim, w.state_size, w.num_heads, w.num_rope_angles, G,
                     w.mimo_rank)
    rows = w.batch_size * w.sequence_length
    projected = _normal(rng, (rows, W))
    dt_bias = rng.uniform(-4.0, -2.0, size=(w.num_heads,)).astype(np.float32)
    bias_shape = (w.num_heads, w.state_size)
    return dict(projected=projected, dt_bias=dt_bias, c_bias=_normal(rng, bias_shape, 0.1),
                b_bias=_normal(rng, bias_shape, 0.1),
                d=np.ones((w.num_heads,), dtype=np.float32))


def layer_projection(w: Workload, salt: int = 0):
    """Packed projection [B*L, W] at a workload's layer shape, drawn per column
    block so that the preprocess outputs follow that workload's scan-input
    distributions: z, x, B, C, trap ~ N(0,1); dt_raw ~ U(ln 1e-3, ln 0.1) with
    dt_bias = 0 (softplus is close to exp there, so dt is close to log-uniform
    on [1e-3, 0.1]); a_raw ~ U(1,16) (softplus is close to the identity there);
    angle ~ N(0, 0.5^2)."""
    rng = rng_for(w, 200 + salt)
    H, P, N, A = w.num_heads, w.head_dim, w.state_size, w.num_rope_angles
    G = H if w.num_groups == 0 else w.num_groups
    R = w.mimo_rank
    I = H * P
    rows = w.batch_size * w.sequence_length
    W = packed_width(I, N, H, A, G, R)
    proj = np.empty((rows, W), dtype=np.float32)
    o = 0
    proj[:, o:o + 2 * I + 2 * G * R * N] = _normal(rng, (rows, 2 * I + 2 * G * R * N))
    o += 2 * I + 2 * G * R * N
    proj[:, o:o + H] = rng.uniform(math.log(1e-3), math.log(0.1), size=(rows, H))
    o += H
    proj[:, o:o + H] = rng.uniform(1.0, 16.0, size=(rows, H))
    o += H
    proj[:, o:o + H] = _normal(rng, (rows, H))
    o += H
    proj[:, o:o + A] = _normal(rng, (rows, A), 0.5)
    dt_bias = np.zeros((H,), dtype=np.float32)
    return dict(projected=proj, dt_bias=dt_bias)


PRE_DEFAULT = dict(epsilon=1e-6, dt_min=1e-3, dt_max=0.1, a_floor=1e-4)


def decode_inputs(w: Workload, steps=None, salt: int = 0):
    """Per-token operands for `steps` decode calls: the scan inputs of a
    length-`steps` sequence (workload distributions), sliced one token per call."""
    steps = steps or w.steps
    return scan_inputs(w, salt, length=steps)


def scan_params(w: Workload, salt: int = 0):
    """Per-head parameters only (no per-token operands): c_bias, b_bias
    ~ N(0, 0.1^2), D = 1, and for MIMO mimo_x/z/o ~ N(0, 1/R), norm_weight
    = 1 + N(0, 0.02^2)."""
    rng = rng_for(w, 300 + salt)
    H, P, N, R = w.num_heads, w.head_dim, w.state_size, w.mimo_rank
    bias_shape = (H, N) if R == 1 else (H, R, N)
    out = dict(c_bias=_normal(rng, bias_shape, 0.1), b_bias=_normal(rng, bias_shape, 0.1),
               d=np.ones((H,), dtype=np.float32))
    if R > 1 or w.has_output_norm:
        s = 1.0 / math.sqrt(R)
        out["mimo_x"] = _normal(rng, (H, R, P), s)
        out["mimo_z"] = _normal(rng, (H, R, P), s)
        out["mimo_o"] = _normal(rng, (H, R, P), s)
        out["norm_weight"] = (1.0 + _normal(rng, (H, P), 0.02)).astype(np.float32)
    return out


PRE_OUTPUTS = ("x", "z", "bh", "ch", "dt", "adt", "trap", "angle")


def preprocess_output_gradient(w: Workload, shapes: dict, salt: int = 0):
    """Gradients of the eight preprocess outputs fed to the preprocess adjoint:
    each ~ N(0,1), in the shape `shapes` gives for it (name -> shape)."""
    rng = rng_for(w, 600 + salt)
    return {k: _normal(rng, shapes[k]) for k in PRE_OUTPUTS}


def output_gradient(w: Workload, salt: int = 0, *, length=None):
    """The gradient of the scan output fed to the SISO backward: dout ~ N(0,1)
    in the output layout [B, L, H, P]."""
    rng = rng_for(w, 500 + salt)
    L = length or w.sequence_length
    return _normal(rng, (w.batch_size, L, w.num_heads, w.head_dim))
