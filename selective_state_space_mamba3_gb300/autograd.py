"""torch.autograd bindings of the SISO and MIMO scans: the forward through
m3_siso_forward / m3_mimo_forward and the gradients through m3_siso_backward /
m3_mimo_backward (oarust mamba3.rs `mamba3_siso` / `mamba3_siso_backward` and
`mamba3_mimo` / `mamba3_mimo_backward`: each scan with its adjoint). Argument marshalling only: outputs, gradients and workspaces are
torch allocations on the inputs' device and stream, and every step runs in
libm3's kernels.

    out = siso_scan(cfg, c, b, x, z, adt, dt, trap, angle, c_bias, b_bias, d)
    out = mimo_scan(cfg, c, b, x, z, adt, dt, trap, angle, c_bias, b_bias, d,
                    mimo_x, mimo_z, mimo_o, norm_weight)
    x, z, bh, ch, dt, adt, trap, angle = preprocess(pcfg, projected, dt_bias)

preprocess pairs m3_preprocess with m3_preprocess_backward (`mamba3_preprocess`
/ `mamba3_preprocess_backward`); pcfg is the preprocess config dict of the C
ABI (inner_size, state_size, num_heads, num_rope_angles, num_groups,
mimo_rank, epsilon, dt_min, dt_max, a_floor) and the outputs are 2-D, one row
per packed row.

cfg is the SsmConfig dict of the C ABI (batch_size, sequence_length, num_heads,
num_groups, head_dim, state_size, num_rope_angles, mimo_rank, has_z, has_d,
has_output_norm); math_mode picks the forward's arithmetic (the gradients are
FP32 in either mode). Every tensor must be a contiguous float32 CUDA tensor in
the C ABI's layout; angle may be None when num_rope_angles is 0.
"""
from __future__ import annotations

import torch

from . import _binding as m3

def _workspace(nbytes, like):
    return torch.empty(max(int(nbytes), 16), dtype=torch.uint8, device=like.device)


def _grads_like(tensors):
    return [None if t is None else torch.empty_like(t) for t in tensors]


class _SisoScan(torch.autograd.Function):
    @staticmethod
    def forward(ctx, cfg, math_mode, *ops):
        c = m3.ssm_config(cfg, math_mode)
        x = ops[2]
        out = torch.empty_like(x)
        ws = _workspace(m3.m3_siso_forward_workspace(c), x)
        m3.m3_siso_forward(c, *ops, out, ws)
        ctx.cfg = cfg
        ctx.save_for_backward(*[t if t is not None else torch.empty(0) for t in ops])
        ctx.angle_none = ops[7] is None
        return out

    @staticmethod
    def backward(ctx, grad_out):
        ops = list(ctx.saved_tensors)
        if ctx.angle_none:
            ops[7] = None
        c = m3.ssm_config(ctx.cfg, m3.M3_MATH_FP32)
        grads = _grads_like(ops)
        ws = _workspace(m3.m3_siso_backward_workspace(c), grad_out)
        m3.m3_siso_backward(c, grad_out.contiguous(), *ops, *grads, ws)
        return (None, None, *grads)


class _MimoScan(torch.autograd.Function):
    @staticmethod
    def forward(ctx, cfg, math_mode, *ops):
        c = m3.ssm_config(cfg, math_mode)
        x = ops[2]
        out = torch.empty_like(x)
        ws = _workspace(m3.m3_mimo_forward_workspace(c), x)
        m3.m3_mimo_forward(c, *ops, out, ws)
        ctx.cfg = cfg
        ctx.save_for_backward(*[t if t is not None else torch.empty(0) for t in ops])
        ctx.angle_none = ops[7] is None
        return out

    @staticmethod
    def backward(ctx, grad_out):
        ops = list(ctx.saved_tensors)
        if ctx.angle_none:
            ops[7] = None
        c = m3.ssm_config(ctx.cfg, m3.M3_MATH_FP32)
        grads = _grads_like(ops)
        ws = _workspace(m3.m3_mimo_backward_workspace(c), grad_out)
        m3.m3_mimo_backward(c, grad_out.contiguous(), *ops, *grads, ws)
        return (None, None, *grads)


def _widths(pcfg):
    """Columns of the eight preprocess outputs: x, z, bh, ch, dt, adt, trap, angle."""
    I, H, A = pcfg["inner_size"], pcfg["num_heads"], pcfg["num_rope_angles"]
    bc = pcfg["num_groups"] * pcfg["mimo_rank"] * pcfg["state_size"]
    return (I, I, bc, bc, H, H, H, A)


class _Preprocess(torch.autograd.Function):
    @staticmethod
    def forward(ctx, pcfg, projected, dt_bias):
        c = m3.preprocess_config(**pcfg)
        rows = projected.shape[0]
        outs = [torch.empty(rows, n, device=projected.device) for n in _widths(pcfg)]
        m3.m3_preprocess(c, rows, projected, dt_bias, *outs)
        ctx.pcfg = pcfg
        ctx.save_for_backward(projected, dt_bias)
        return tuple(outs)

    @staticmethod
    def backward(ctx, *grads):
        projected, dt_bias = ctx.saved_tensors
        c = m3.preprocess_config(**ctx.pcfg)
        rows = projected.shape[0]
        # an output the loss does not use contributes a zero gradient
        g = [torch.zeros(rows, n, device=projected.device) if gr is None else gr.contiguous()
             for gr, n in zip(grads, _widths(ctx.pcfg))]
        gp = torch.empty_like(projected)
        gb = torch.empty_like(dt_bias)
        ws = _workspace(m3.m3_preprocess_backward_workspace(c, rows), projected)
        m3.m3_preprocess_backward(c, rows, projected, dt_bias, *g, gp, gb, ws)
        return None, gp, gb


def preprocess(pcfg, projected, dt_bias):
    """`mamba3_preprocess` with its adjoint: (x, z, bh, ch, dt, adt, trap, angle)."""
    return _Preprocess.apply(dict(pcfg), projected, dt_bias)


def siso_scan(cfg, c, b, x, z, adt, dt, trap, angle, c_bias, b_bias, d,
              math_mode=m3.M3_MATH_FP32):
    """`mamba3_siso` with its adjoints: out [B,L,H,P]."""
    return _SisoScan.apply(dict(cfg), math_mode, c, b, x, z, adt, dt, trap, angle, c_bias,
                           b_bias, d)


def mimo_scan(cfg, c, b, x, z, adt, dt, trap, angle, c_bias, b_bias, d, mimo_x, mimo_z, mimo_o,
              norm_weight, math_mode=m3.M3_MATH_FP32):
    """`mamba3_mimo` with its adjoints: out [B,L,H,P]."""
    return _MimoScan.apply(dict(cfg), math_mode, c, b, x, z, adt, dt, trap, angle, c_bias,
                           b_bias, d, mimo_x, mimo_z, mimo_o, norm_weight)
