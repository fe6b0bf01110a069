"""Helpers for the GPU parity tests: move seeded inputs to the device, run the
library through its C ABI, run the oracle on the same inputs, and compare.

Tolerance metric (normwise max-relative error): max|gpu - oracle| / max|oracle|
per output tensor. FP32-exact paths must stay below 1e-5, TF32 tensor-core
paths below 2e-3. The elementwise error max|gpu - oracle| / (|oracle| +
1e-6 max|oracle|) is computed and reported beside it (it is large wherever an
output is tiny, e.g. where the SiLU gate is near zero, so it is not the bar).
"""
import json
import os

import numpy as np

import oracle
import selective_state_space_mamba3_gb300 as m3

SCAN_KEYS = ("c", "b", "x", "z", "adt", "dt", "trap", "angle", "c_bias", "b_bias", "d")
MIMO_KEYS = ("mimo_x", "mimo_z", "mimo_o", "norm_weight")
TOL = {m3.M3_MATH_FP32: 1e-5, m3.M3_MATH_TF32: 2e-3}


def dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def normwise(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    scale = np.max(np.abs(ref)) if ref.size else 0.0
    if scale == 0.0:
        return float(np.max(np.abs(got))) if got.size else 0.0
    return float(np.max(np.abs(got - ref)) / scale)


def elementwise(got, ref):
    """max_i |got_i - ref_i| / (|ref_i| + 1e-6 max|ref|)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if not ref.size:
        return 0.0
    floor = 1e-6 * np.max(np.abs(ref))
    den = np.abs(ref) + (floor if floor > 0 else 1e-300)
    return float(np.max(np.abs(got - ref) / den))


def is_mimo(cfg):
    return cfg["mimo_rank"] > 1 or cfg.get("has_output_norm", 0) or cfg.get("mimo", False)


def gpu_scan(cfg, ins, math_mode=m3.M3_MATH_FP32, mimo=None):
    """Runs m3_siso_forward or m3_mimo_forward on device copies of `ins`;
    returns the output as a numpy float32 array."""
    import torch
    mimo = is_mimo(cfg) if mimo is None else mimo
    c = m3.ssm_config(cfg, math_mode)
    B, L, H, P = cfg["batch_size"], cfg["sequence_length"], cfg["num_heads"], cfg["head_dim"]
    d = {k: dev(ins[k]) for k in SCAN_KEYS}
    if cfg["num_rope_angles"] == 0:
        d["angle"] = None
    out = torch.full((B, L, H, P), float("nan"), device="cuda")
    if mimo:
        for k in MIMO_KEYS:
            d[k] = dev(ins[k])
        wsb = m3.m3_mimo_forward_workspace(c)
        ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device="cuda") if wsb else None
        m3.m3_mimo_forward(c, *[d[k] for k in SCAN_KEYS], *[d[k] for k in MIMO_KEYS], out, ws)
    else:
        wsb = m3.m3_siso_forward_workspace(c)
        ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device="cuda") if wsb else None
        m3.m3_siso_forward(c, *[d[k] for k in SCAN_KEYS], out, ws)
    torch.cuda.synchronize()
    if ws is not None:
        assert m3.m3_workspace_status(ws) == m3.M3_OK
    return out.cpu().numpy()


def oracle_scan(cfg, ins, mimo=None, batch=None):
    """Oracle output; `batch` = slice of batch indices to compute (the
    recurrence is independent per batch row)."""
    mimo = is_mimo(cfg) if mimo is None else mimo
    if batch is not None:
        cfg = dict(cfg, batch_size=batch.stop - batch.start)
        ins = {k: (v[batch] if k in SCAN_KEYS[:8] else v) for k, v in ins.items()}
    extra = {k: ins[k] for k in MIMO_KEYS} if mimo else {}
    return oracle.scan(cfg, *[ins[k] for k in SCAN_KEYS], **extra)


def check_close(got, ref, tol, label=""):
    """Asserts normwise(got, ref) <= tol; when M3_PARITY_REPORT names a file,
    appends the test id, label, both error metrics and the tolerance to it as a
    JSON line."""
    err = normwise(got, ref)
    path = os.environ.get("M3_PARITY_REPORT")
    if path:
        name = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
        with open(path, "a") as f:
            f.write(json.dumps({"test": name, "label": label, "err": err,
                                "elementwise": elementwise(got, ref), "tol": tol}) + "\n")
    assert err <= tol, (label, err, tol)
    return err
