"""ctypes binding of libm3.so (argument marshalling only).

Each function has the name of the C entry point it calls and takes torch
tensors (CUDA, float32, contiguous) in the C argument order; it passes their
device pointers and the current CUDA stream, and raises M3Error on a nonzero
status. No step of the computation runs here: if libm3.so is missing the call
fails loudly, there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libm3.so")

M3_OK = 0
M3_ERR_INVALID_ARGUMENT = 1
M3_ERR_UNALIGNED = 2
M3_ERR_WORKSPACE = 3
M3_ERR_CUDA = 4
M3_ERR_TIMEOUT = 5
M3_ERR_DEVICE_STATE = 6
M3_MATH_FP32 = 0
M3_MATH_TF32 = 1

EXPORTED = ("m3_preprocess", "m3_preprocess_backward_workspace", "m3_preprocess_backward",
            "m3_siso_forward_workspace", "m3_siso_forward",
            "m3_siso_forward_static", "m3_siso_forward_static_status",
            "m3_siso_forward_packed_workspace", "m3_siso_forward_packed",
            "m3_mimo_forward_packed_workspace", "m3_mimo_forward_packed", "m3_siso_prefill_workspace", "m3_siso_prefill",
            "m3_mimo_prefill_workspace", "m3_mimo_prefill",
            "m3_siso_backward_workspace", "m3_siso_backward",
            "m3_mimo_backward_workspace", "m3_mimo_backward",
            "m3_mimo_forward_workspace", "m3_mimo_forward", "m3_siso_step", "m3_mimo_step",
            "m3_workspace_status", "m3_selftest_wait_timeout", "m3_status_string",
            "m3_launch_count")


class M3Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: status {status} ({status_string(status)})")


class PreprocessConfig(ctypes.Structure):
    """m3_preprocess_config (mirrors Mamba3PreprocessConfig)."""
    _fields_ = [("inner_size", ctypes.c_int64), ("state_size", ctypes.c_int64),
                ("num_heads", ctypes.c_int64), ("num_rope_angles", ctypes.c_int64),
                ("num_groups", ctypes.c_int64), ("mimo_rank", ctypes.c_int64),
                ("epsilon", ctypes.c_float), ("dt_min", ctypes.c_float),
                ("dt_max", ctypes.c_float), ("a_floor", ctypes.c_float)]


class SsmConfig(ctypes.Structure):
    """m3_ssm_config (mirrors SsmConfig, plus math_mode)."""
    _fields_ = [("batch_size", ctypes.c_int64), ("sequence_length", ctypes.c_int64),
                ("num_heads", ctypes.c_int64), ("num_groups", ctypes.c_int64),
                ("head_dim", ctypes.c_int64), ("state_size", ctypes.c_int64),
                ("num_rope_angles", ctypes.c_int64), ("mimo_rank", ctypes.c_int64),
                ("has_z", ctypes.c_int32), ("has_d", ctypes.c_int32),
                ("has_output_norm", ctypes.c_int32), ("math_mode", ctypes.c_int32)]


def ssm_config(d: dict, math_mode: int = M3_MATH_FP32) -> SsmConfig:
    return SsmConfig(d["batch_size"], d["sequence_length"], d["num_heads"], d["num_groups"],
                     d["head_dim"], d["state_size"], d["num_rope_angles"], d.get("mimo_rank", 1),
                     int(d.get("has_z", 1)), int(d.get("has_d", 1)),
                     int(d.get("has_output_norm", 0)), int(d.get("math_mode", math_mode)))


def preprocess_config(**kw) -> PreprocessConfig:
    return PreprocessConfig(kw["inner_size"], kw["state_size"], kw["num_heads"],
                            kw["num_rope_angles"], kw["num_groups"], kw["mimo_rank"],
                            kw["epsilon"], kw["dt_min"], kw["dt_max"], kw["a_floor"])


_lock = threading.Lock()
_lib = None
_vp = ctypes.c_void_p


def load_library():
    """Loads libm3.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libm3.so not built ({LIB_PATH}); run "
                               "selective_state_space_mamba3_gb300.build.build()")
        lib = ctypes.CDLL(LIB_PATH)
        cfgp = ctypes.POINTER(SsmConfig)
        lib.m3_preprocess.argtypes = [ctypes.POINTER(PreprocessConfig), ctypes.c_int64] + [_vp] * 11
        lib.m3_preprocess_backward_workspace.argtypes = [ctypes.POINTER(PreprocessConfig),
                                                         ctypes.c_int64,
                                                         ctypes.POINTER(ctypes.c_size_t)]
        lib.m3_preprocess_backward.argtypes = ([ctypes.POINTER(PreprocessConfig), ctypes.c_int64] +
                                               [_vp] * 13 + [ctypes.c_size_t, _vp])
        lib.m3_siso_forward_workspace.argtypes = [cfgp, ctypes.POINTER(ctypes.c_size_t)]
        lib.m3_mimo_forward_workspace.argtypes = [cfgp, ctypes.POINTER(ctypes.c_size_t)]
        lib.m3_siso_forward.argtypes = [cfgp] + [_vp] * 13 + [ctypes.c_size_t, _vp]
        lib.m3_mimo_forward.argtypes = [cfgp] + [_vp] * 17 + [ctypes.c_size_t, _vp]
        lib.m3_siso_forward_static.argtypes = [cfgp] + [_vp] * 12 + [_vp]
        lib.m3_siso_forward_static_status.argtypes = [_vp]
        pcfgp = ctypes.POINTER(PreprocessConfig)
        lib.m3_siso_forward_packed_workspace.argtypes = [cfgp, pcfgp, ctypes.POINTER(ctypes.c_size_t)]
        lib.m3_siso_forward_packed.argtypes = [cfgp, pcfgp] + [_vp] * 7 + [ctypes.c_size_t, _vp]
        lib.m3_mimo_forward_packed_workspace.argtypes = [cfgp, pcfgp, ctypes.POINTER(ctypes.c_size_t)]
        lib.m3_mimo_forward_packed.argtypes = [cfgp, pcfgp] + [_vp] * 11 + [ctypes.c_size_t, _vp]
        lib.m3_siso_prefill_workspace.argtypes = [cfgp, ctypes.POINTER(ctypes.c_size_t)]
        lib.m3_mimo_prefill_workspace.argtypes = [cfgp, ctypes.POINTER(ctypes.c_size_t)]
        lib.m3_siso_prefill.argtypes = [cfgp] + [_vp] * 17 + [ctypes.c_size_t, _vp]
        lib.m3_mimo_prefill.argtypes = [cfgp] + [_vp] * 21 + [ctypes.c_size_t, _vp]
        lib.m3_siso_step.argtypes = [cfgp] + [_vp] * 16 + [_vp]
        lib.m3_siso_backward_workspace.argtypes = [cfgp, ctypes.POINTER(ctypes.c_size_t)]
        lib.m3_siso_backward.argtypes = [cfgp] + [_vp] * 24 + [ctypes.c_size_t, _vp]
        lib.m3_mimo_backward_workspace.argtypes = [cfgp, ctypes.POINTER(ctypes.c_size_t)]
        lib.m3_mimo_backward.argtypes = [cfgp] + [_vp] * 32 + [ctypes.c_size_t, _vp]
        lib.m3_mimo_step.argtypes = [cfgp] + [_vp] * 20 + [_vp]
        lib.m3_workspace_status.argtypes = [_vp, ctypes.c_size_t, _vp]
        lib.m3_selftest_wait_timeout.argtypes = [_vp, ctypes.c_size_t, ctypes.c_int64, _vp]
        lib.m3_status_string.argtypes = [ctypes.c_int]
        lib.m3_status_string.restype = ctypes.c_char_p
        lib.m3_launch_count.restype = ctypes.c_uint64
        for name in EXPORTED:
            if name not in ("m3_status_string", "m3_launch_count"):
                getattr(lib, name).restype = ctypes.c_int
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load_library().m3_status_string(int(status)).decode()


def launch_count() -> int:
    return int(load_library().m3_launch_count())


def _ptr(t):
    """Device pointer of a CUDA float32 contiguous tensor (None passes NULL)."""
    if t is None:
        return None
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch.Tensor")
    if t.device.type != "cuda" or t.dtype != torch.float32 or not t.is_contiguous():
        raise TypeError("operands must be contiguous float32 CUDA tensors")
    return t.data_ptr() if t.numel() > 0 else None


def _stream(stream):
    if stream is not None:
        return stream if isinstance(stream, int) else stream.cuda_stream
    import torch
    return torch.cuda.current_stream().cuda_stream


def _check(status, where):
    if status != M3_OK:
        raise M3Error(status, where)


def m3_preprocess(cfg: PreprocessConfig, rows, projected, dt_bias, x, z, bh, ch, dt, adt, trap,
                  angle, stream=None):
    lib = load_library()
    _check(lib.m3_preprocess(ctypes.byref(cfg), int(rows), *[_ptr(t) for t in (
        projected, dt_bias, x, z, bh, ch, dt, adt, trap, angle)], _stream(stream)), "m3_preprocess")


def m3_preprocess_backward_workspace(cfg: PreprocessConfig, rows) -> int:
    n = ctypes.c_size_t(0)
    _check(load_library().m3_preprocess_backward_workspace(ctypes.byref(cfg), int(rows),
                                                           ctypes.byref(n)),
           "m3_preprocess_backward_workspace")
    return n.value


def m3_preprocess_backward(cfg: PreprocessConfig, rows, projected, dt_bias, grad_x, grad_z,
                           grad_bh, grad_ch, grad_dt, grad_adt, grad_trap, grad_angle,
                           grad_projected, grad_dt_bias, workspace=None, stream=None):
    wp, wn = _ws(workspace)
    _check(load_library().m3_preprocess_backward(ctypes.byref(cfg), int(rows), *[_ptr(t) for t in (
        projected, dt_bias, grad_x, grad_z, grad_bh, grad_ch, grad_dt, grad_adt, grad_trap,
        grad_angle, grad_projected, grad_dt_bias)], wp, wn, _stream(stream)),
        "m3_preprocess_backward")


def m3_siso_forward_workspace(cfg: SsmConfig) -> int:
    n = ctypes.c_size_t(0)
    _check(load_library().m3_siso_forward_workspace(ctypes.byref(cfg), ctypes.byref(n)),
           "m3_siso_forward_workspace")
    return n.value


def m3_mimo_forward_workspace(cfg: SsmConfig) -> int:
    n = ctypes.c_size_t(0)
    _check(load_library().m3_mimo_forward_workspace(ctypes.byref(cfg), ctypes.byref(n)),
           "m3_mimo_forward_workspace")
    return n.value


def _ws(workspace):
    if workspace is None:
        return None, 0
    return workspace.data_ptr(), workspace.numel() * workspace.element_size()


def m3_siso_forward(cfg: SsmConfig, c, b, x, z, adt, dt, trap, angle, c_bias, b_bias, d, out,
                    workspace=None, stream=None):
    wp, wn = _ws(workspace)
    _check(load_library().m3_siso_forward(ctypes.byref(cfg), *[_ptr(t) for t in (
        c, b, x, z, adt, dt, trap, angle, c_bias, b_bias, d, out)], wp, wn, _stream(stream)),
        "m3_siso_forward")


def m3_siso_forward_static(cfg: SsmConfig, c, b, x, z, adt, dt, trap, angle, c_bias, b_bias, d,
                           out, stream=None):
    """m3_siso_forward without a workspace: the library's fixed device scratch
    array is used instead (for callers that cannot allocate device memory)."""
    _check(load_library().m3_siso_forward_static(ctypes.byref(cfg), *[_ptr(t) for t in (
        c, b, x, z, adt, dt, trap, angle, c_bias, b_bias, d, out)], _stream(stream)),
        "m3_siso_forward_static")


def m3_siso_forward_packed_workspace(cfg: SsmConfig, pcfg: PreprocessConfig) -> int:
    n = ctypes.c_size_t(0)
    _check(load_library().m3_siso_forward_packed_workspace(ctypes.byref(cfg), ctypes.byref(pcfg),
                                                            ctypes.byref(n)),
           "m3_siso_forward_packed_workspace")
    return n.value


def m3_siso_forward_packed(cfg: SsmConfig, pcfg: PreprocessConfig, projected, dt_bias, c_bias,
                           b_bias, d, out, workspace=None, stream=None):
    """m3_preprocess and m3_siso_forward in one call (packed projection in,
    scan output out)."""
    wp, wn = _ws(workspace)
    _check(load_library().m3_siso_forward_packed(ctypes.byref(cfg), ctypes.byref(pcfg), *[
        _ptr(t) for t in (projected, dt_bias, c_bias, b_bias, d, out)], wp, wn, _stream(stream)),
        "m3_siso_forward_packed")


def m3_mimo_forward_packed_workspace(cfg: SsmConfig, pcfg: PreprocessConfig) -> int:
    n = ctypes.c_size_t(0)
    _check(load_library().m3_mimo_forward_packed_workspace(ctypes.byref(cfg), ctypes.byref(pcfg),
                                                            ctypes.byref(n)),
           "m3_mimo_forward_packed_workspace")
    return n.value


def m3_mimo_forward_packed(cfg: SsmConfig, pcfg: PreprocessConfig, projected, dt_bias, c_bias,
                           b_bias, d, mimo_x, mimo_z, mimo_o, norm_weight, out, workspace=None,
                           stream=None):
    """m3_preprocess and m3_mimo_forward in one call."""
    wp, wn = _ws(workspace)
    _check(load_library().m3_mimo_forward_packed(ctypes.byref(cfg), ctypes.byref(pcfg), *[
        _ptr(t) for t in (projected, dt_bias, c_bias, b_bias, d, mimo_x, mimo_z, mimo_o,
                          norm_weight, out)], wp, wn, _stream(stream)), "m3_mimo_forward_packed")


def m3_siso_forward_static_status(stream=None) -> int:
    """Status word of the last m3_siso_forward_static call on the current
    device (waits for the stream): M3_OK, M3_ERR_TIMEOUT or M3_ERR_DEVICE_STATE."""
    return int(load_library().m3_siso_forward_static_status(_stream(stream)))


def m3_siso_prefill_workspace(cfg: SsmConfig) -> int:
    n = ctypes.c_size_t(0)
    _check(load_library().m3_siso_prefill_workspace(ctypes.byref(cfg), ctypes.byref(n)),
           "m3_siso_prefill_workspace")
    return n.value


def m3_mimo_prefill_workspace(cfg: SsmConfig) -> int:
    n = ctypes.c_size_t(0)
    _check(load_library().m3_mimo_prefill_workspace(ctypes.byref(cfg), ctypes.byref(n)),
           "m3_mimo_prefill_workspace")
    return n.value


def m3_siso_prefill(cfg: SsmConfig, c, b, x, z, adt, dt, trap, angle, c_bias, b_bias, d,
                    ssm_state, angle_state, k_state, v_state, out, workspace=None, stream=None):
    wp, wn = _ws(workspace)
    _check(load_library().m3_siso_prefill(ctypes.byref(cfg), *[_ptr(t) for t in (
        c, b, x, z, adt, dt, trap, angle, c_bias, b_bias, d, ssm_state, angle_state, k_state,
        v_state, out)], wp, wn, _stream(stream)), "m3_siso_prefill")


def m3_siso_backward_workspace(cfg: SsmConfig) -> int:
    n = ctypes.c_size_t(0)
    _check(load_library().m3_siso_backward_workspace(ctypes.byref(cfg), ctypes.byref(n)),
           "m3_siso_backward_workspace")
    return n.value


def m3_siso_backward(cfg: SsmConfig, grad_out, c, b, x, z, adt, dt, trap, angle, c_bias, b_bias,
                     d, grad_c, grad_b, grad_x, grad_z, grad_adt, grad_dt, grad_trap, grad_angle,
                     grad_c_bias, grad_b_bias, grad_d, workspace=None, stream=None):
    wp, wn = _ws(workspace)
    _check(load_library().m3_siso_backward(ctypes.byref(cfg), *[_ptr(t) for t in (
        grad_out, c, b, x, z, adt, dt, trap, angle, c_bias, b_bias, d, grad_c, grad_b, grad_x,
        grad_z, grad_adt, grad_dt, grad_trap, grad_angle, grad_c_bias, grad_b_bias, grad_d)],
        wp, wn, _stream(stream)), "m3_siso_backward")


def m3_mimo_backward_workspace(cfg: SsmConfig) -> int:
    n = ctypes.c_size_t(0)
    _check(load_library().m3_mimo_backward_workspace(ctypes.byref(cfg), ctypes.byref(n)),
           "m3_mimo_backward_workspace")
    return n.value


def m3_mimo_backward(cfg: SsmConfig, grad_out, c, b, x, z, adt, dt, trap, angle, c_bias, b_bias,
                     d, mimo_x, mimo_z, mimo_o, norm_weight, grad_c, grad_b, grad_x, grad_z,
                     grad_adt, grad_dt, grad_trap, grad_angle, grad_c_bias, grad_b_bias, grad_d,
                     grad_mimo_x, grad_mimo_z, grad_mimo_o, grad_norm_weight, workspace=None,
                     stream=None):
    wp, wn = _ws(workspace)
    _check(load_library().m3_mimo_backward(ctypes.byref(cfg), *[_ptr(t) for t in (
        grad_out, c, b, x, z, adt, dt, trap, angle, c_bias, b_bias, d, mimo_x, mimo_z, mimo_o,
        norm_weight, grad_c, grad_b, grad_x, grad_z, grad_adt, grad_dt, grad_trap, grad_angle,
        grad_c_bias, grad_b_bias, grad_d, grad_mimo_x, grad_mimo_z, grad_mimo_o,
        grad_norm_weight)], wp, wn, _stream(stream)), "m3_mimo_backward")


def m3_mimo_prefill(cfg: SsmConfig, c, b, x, z, adt, dt, trap, angle, c_bias, b_bias, d, mimo_x,
                    mimo_z, mimo_o, norm_weight, ssm_state, angle_state, k_state, v_state, out,
                    workspace=None, stream=None):
    wp, wn = _ws(workspace)
    _check(load_library().m3_mimo_prefill(ctypes.byref(cfg), *[_ptr(t) for t in (
        c, b, x, z, adt, dt, trap, angle, c_bias, b_bias, d, mimo_x, mimo_z, mimo_o,
        norm_weight, ssm_state, angle_state, k_state, v_state, out)], wp, wn, _stream(stream)),
        "m3_mimo_prefill")


def m3_mimo_forward(cfg: SsmConfig, c, b, x, z, adt, dt, trap, angle, c_bias, b_bias, d, mimo_x,
                    mimo_z, mimo_o, norm_weight, out, workspace=None, stream=None):
    wp, wn = _ws(workspace)
    _check(load_library().m3_mimo_forward(ctypes.byref(cfg), *[_ptr(t) for t in (
        c, b, x, z, adt, dt, trap, angle, c_bias, b_bias, d, mimo_x, mimo_z, mimo_o,
        norm_weight, out)], wp, wn, _stream(stream)), "m3_mimo_forward")


def m3_siso_step(cfg: SsmConfig, c, b, x, z, adt, dt, trap, angle, c_bias, b_bias, d, ssm_state,
                 angle_state, k_state, v_state, out, stream=None):
    _check(load_library().m3_siso_step(ctypes.byref(cfg), *[_ptr(t) for t in (
        c, b, x, z, adt, dt, trap, angle, c_bias, b_bias, d, ssm_state, angle_state, k_state,
        v_state, out)], _stream(stream)), "m3_siso_step")


def m3_mimo_step(cfg: SsmConfig, c, b, x, z, adt, dt, trap, angle, c_bias, b_bias, d, mimo_x,
                 mimo_z, mimo_o, norm_weight, ssm_state, angle_state, k_state, v_state, out,
                 stream=None):
    _check(load_library().m3_mimo_step(ctypes.byref(cfg), *[_ptr(t) for t in (
        c, b, x, z, adt, dt, trap, angle, c_bias, b_bias, d, mimo_x, mimo_z, mimo_o,
        norm_weight, ssm_state, angle_state, k_state, v_state, out)], _stream(stream)),
        "m3_mimo_step")


def m3_workspace_status(workspace, stream=None) -> int:
    wp, wn = _ws(workspace)
    return int(load_library().m3_workspace_status(wp, wn, _stream(stream)))


def m3_selftest_wait_timeout(workspace, budget_cycles, stream=None):
    wp, wn = _ws(workspace)
    _check(load_library().m3_selftest_wait_timeout(wp, wn, int(budget_cycles), _stream(stream)),
           "m3_selftest_wait_timeout")
