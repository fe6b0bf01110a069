"""GB300 (sm_103a) Mamba-3 selective-state scan.

The product is the C-ABI library `libm3.so` (declared in include/m3.h):
m3_preprocess, m3_siso_forward, m3_mimo_forward, m3_siso_step, m3_mimo_step,
m3_siso_backward, m3_mimo_backward, m3_preprocess_backward.
This package holds its CUDA sources (`csrc/`), the in-tree build (`build.py`),
a ctypes binding with the same entry-point names (`_binding.py`), torch.autograd
bindings that pair each scan with its adjoints (`autograd.py`) and the seeded
synthetic input generators (`inputs.py`).
"""
from ._binding import (  # noqa: F401
    M3_OK, M3_ERR_INVALID_ARGUMENT, M3_ERR_UNALIGNED, M3_ERR_WORKSPACE, M3_ERR_CUDA,
    M3_ERR_TIMEOUT, M3_ERR_DEVICE_STATE, M3_MATH_FP32, M3_MATH_TF32, EXPORTED, M3Error, PreprocessConfig, SsmConfig,
    ssm_config, preprocess_config, load_library, status_string, launch_count, m3_preprocess,
    m3_siso_forward_workspace, m3_siso_forward, m3_siso_forward_static,
    m3_siso_forward_static_status, m3_siso_forward_packed_workspace, m3_siso_forward_packed,
    m3_mimo_forward_packed_workspace, m3_mimo_forward_packed,
    m3_mimo_forward_workspace, m3_mimo_forward,
    m3_siso_step, m3_mimo_step, m3_workspace_status, LIB_PATH, m3_siso_prefill_workspace,
    m3_mimo_prefill_workspace, m3_siso_prefill, m3_mimo_prefill, m3_selftest_wait_timeout,
    m3_siso_backward_workspace, m3_siso_backward, m3_mimo_backward_workspace,
    m3_mimo_backward, m3_preprocess_backward_workspace, m3_preprocess_backward)
from . import inputs  # noqa: F401
