"""Host-only tests of the C ABI (no GPU needed): the library loads, exports
every entry point declared in include/m3.h, and rejects every geometry the
source pages reject (oarust mamba3.rs `Geometry::resolve`,
`MimoGeometry::resolve`, `PreprocessGeometry::resolve`, the step functions'
L == 1 rule) before it enqueues anything. Pointers here are fake but aligned
addresses: a rejected call never dereferences them."""
import ctypes
import os
import re

import pytest

import selective_state_space_mamba3_gb300 as m3
from selective_state_space_mamba3_gb300 import build as m3build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FAKE = 0x10000          # 16-byte aligned, never dereferenced by a rejected call
FAKE_ODD = 0x10004


@pytest.fixture(scope="module")
def lib():
    m3build.build()
    return m3.load_library()


def header_symbols():
    text = open(os.path.join(ROOT, "include", "m3.h")).read()
    return sorted(set(re.findall(r"^(?:int|const char\*|uint64_t)\s+(m3_\w+)\(", text, re.M)))


def test_exports_every_declared_symbol(lib):
    syms = header_symbols()
    assert len(syms) >= 10
    for s in syms:
        assert hasattr(lib, s), s
    assert set(syms) == set(m3.EXPORTED)


def test_status_strings(lib):
    for code in range(7):
        assert m3.status_string(code)
    assert "unknown" in m3.status_string(99)


def siso_cfg(**kw):
    d = dict(batch_size=2, sequence_length=8, num_heads=4, num_groups=2, head_dim=16,
             state_size=32, num_rope_angles=8, mimo_rank=1, has_z=1, has_d=1,
             has_output_norm=0)
    d.update(kw)
    return m3.ssm_config(d, kw.get("math_mode", 0))


def call_siso(lib, cfg, ptr=FAKE, ws=None, wsn=0, angle=FAKE):
    p = [ptr] * 12
    p[7] = angle
    return lib.m3_siso_forward(ctypes.byref(cfg), *p, ws, wsn, None)


def call_mimo(lib, cfg, ptr=FAKE):
    return lib.m3_mimo_forward(ctypes.byref(cfg), *([ptr] * 16), None, 0, None)


def call_step(lib, cfg, ptr=FAKE, mimo=False):
    if mimo:
        return lib.m3_mimo_step(ctypes.byref(cfg), *([ptr] * 20), None)
    return lib.m3_siso_step(ctypes.byref(cfg), *([ptr] * 16), None)


BAD_SISO = [
    dict(batch_size=0), dict(sequence_length=0), dict(num_heads=0), dict(num_groups=3),
    dict(num_groups=-1), dict(head_dim=0), dict(head_dim=129), dict(state_size=0),
    dict(state_size=129), dict(num_rope_angles=17), dict(state_size=64, num_rope_angles=65),
    dict(mimo_rank=2), dict(has_output_norm=1), dict(math_mode=2),
    dict(batch_size=1 << 20, sequence_length=1 << 12, num_heads=1, num_groups=1),  # >= 2^32 elems
]


@pytest.mark.parametrize("bad", BAD_SISO)
def test_siso_rejects(lib, bad):
    assert call_siso(lib, siso_cfg(**bad)) == m3.M3_ERR_INVALID_ARGUMENT
    n = ctypes.c_size_t(0)
    assert lib.m3_siso_forward_workspace(ctypes.byref(siso_cfg(**bad)), ctypes.byref(n)) == \
        m3.M3_ERR_INVALID_ARGUMENT


BAD_MIMO = [dict(mimo_rank=0), dict(mimo_rank=9), dict(head_dim=128, state_size=64),
            dict(num_groups=3), dict(state_size=16, num_rope_angles=9)]


@pytest.mark.parametrize("bad", BAD_MIMO)
def test_mimo_rejects(lib, bad):
    cfg = siso_cfg(mimo_rank=4, has_output_norm=1, state_size=32, head_dim=32)
    for k, v in bad.items():
        setattr(cfg, k, v)
    assert call_mimo(lib, cfg) == m3.M3_ERR_INVALID_ARGUMENT


def test_null_and_unaligned(lib):
    assert lib.m3_siso_forward(None, *([FAKE] * 12), None, 0, None) == m3.M3_ERR_INVALID_ARGUMENT
    assert call_siso(lib, siso_cfg(), ptr=None) == m3.M3_ERR_INVALID_ARGUMENT
    assert call_siso(lib, siso_cfg(), ptr=FAKE_ODD) == m3.M3_ERR_UNALIGNED
    assert call_siso(lib, siso_cfg(), angle=None) == m3.M3_ERR_INVALID_ARGUMENT
    assert call_mimo(lib, siso_cfg(mimo_rank=2), ptr=None) == m3.M3_ERR_INVALID_ARGUMENT


def test_step_requires_single_token(lib):
    assert call_step(lib, siso_cfg(sequence_length=2)) == m3.M3_ERR_INVALID_ARGUMENT
    assert call_step(lib, siso_cfg(sequence_length=2, mimo_rank=2), mimo=True) == \
        m3.M3_ERR_INVALID_ARGUMENT
    assert call_step(lib, siso_cfg(sequence_length=1, mimo_rank=2)) == m3.M3_ERR_INVALID_ARGUMENT
    assert call_step(lib, siso_cfg(sequence_length=1), ptr=FAKE_ODD) == m3.M3_ERR_UNALIGNED


def pre_cfg(**kw):
    d = dict(inner_size=32, state_size=16, num_heads=2, num_rope_angles=8, num_groups=1,
             mimo_rank=1, epsilon=1e-6, dt_min=1e-3, dt_max=0.1, a_floor=1e-4)
    d.update(kw)
    return m3.preprocess_config(**d)


BAD_PRE = [dict(inner_size=0), dict(state_size=0), dict(num_heads=0), dict(num_groups=0),
           dict(mimo_rank=0), dict(num_rope_angles=9), dict(epsilon=0.0),
           dict(epsilon=float("nan")), dict(dt_min=0.0), dict(dt_min=0.2),
           dict(dt_max=float("inf")), dict(a_floor=0.0), dict(a_floor=float("inf")),
           dict(num_rope_angles=-1)]


@pytest.mark.parametrize("bad", BAD_PRE)
def test_preprocess_rejects(lib, bad):
    assert lib.m3_preprocess(ctypes.byref(pre_cfg(**bad)), 64, *([FAKE] * 10), None) == \
        m3.M3_ERR_INVALID_ARGUMENT


def test_preprocess_rows_and_pointers(lib):
    cfg = pre_cfg()
    assert lib.m3_preprocess(ctypes.byref(cfg), 0, *([FAKE] * 10), None) == m3.M3_ERR_INVALID_ARGUMENT
    assert lib.m3_preprocess(ctypes.byref(cfg), 1 << 30, *([FAKE] * 10), None) == \
        m3.M3_ERR_INVALID_ARGUMENT     # rows * W >= 2^32
    assert lib.m3_preprocess(ctypes.byref(cfg), 64, *([FAKE_ODD] * 10), None) == m3.M3_ERR_UNALIGNED
    # angle may be NULL only when A == 0
    assert lib.m3_preprocess(ctypes.byref(cfg), 64, *([FAKE] * 9), None, None) == \
        m3.M3_ERR_INVALID_ARGUMENT


def test_workspace_status_rejects_null(lib):
    assert lib.m3_workspace_status(None, 0, None) == m3.M3_ERR_INVALID_ARGUMENT


def test_selftest_wait_checks_arguments(lib):
    """The diagnostic timeout entry point validates before any launch."""
    assert lib.m3_selftest_wait_timeout(None, 64, 1000, None) == m3.M3_ERR_INVALID_ARGUMENT
    assert lib.m3_selftest_wait_timeout(FAKE, 8, 1000, None) == m3.M3_ERR_INVALID_ARGUMENT
    assert lib.m3_selftest_wait_timeout(FAKE, 64, 0, None) == m3.M3_ERR_INVALID_ARGUMENT
    assert lib.m3_selftest_wait_timeout(FAKE, 64, 5_000_000_000, None) == m3.M3_ERR_INVALID_ARGUMENT
    assert lib.m3_selftest_wait_timeout(FAKE_ODD, 64, 1000, None) == m3.M3_ERR_UNALIGNED


@pytest.mark.skipif(os.path.exists("/dev/nvidia0") or os.path.exists("/dev/nvidiactl"),
                    reason="a GPU is present: fake pointers must never reach a launch")
def test_failed_launch_is_reported(lib):
    """With no GPU the first launch of a valid call fails inside the CUDA
    runtime: the library must return M3_ERR_CUDA, not crash or succeed."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    # FP32 mode takes the chunked split-operand path here, which needs a
    # workspace; the fake one is never touched because the first CUDA call fails
    assert call_siso(lib, siso_cfg(), ws=FAKE, wsn=1 << 20) == m3.M3_ERR_CUDA
    assert lib.m3_preprocess(ctypes.byref(pre_cfg()), 64, *([FAKE] * 10), None) == m3.M3_ERR_CUDA


def test_static_entry_rejects_workspace_above_its_array(lib):
    """m3_siso_forward_static serves only geometries whose workspace fits its
    fixed 1 MiB device array: the long-context SISO shape in TF32 mode splits
    its 64 sequences into segments whose summary states need about 16 MiB, so
    the call is refused with M3_ERR_WORKSPACE before anything is enqueued (the
    fake pointers are never dereferenced)."""
    cfg = siso_cfg(batch_size=2, sequence_length=16384, num_heads=32, num_groups=4, head_dim=64,
                   state_size=128, num_rope_angles=64, math_mode=m3.M3_MATH_TF32)
    n = ctypes.c_size_t(0)
    assert lib.m3_siso_forward_workspace(ctypes.byref(cfg), ctypes.byref(n)) == m3.M3_OK
    assert n.value > (1 << 20)
    assert lib.m3_siso_forward_static(ctypes.byref(cfg), *([FAKE] * 12), None) == \
        m3.M3_ERR_WORKSPACE
    # invalid geometries are still refused as such
    assert lib.m3_siso_forward_static(ctypes.byref(siso_cfg(head_dim=129)), *([FAKE] * 12),
                                      None) == m3.M3_ERR_INVALID_ARGUMENT


def test_packed_entry_checks_both_configs(lib):
    """m3_siso_forward_packed validates the SsmConfig as m3_siso_forward does
    and requires a preprocess config that describes the same layer."""
    cfg = siso_cfg(head_dim=16, state_size=32, num_heads=4, num_groups=2, num_rope_angles=8)
    good = dict(inner_size=64, state_size=32, num_heads=4, num_rope_angles=8, num_groups=2,
                mimo_rank=1, epsilon=1e-6, dt_min=1e-3, dt_max=0.1, a_floor=1e-4)
    n = ctypes.c_size_t(0)
    pc = m3.preprocess_config(**good)
    assert lib.m3_siso_forward_packed_workspace(ctypes.byref(cfg), ctypes.byref(pc),
                                                ctypes.byref(n)) == m3.M3_OK
    call = lambda c, p, ws=FAKE, wsn=1 << 30: lib.m3_siso_forward_packed(
        ctypes.byref(c), p, *([FAKE] * 6), ws, wsn, None)
    assert call(cfg, None) == m3.M3_ERR_INVALID_ARGUMENT
    for bad in (dict(inner_size=32), dict(state_size=16), dict(num_heads=2),
                dict(num_rope_angles=4), dict(num_groups=4), dict(mimo_rank=2),
                dict(epsilon=0.0), dict(dt_min=0.5)):
        assert call(cfg, ctypes.byref(m3.preprocess_config(**dict(good, **bad)))) == \
            m3.M3_ERR_INVALID_ARGUMENT, bad
    assert call(siso_cfg(head_dim=129), ctypes.byref(pc)) == m3.M3_ERR_INVALID_ARGUMENT
    # a workspace is required (the preprocess outputs live there for this shape)
    assert n.value > 0
    assert call(cfg, ctypes.byref(pc), ws=None, wsn=0) == m3.M3_ERR_WORKSPACE
    assert call(cfg, ctypes.byref(pc), wsn=n.value - 1) == m3.M3_ERR_WORKSPACE
    assert lib.m3_siso_forward_packed(ctypes.byref(cfg), ctypes.byref(pc), *([FAKE_ODD] * 6),
                                      FAKE, 1 << 30, None) == m3.M3_ERR_UNALIGNED


def test_mimo_packed_entry_checks_rank(lib):
    """m3_mimo_forward_packed takes the MIMO geometry rules and a preprocess
    config whose mimo_rank matches the scan's rank."""
    cfg = siso_cfg(head_dim=16, state_size=32, num_heads=4, num_groups=2, num_rope_angles=8,
                   mimo_rank=4, has_output_norm=1)
    good = dict(inner_size=64, state_size=32, num_heads=4, num_rope_angles=8, num_groups=2,
                mimo_rank=4, epsilon=1e-6, dt_min=1e-3, dt_max=0.1, a_floor=1e-4)
    n = ctypes.c_size_t(0)
    pc = m3.preprocess_config(**good)
    assert lib.m3_mimo_forward_packed_workspace(ctypes.byref(cfg), ctypes.byref(pc),
                                                ctypes.byref(n)) == m3.M3_OK and n.value > 0
    call = lambda c, p, ptr=FAKE: lib.m3_mimo_forward_packed(ctypes.byref(c), p, *([ptr] * 10),
                                                             FAKE, 1 << 30, None)
    assert call(cfg, ctypes.byref(m3.preprocess_config(**dict(good, mimo_rank=1)))) == \
        m3.M3_ERR_INVALID_ARGUMENT
    assert call(siso_cfg(mimo_rank=9), ctypes.byref(pc)) == m3.M3_ERR_INVALID_ARGUMENT
    assert call(cfg, ctypes.byref(pc), ptr=None) == m3.M3_ERR_INVALID_ARGUMENT


def test_backward_entries_check_before_launch(lib):
    """m3_siso_backward / m3_mimo_backward: the geometry rules of the forward
    calls, a workspace of the queried size (never 0 bytes), and non-NULL,
    16-byte-aligned pointers, all checked on the host (the fake pointers are
    never dereferenced)."""
    n = ctypes.c_size_t(0)
    good = siso_cfg()
    assert lib.m3_siso_backward_workspace(ctypes.byref(good), ctypes.byref(n)) == m3.M3_OK
    need = n.value
    assert need > 0
    for bad in (siso_cfg(mimo_rank=2), siso_cfg(has_output_norm=1), siso_cfg(head_dim=129),
                siso_cfg(num_heads=3, num_groups=2)):
        assert lib.m3_siso_backward_workspace(ctypes.byref(bad), ctypes.byref(n)) == \
            m3.M3_ERR_INVALID_ARGUMENT
    args = [FAKE] * 23  # grad_out, the 11 operands, the 11 gradients
    assert lib.m3_siso_backward(ctypes.byref(good), *args, None, 0, None) == m3.M3_ERR_WORKSPACE
    assert lib.m3_siso_backward(ctypes.byref(good), *args, FAKE, need - 1, None) == \
        m3.M3_ERR_WORKSPACE
    assert lib.m3_siso_backward(ctypes.byref(good), *args, FAKE_ODD, need, None) == \
        m3.M3_ERR_UNALIGNED
    for i in range(23):
        if i in (8, 19):  # angle and grad_angle may be NULL only when A == 0
            continue
        a = list(args)
        a[i] = None
        assert lib.m3_siso_backward(ctypes.byref(good), *a, FAKE, need, None) == \
            m3.M3_ERR_INVALID_ARGUMENT, i
        a[i] = FAKE_ODD
        assert lib.m3_siso_backward(ctypes.byref(good), *a, FAKE, need, None) == \
            m3.M3_ERR_UNALIGNED, i
    a = list(args)
    a[8] = None  # angle with A > 0
    assert lib.m3_siso_backward(ctypes.byref(good), *a, FAKE, need, None) == \
        m3.M3_ERR_INVALID_ARGUMENT
    mimo = siso_cfg(mimo_rank=4, has_output_norm=1, head_dim=16, state_size=32)
    assert lib.m3_mimo_backward_workspace(ctypes.byref(mimo), ctypes.byref(n)) == m3.M3_OK
    assert n.value > 0
    for bad in (siso_cfg(mimo_rank=9), siso_cfg(mimo_rank=4, head_dim=128, state_size=64)):
        assert lib.m3_mimo_backward_workspace(ctypes.byref(bad), ctypes.byref(n)) == \
            m3.M3_ERR_INVALID_ARGUMENT
    margs = [FAKE] * 31  # grad_out, the 15 operands, the 15 gradients
    assert lib.m3_mimo_backward(ctypes.byref(mimo), *margs, None, 0, None) == m3.M3_ERR_WORKSPACE
    margs[15] = None  # norm_weight
    assert lib.m3_mimo_backward(ctypes.byref(mimo), *margs, FAKE, 1 << 40, None) == \
        m3.M3_ERR_INVALID_ARGUMENT


def test_preprocess_backward_checks_before_launch(lib):
    """m3_preprocess_backward: the m3_preprocess geometry rules, a workspace of
    the queried size, non-NULL 16-byte-aligned pointers (grad_angle may be NULL
    only when A == 0), all checked on the host."""
    n = ctypes.c_size_t(0)
    good = pre_cfg()
    assert lib.m3_preprocess_backward_workspace(ctypes.byref(good), 64, ctypes.byref(n)) == m3.M3_OK
    need = n.value
    assert need > 0
    assert lib.m3_preprocess_backward_workspace(ctypes.byref(good), 64, None) == \
        m3.M3_ERR_INVALID_ARGUMENT
    for bad in BAD_PRE:
        assert lib.m3_preprocess_backward_workspace(ctypes.byref(pre_cfg(**bad)), 64,
                                                    ctypes.byref(n)) == m3.M3_ERR_INVALID_ARGUMENT
        assert lib.m3_preprocess_backward(ctypes.byref(pre_cfg(**bad)), 64, *([FAKE] * 12), FAKE,
                                          need, None) == m3.M3_ERR_INVALID_ARGUMENT
    assert lib.m3_preprocess_backward(ctypes.byref(good), 0, *([FAKE] * 12), FAKE, need, None) == \
        m3.M3_ERR_INVALID_ARGUMENT
    args = [FAKE] * 12  # projected, dt_bias, the 8 output gradients, the 2 results
    assert lib.m3_preprocess_backward(ctypes.byref(good), 64, *args, None, 0, None) == \
        m3.M3_ERR_WORKSPACE
    assert lib.m3_preprocess_backward(ctypes.byref(good), 64, *args, FAKE, need - 1, None) == \
        m3.M3_ERR_WORKSPACE
    assert lib.m3_preprocess_backward(ctypes.byref(good), 64, *args, FAKE_ODD, need, None) == \
        m3.M3_ERR_UNALIGNED
    for i in range(12):
        a = list(args)
        a[i] = None
        assert lib.m3_preprocess_backward(ctypes.byref(good), 64, *a, FAKE, need, None) == \
            m3.M3_ERR_INVALID_ARGUMENT, i
        a[i] = FAKE_ODD
        assert lib.m3_preprocess_backward(ctypes.byref(good), 64, *a, FAKE, need, None) == \
            m3.M3_ERR_UNALIGNED, i
    # grad_angle NULL is accepted without rotary angles (no GPU here: the launch fails)
    a = list(args)
    a[9] = None
    no_rot = pre_cfg(num_rope_angles=0)
    assert lib.m3_preprocess_backward_workspace(ctypes.byref(no_rot), 64, ctypes.byref(n)) == m3.M3_OK
    assert lib.m3_preprocess_backward(ctypes.byref(no_rot), 64, *a, FAKE, n.value, None) == \
        m3.M3_ERR_CUDA
