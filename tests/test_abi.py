"""The C ABI library builds, loads and exports every entry point that
include/ssd.h declares; host-side argument checks (no GPU needed)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "ssd.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ssd_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from state_space_model_ssd_gb300 import build, _lib
    build.build()
    return _lib.lib()


def _prob(**kw):
    from state_space_model_ssd_gb300 import _lib
    p = dict(batch=1, seqlen=256, nheads=2, headdim=16, dstate=16, ngroups=1, chunk_size=64,
             nseq=0, delta_init=-4.6, dtype=_lib.DTYPE_F32)
    p.update(kw)
    return _lib.Problem(**p)


def test_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert "ssd_forward" in names and "ssd_backward" in names
    for n in names:
        assert hasattr(lib, n), n


def test_version_and_status_strings(lib):
    assert lib.ssd_version() == 1
    for code in range(8):
        assert lib.ssd_status_string(code)


def test_workspace_size_and_dispatch(lib):
    n = ctypes.c_size_t()
    p = _prob()
    assert lib.ssd_workspace_size(ctypes.byref(p), 0, ctypes.byref(n)) == 0
    fwd = n.value
    assert lib.ssd_workspace_size(ctypes.byref(p), 1, ctypes.byref(n)) == 0
    assert n.value > fwd > 0 and fwd % 256 == 0
    assert lib.ssd_dispatch_path(ctypes.byref(p), 0) == b"simt"


@pytest.mark.parametrize("kw,code", [
    (dict(headdim=12), 2), (dict(dstate=256), 2), (dict(chunk_size=48), 2),
    (dict(nheads=3, ngroups=2), 1), (dict(batch=0), 1), (dict(seqlen=-1), 1),
    (dict(dtype=9), 1), (dict(batch=2, nseq=3), 1), (dict(delta_init=float("nan")), 1),
])
def test_rejects_bad_problems(lib, kw, code):
    n = ctypes.c_size_t()
    p = _prob(**kw)
    assert lib.ssd_workspace_size(ctypes.byref(p), 0, ctypes.byref(n)) == code
    assert lib.ssd_dispatch_path(ctypes.byref(p), 0) is None


def test_forward_checks_arguments_before_launch(lib):
    """Bad arguments return an error without touching the GPU (none is present here)."""
    p = _prob()
    fake = ctypes.c_void_p(0x10000)
    ws = ctypes.c_void_p(0x20000)
    # missing workspace
    assert lib.ssd_forward(ctypes.byref(p), fake, fake, fake, fake, None, fake, None, None, 0,
                           None) == 4
    # workspace too small
    assert lib.ssd_forward(ctypes.byref(p), fake, fake, fake, fake, None, fake, None, ws, 16,
                           None) == 4
    # misaligned workspace
    assert lib.ssd_forward(ctypes.byref(p), fake, fake, fake, fake, None, fake, None,
                           ctypes.c_void_p(0x20010), 1 << 30, None) == 3
    # misaligned x
    assert lib.ssd_forward(ctypes.byref(p), ctypes.c_void_p(0x10002), fake, fake, fake, None,
                           fake, None, ws, 1 << 30, None) == 3
    # null y
    assert lib.ssd_forward(ctypes.byref(p), fake, fake, fake, fake, None, None, None, ws,
                           1 << 30, None) == 1
    # cu_seqlens given for a dense problem, and missing for a packed one
    assert lib.ssd_forward(ctypes.byref(p), fake, fake, fake, fake, fake, fake, None, ws,
                           1 << 30, None) == 1
    pv = _prob(nseq=3)
    assert lib.ssd_forward(ctypes.byref(pv), fake, fake, fake, fake, None, fake, None, ws,
                           1 << 30, None) == 1
    # backward: null gradient output
    assert lib.ssd_backward(ctypes.byref(p), fake, fake, fake, fake, None, fake, fake, fake,
                            None, fake, ws, 1 << 30, None) == 1


def test_python_binding_refuses_cpu_tensors(lib):
    import torch
    import state_space_model_ssd_gb300 as ssd
    x = torch.zeros(1, 8, 2, 16)
    with pytest.raises(ValueError):
        ssd.forward(x, torch.zeros(1, 8, 2), torch.zeros(1, 8, 1, 16), torch.zeros(1, 8, 1, 16),
                    delta_init=-4.6)


def test_step_host_checks_arguments_before_any_cuda_call(lib):
    """ssd_step_host sizes its device region on the host and refuses a missing, small or
    misaligned region, or a cu_seqlens that does not match the problem, before it makes
    any CUDA call (none can succeed here)."""
    p = _prob()
    n = ctypes.c_size_t()
    assert lib.ssd_step_host_size(ctypes.byref(p), ctypes.byref(n)) == 0
    ws = ctypes.c_size_t()
    assert lib.ssd_workspace_size(ctypes.byref(p), 1, ctypes.byref(ws)) == 0
    T, H, P, N = 256, 2, 16, 16
    inputs = 4 * (2 * T * H * P + T * H + 2 * T * N)      # x, dy, raw_dt, B, C (f32)
    outputs = 4 * (2 * T * H * P + T * H + 2 * T * N + H * P * N)
    assert n.value >= ws.value + inputs + outputs and n.value % 256 == 0
    h = ctypes.c_void_p(0x10000)
    dev = ctypes.c_void_p(0x40000)

    def call(device, nbytes, cu=None, prob=p):
        return lib.ssd_step_host(ctypes.byref(prob), h, h, h, h, cu, h, h, None, h, h, h, h,
                                 device, nbytes, None)
    assert call(None, n.value) == 4                       # no device region
    assert call(dev, n.value - 256) == 4                  # too small
    assert call(ctypes.c_void_p(0x40010), n.value) == 3   # not 256-byte aligned
    assert call(dev, n.value, cu=h) == 1                  # cu_seqlens for a dense batch
    assert call(dev, n.value, prob=_prob(headdim=12)) == 2


def test_profiler_filter_is_host_only(lib):
    """Setting or clearing the profiler's kernel filter touches no GPU state."""
    assert lib.ssd_profiler_only(b"tc_bwd_dxdb") == 0
    assert lib.ssd_profiler_only(None) == 0


def test_decode_step_host_checks(lib):
    """Host-side checks of ssd_decode_step (nothing is launched): seqlen must be 1, packed
    input is refused, overlapping distinct state buffers are refused, misaligned ones too."""
    p = _prob(seqlen=1, batch=3)
    a = ctypes.c_void_p(1 << 20)
    assert lib.ssd_decode_step(ctypes.byref(_prob(seqlen=2)), a, a, a, a, a, a, a, None) == 1
    assert lib.ssd_decode_step(ctypes.byref(_prob(seqlen=1, nseq=1)), a, a, a, a, a, a, a,
                               None) == 1
    # state_out starts 16 bytes into state_in: an overlap that is not in place
    assert lib.ssd_decode_step(ctypes.byref(p), a, ctypes.c_void_p((1 << 20) + 16), a, a, a, a,
                               a, None) == 1
    assert lib.ssd_decode_step(ctypes.byref(p), ctypes.c_void_p((1 << 20) + 4), a, a, a, a, a,
                               a, None) == 3
    assert lib.ssd_decode_step(ctypes.byref(p), None, a, a, a, a, a, a, None) == 1
