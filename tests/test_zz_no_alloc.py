"""ssd_forward_noalloc: the forward scan for callers that cannot allocate
device memory (a plugin whose host framework owns all device memory and
offers no workspace, or a latency-critical path where cudaMalloc/cudaFree are
not allowed).  It must give the same results as ssd_forward, call after call,
although every call reuses one library-owned scratch array.

This file is collected last on purpose, so that a run that stops at the first
failure has already run every other test.
"""

import ctypes
import os
import re

import numpy as np
import pytest

from helpers import TOL, rel_err, to_device, to_np

pytestmark = pytest.mark.gpu



def _scratch_bytes() -> int:
    """SSD_NOALLOC_SCRATCH_BYTES as include/ssd.h defines it."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    text = open(os.path.join(root, "include", "ssd.h")).read()
    m = re.search(r"#define\s+SSD_NOALLOC_SCRATCH_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)", text)
    assert m, "SSD_NOALLOC_SCRATCH_BYTES not found in ssd.h"
    return int(m.group(1)) << int(m.group(2))


SCRATCH_BYTES = _scratch_bytes()


@pytest.fixture(scope="module")
def ssd():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import state_space_model_ssd_gb300 as m
    from state_space_model_ssd_gb300 import build
    build.build()
    return m


def _draw(seed, bsz, L, H, P, N, dtype, cu=None):
    from state_space_model_ssd_gb300.inputs import bf16_round
    rng = np.random.default_rng(seed)
    rnd = bf16_round if dtype == "bf16" else (lambda a: a)
    return {
        "x": rnd(rng.standard_normal((bsz, L, H, P), dtype=np.float32)),
        "B": rnd(rng.standard_normal((bsz, L, 1, N), dtype=np.float32) / np.float32(np.sqrt(N))),
        "C": rnd(rng.standard_normal((bsz, L, 1, N), dtype=np.float32) / np.float32(np.sqrt(N))),
        "raw_dt": rng.standard_normal((bsz, L, H), dtype=np.float32) * np.float32(0.5),
        "cu_seqlens": None if cu is None else np.asarray(cu, dtype=np.int32),
    }


def _noalloc(ssd, t, dinit, Q=64):
    """One call of ssd_forward_noalloc through the C ABI; returns (status, y, final_state)."""
    import torch
    from state_space_model_ssd_gb300 import _lib
    prob = ssd.make_problem(t["x"], t["B"], dinit, Q, t["cu_seqlens"])
    nseq = prob.nseq if prob.nseq > 0 else prob.batch
    y = torch.full_like(t["x"], float("nan"))
    fs = torch.full((nseq, prob.nheads, prob.headdim, prob.dstate), float("nan"),
                    dtype=torch.float32, device=t["x"].device)
    cu = t["cu_seqlens"]
    st = _lib.lib().ssd_forward_noalloc(
        ctypes.byref(prob), t["x"].data_ptr(), t["raw_dt"].data_ptr(), t["B"].data_ptr(),
        t["C"].data_ptr(), None if cu is None else cu.data_ptr(), y.data_ptr(), fs.data_ptr(),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    return st, y, fs


CASES = [
    ("f32", dict(bsz=1, L=256, H=2, P=16, N=16)),
    ("bf16", dict(bsz=2, L=700, H=6, P=64, N=128)),
    ("bf16", dict(bsz=1, L=900, H=4, P=64, N=64, cu=[0, 1, 300, 364, 900])),
]


@pytest.mark.parametrize("dtype,shape", CASES)
def test_noalloc_matches_forward_on_consecutive_calls(ssd, dtype, shape):
    shape = dict(shape)
    cu = shape.pop("cu", None)
    d = _draw(21, dtype=dtype, cu=cu, **shape)
    t = to_device(d, dtype)
    y_ref, fs_ref = ssd.forward(t["x"], t["raw_dt"], t["B"], t["C"], delta_init=-4.6,
                                cu_seqlens=t["cu_seqlens"])
    y_ref, fs_ref = to_np(y_ref), to_np(fs_ref)
    for _ in range(2):
        st, y, fs = _noalloc(ssd, t, -4.6)
        assert st == 0
        assert rel_err(to_np(y), y_ref) <= TOL[dtype]
        assert rel_err(to_np(fs), fs_ref) <= TOL[dtype]


def test_noalloc_rejects_problems_beyond_its_scratch(ssd):
    import torch
    # the shortest power-of-two length whose forward workspace exceeds the scratch
    L = 1 << 10
    while True:
        x = torch.empty(1, L, 16, 64, dtype=torch.bfloat16, device="meta")
        B = torch.empty(1, L, 1, 128, dtype=torch.bfloat16, device="meta")
        if ssd.workspace_size(ssd.make_problem(x, B, -4.6), False) > SCRATCH_BYTES:
            break
        L *= 2
    x = torch.zeros(1, L, 16, 64, dtype=torch.bfloat16, device="cuda")
    B = torch.zeros(1, L, 1, 128, dtype=torch.bfloat16, device="cuda")
    raw = torch.zeros(1, L, 16, device="cuda")
    t = {"x": x, "B": B, "C": B, "raw_dt": raw, "cu_seqlens": None}
    st, y, _ = _noalloc(ssd, t, -4.6)
    assert st == 4  # SSD_ERR_WORKSPACE, nothing launched
    assert bool(torch.isnan(y[0, :4]).all())


def test_noalloc_reports_device_status(ssd):
    """A non-monotone cu_seqlens is caught on the device; the no-alloc path's status query
    reports it, and a following good call clears it."""
    import torch
    from state_space_model_ssd_gb300 import _lib
    d = _draw(23, 1, 100, 2, 16, 16, "f32", cu=[0, 60, 40, 100])
    t = to_device(d, "f32")
    st, _, _ = _noalloc(ssd, t, -4.6)
    assert st == 0
    v = ctypes.c_int32(-1)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert _lib.lib().ssd_forward_noalloc_status(stream, ctypes.byref(v)) == 0
    assert v.value == 7  # SSD_ERR_DEVICE
    t["cu_seqlens"] = torch.tensor([0, 40, 60, 100], dtype=torch.int32, device="cuda")
    st, _, _ = _noalloc(ssd, t, -4.6)
    assert st == 0
    assert _lib.lib().ssd_forward_noalloc_status(stream, ctypes.byref(v)) == 0
    assert v.value == 0
