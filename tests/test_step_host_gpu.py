"""ssd_step_host (host buffers in and out) gives the results of ssd_forward +
ssd_backward_after_forward on the same inputs in device memory."""

import numpy as np
import pytest

from helpers import rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ssd():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import state_space_model_ssd_gb300 as m
    from state_space_model_ssd_gb300 import build
    build.build()
    return m


def _inputs(seed, L, H, P, N, dtype, cu=None):
    import torch
    g = torch.Generator().manual_seed(seed)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    host = {
        "x": torch.randn(1, L, H, P, generator=g).to(tdt),
        "B": (torch.randn(1, L, 1, N, generator=g) / N ** 0.5).to(tdt),
        "C": (torch.randn(1, L, 1, N, generator=g) / N ** 0.5).to(tdt),
        "raw_dt": torch.randn(1, L, H, generator=g) * 0.5,
        "dy": torch.randn(1, L, H, P, generator=g).to(tdt),
    }
    host = {k: v.pin_memory() for k, v in host.items()}
    cu_h = None if cu is None else torch.tensor(cu, dtype=torch.int32)
    return host, cu_h


def _device_reference(ssd, host, cu_h, dinit):
    import torch
    dv = {k: v.cuda() for k, v in host.items()}
    cu = None if cu_h is None else cu_h.cuda()
    prob = ssd.make_problem(dv["x"], dv["B"], dinit, 64, cu)
    ws = torch.empty(ssd.workspace_size(prob, True), dtype=torch.uint8, device="cuda")
    y, fs = ssd.forward(dv["x"], dv["raw_dt"], dv["B"], dv["C"], dinit, cu_seqlens=cu,
                        workspace=ws)
    g = ssd.backward(dv["x"], dv["raw_dt"], dv["B"], dv["C"], dv["dy"], dinit, cu_seqlens=cu,
                     workspace=ws, after_forward=True)
    torch.cuda.synchronize()
    return {"y": y.cpu(), "final_state": fs.cpu(), **{k: v.cpu() for k, v in g.items()}}


@pytest.mark.parametrize("dtype,L,H,P,N,cu", [
    ("bf16", 1000, 4, 64, 128, None),                 # tensor-core path
    ("bf16", 1500, 2, 64, 64, [0, 700, 701, 1500]),   # tensor-core path, packed sequences
    ("f32", 600, 3, 16, 32, [0, 250, 600]),           # SIMT path
])
def test_step_host_matches_device_calls(ssd, dtype, L, H, P, N, cu):
    import torch
    host, cu_h = _inputs(7, L, H, P, N, dtype, cu)
    ref = _device_reference(ssd, host, cu_h, -4.6)
    s = torch.cuda.Stream()
    out = ssd.step_host(host["x"], host["raw_dt"], host["B"], host["C"], host["dy"], -4.6,
                        cu_seqlens=cu_h, stream=s)
    s.synchronize()
    for k in ("y", "final_state", "dx", "d_raw_dt"):
        assert torch.equal(out[k], ref[k]), k
    # dB and dC are summed over head pairs in completion order: equal up to a rounding step
    for k in ("dB", "dC"):
        assert rel_err(out[k].float().numpy(), ref[k].float().numpy()) <= 2.0 ** -6, k


def test_step_host_forward_only_and_two_streams(ssd):
    """dy = None runs the forward alone; two calls on two streams with two device buffers
    (the pipelined use) both give the reference results."""
    import torch
    host, _ = _inputs(8, 900, 4, 64, 128, "bf16")
    ref = _device_reference(ssd, host, None, -4.6)
    out = ssd.step_host(host["x"], host["raw_dt"], host["B"], host["C"], None, -4.6)
    torch.cuda.synchronize()
    assert out["dx"] is None and torch.equal(out["y"], ref["y"])
    assert torch.equal(out["final_state"], ref["final_state"])
    prob = ssd.make_problem(host["x"], host["B"], -4.6, 64, None)
    bufs = [torch.empty(ssd.step_host_size(prob), dtype=torch.uint8, device="cuda")
            for _ in range(2)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = [ssd.step_host(host["x"], host["raw_dt"], host["B"], host["C"], host["dy"], -4.6,
                          device_buffer=bufs[i], stream=streams[i]) for i in range(2)]
    torch.cuda.synchronize()
    for o in outs:
        assert torch.equal(o["y"], ref["y"]) and torch.equal(o["dx"], ref["dx"])
        assert torch.equal(o["d_raw_dt"], ref["d_raw_dt"])
    assert ssd.device_status(bufs[0]) == 0 and ssd.device_status(bufs[1]) == 0
