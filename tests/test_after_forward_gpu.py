"""ssd_backward_after_forward: the backward that takes the forward's segment table,
C B^T tiles, chunk factors and segment states from the workspace must give the
results of ssd_backward (dx, d_raw_dt bit for bit; dB, dC up to the order of their
fp32 reduce-adds), keep the forward's device status, and refuse a workspace that
holds a forward of other inputs (device status SSD_ERR_WORKSPACE, no gradient)."""

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

SSD_ERR_WORKSPACE = 4


@pytest.fixture(scope="module")
def ssd():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import state_space_model_ssd_gb300 as m
    from state_space_model_ssd_gb300 import build
    build.build()
    return m


def _bits(t):
    import torch
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


def _ws(ssd, t, w):
    import torch
    prob = ssd.make_problem(t["x"], t["B"], w.delta_init, w.chunk_size, t["cu_seqlens"])
    n = max(ssd.workspace_size(prob, False), ssd.workspace_size(prob, True))
    return torch.empty(n, dtype=torch.uint8, device="cuda")


@pytest.mark.parametrize("name,tokens", [("mamba3_2x2048", None), ("varlen_64k", None),
                                         ("genomics_2m", 65536), ("tiny_f32", None)])
def test_matches_backward(ssd, name, tokens):
    import torch
    from helpers import to_device
    from state_space_model_ssd_gb300.inputs import WORKLOADS, make_inputs
    w = WORKLOADS[name]
    d = make_inputs(w, seed=5, with_dy=True, tokens=tokens)
    t = to_device(d, w.dtype)
    kw = dict(delta_init=w.delta_init, chunk_size=w.chunk_size, cu_seqlens=t["cu_seqlens"])
    ref = ssd.backward(t["x"], t["raw_dt"], t["B"], t["C"], t["dy"], **kw)
    ws = _ws(ssd, t, w)
    ssd.forward(t["x"], t["raw_dt"], t["B"], t["C"], workspace=ws, **kw)
    got = ssd.backward(t["x"], t["raw_dt"], t["B"], t["C"], t["dy"], workspace=ws,
                       after_forward=True, **kw)
    assert ssd.device_status(ws) == 0
    for k in ("dx", "d_raw_dt"):
        assert torch.equal(_bits(got[k]), _bits(ref[k])), k
    for k in ("dB", "dC"):
        a, b = got[k].float(), ref[k].float()
        assert float((a - b).abs().max()) <= 2 ** -6 * float(b.abs().max()), k


def test_refuses_other_inputs(ssd):
    import torch
    from helpers import to_device
    from state_space_model_ssd_gb300.inputs import WORKLOADS, make_inputs
    w = WORKLOADS["mamba3_2x2048"]
    d = make_inputs(w, seed=6, with_dy=True)
    t = to_device(d, w.dtype)
    kw = dict(delta_init=w.delta_init, chunk_size=w.chunk_size, cu_seqlens=t["cu_seqlens"])
    ws = _ws(ssd, t, w)
    ssd.forward(t["x"], t["raw_dt"], t["B"], t["C"], workspace=ws, **kw)
    x2 = t["x"].clone()  # same values, another buffer: not the forward's input
    out = ssd.backward(x2, t["raw_dt"], t["B"], t["C"], t["dy"], workspace=ws,
                       after_forward=True, **kw)
    assert ssd.device_status(ws) == SSD_ERR_WORKSPACE
    del out
    # a workspace that never saw a forward is refused the same way
    ws2 = _ws(ssd, t, w)
    ws2.zero_()
    ssd.backward(t["x"], t["raw_dt"], t["B"], t["C"], t["dy"], workspace=ws2,
                 after_forward=True, **kw)
    assert ssd.device_status(ws2) == SSD_ERR_WORKSPACE
