"""Run-to-run determinism of the CUDA path: repeated calls on the same inputs must
give bit-identical y, final_state, dx and d_raw_dt (each is written by exactly one
thread, so any difference exposes a race between the warps of a kernel).  dB and dC
are summed over heads by reduce-adds in whatever order the segments finish, so they
are compared within a few bf16 units instead.

Inputs: the workload generators at full width, on enough tokens that every kernel
runs many waves of CTAs."""

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

REPEATS = 4


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


@pytest.mark.parametrize("name,tokens", [("genomics_2m", 524288), ("mamba2.8b_32k", None),
                                         ("varlen_64k", None)])
def test_repeatable(ssd, name, tokens):
    import torch
    from helpers import to_device
    from state_space_model_ssd_gb300.inputs import WORKLOADS, make_inputs
    w = WORKLOADS[name]
    d = make_inputs(w, seed=3, with_dy=True, tokens=tokens)
    t = to_device(d, w.dtype)
    kw = dict(delta_init=w.delta_init, chunk_size=w.chunk_size, cu_seqlens=t["cu_seqlens"])
    y0, f0 = ssd.forward(t["x"], t["raw_dt"], t["B"], t["C"], **kw)
    g0 = ssd.backward(t["x"], t["raw_dt"], t["B"], t["C"], t["dy"], **kw)
    for _ in range(REPEATS):
        y, f = ssd.forward(t["x"], t["raw_dt"], t["B"], t["C"], **kw)
        assert torch.equal(_bits(y), _bits(y0)), "y differs between runs"
        assert torch.equal(_bits(f), _bits(f0)), "final_state differs between runs"
        g = ssd.backward(t["x"], t["raw_dt"], t["B"], t["C"], t["dy"], **kw)
        for k in ("dx", "d_raw_dt"):
            assert torch.equal(_bits(g[k]), _bits(g0[k])), "%s differs between runs" % k
        for k in ("dB", "dC"):
            a, b = g[k].float(), g0[k].float()
            # order of the fp32 reduce-adds: at most a couple of bf16 rounding steps
            assert float((a - b).abs().max()) <= 2 ** -6 * float(b.abs().max()), k
