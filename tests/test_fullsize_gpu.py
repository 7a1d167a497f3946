"""Full-size workloads on the GPU, checked against the oracle on outputs it can
compute exactly at that size:

* heads are independent, so y, final_state, dx and d_raw_dt of a few sampled heads
  over the whole sequence come from the oracle run on those heads alone;
* dC_t = sum_h H_t^T dy_t depends only on tokens <= t, so dC on a prefix of the
  sequence comes from the oracle run on that prefix (all heads);
* dB_t and dx_t depend only on tokens >= t (the upstream gradient of the final
  state is zero), so dB and dx on a suffix come from the oracle run on that suffix;
* packed sequences are independent runs, so whole sequences of a packed batch come
  from the oracle run on each sequence.

The GPU side always runs the whole workload in the launch configuration bench.py
times.  Bar: max|gpu - oracle| / max|oracle| <= 1e-2 (bf16) per checked tensor.
"""

import numpy as np
import pytest

from helpers import TOL, rel_err, to_device, to_np

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


def _run(ssd, d, w, backward):
    import torch
    t = to_device(d, w.dtype)
    y, fs = ssd.forward(t["x"], t["raw_dt"], t["B"], t["C"], delta_init=w.delta_init,
                        chunk_size=w.chunk_size, cu_seqlens=t["cu_seqlens"])
    out = {"y": to_np(y), "final_state": to_np(fs)}
    if backward:
        g = ssd.backward(t["x"], t["raw_dt"], t["B"], t["C"], t["dy"], delta_init=w.delta_init,
                         chunk_size=w.chunk_size, cu_seqlens=t["cu_seqlens"])
        out.update({k: to_np(v) for k, v in g.items()})
    del t
    torch.cuda.empty_cache()
    return out


def _heads(d, hs):
    return {k: (None if v is None else (np.ascontiguousarray(v[:, :, hs])
                                        if k in ("x", "raw_dt", "dy") else v))
            for k, v in d.items()}


def _span(d, a, b):
    return {k: (None if (v is None or k == "cu_seqlens") else np.ascontiguousarray(v[:, a:b]))
            for k, v in d.items()}


def _check(got, ref, name, tol):
    e = rel_err(got, ref)
    assert e <= tol, "%s rel err %g" % (name, e)


def test_mamba3_example_shape(ssd, oracle_mod):
    """Mamba-3 constructor example: 2 x 2048 tokens, 24 heads, P=64, N=128 (all outputs)."""
    from state_space_model_ssd_gb300.inputs import WORKLOADS, make_inputs
    w = WORKLOADS["mamba3_2x2048"]
    d = make_inputs(w, seed=0)
    out = _run(ssd, d, w, backward=False)
    y, fs = oracle_mod.forward(d["x"], d["raw_dt"], d["B"], d["C"], w.delta_init)
    _check(out["y"], y, "y", TOL["bf16"])
    _check(out["final_state"], fs, "final_state", TOL["bf16"])


def test_mamba28b_layer_32k(ssd, oracle_mod):
    """mamba-2.8b layer: L=32768, 80 heads, P=64, N=128, forward and backward."""
    from state_space_model_ssd_gb300.inputs import WORKLOADS, make_inputs
    w = WORKLOADS["mamba2.8b_32k"]
    d = make_inputs(w, seed=0)
    out = _run(ssd, d, w, backward=True)
    hs = [0, 37, 79]
    sub = _heads(d, hs)
    y, fs = oracle_mod.forward(sub["x"], sub["raw_dt"], sub["B"], sub["C"], w.delta_init)
    _check(out["y"][:, :, hs], y, "y (sampled heads)", TOL["bf16"])
    _check(out["final_state"][:, hs], fs, "final_state (sampled heads)", TOL["bf16"])
    g = oracle_mod.backward(sub["x"], sub["raw_dt"], sub["B"], sub["C"], sub["dy"], w.delta_init)
    _check(out["dx"][:, :, hs], g["dx"], "dx (sampled heads)", TOL["bf16"])
    _check(out["d_raw_dt"][:, :, hs], g["d_raw_dt"], "d_raw_dt (sampled heads)", TOL["bf16"])
    W = 1536
    pre = _span(d, 0, W)
    gp = oracle_mod.backward(pre["x"], pre["raw_dt"], pre["B"], pre["C"], pre["dy"], w.delta_init)
    _check(out["dC"][:, :W], gp["dC"], "dC (prefix)", TOL["bf16"])
    T = w.seqlen
    suf = _span(d, T - W, T)
    gs = oracle_mod.backward(suf["x"], suf["raw_dt"], suf["B"], suf["C"], suf["dy"], w.delta_init)
    _check(out["dB"][:, T - W:], gs["dB"], "dB (suffix)", TOL["bf16"])
    _check(out["dx"][:, T - W:], gs["dx"], "dx (suffix, all heads)", TOL["bf16"])


def test_varlen_packed_64k(ssd, oracle_mod):
    """65536 packed tokens, lengths in [512, 8192], 24 heads: whole sequences checked."""
    from state_space_model_ssd_gb300.inputs import WORKLOADS, make_inputs
    w = WORKLOADS["varlen_64k"]
    d = make_inputs(w, seed=0)
    out = _run(ssd, d, w, backward=True)
    cu = d["cu_seqlens"]
    for s in (0, 1, len(cu) - 2):
        a, b = int(cu[s]), int(cu[s + 1])
        one = _span(d, a, b)
        y, fs = oracle_mod.forward(one["x"], one["raw_dt"], one["B"], one["C"], w.delta_init)
        _check(out["y"][:, a:b], y, "y (sequence %d)" % s, TOL["bf16"])
        _check(out["final_state"][s], fs[0], "final_state (sequence %d)" % s, TOL["bf16"])
        g = oracle_mod.backward(one["x"], one["raw_dt"], one["B"], one["C"], one["dy"],
                                w.delta_init)
        for k in ("dx", "d_raw_dt", "dB", "dC"):
            _check(out[k][:, a:b], g[k], "%s (sequence %d)" % (k, s), TOL["bf16"])


def test_genomics_2m(ssd, oracle_mod):
    """2,097,152 tokens, 16 heads, P=N=64, delta_init -5.0, forward with final_state."""
    from state_space_model_ssd_gb300.inputs import WORKLOADS, make_inputs
    w = WORKLOADS["genomics_2m"]
    d = make_inputs(w, seed=0)
    out = _run(ssd, d, w, backward=False)
    hs = [0, 11]
    sub = _heads(d, hs)
    y, fs = oracle_mod.forward(sub["x"], sub["raw_dt"], sub["B"], sub["C"], w.delta_init)
    _check(out["y"][:, :, hs], y, "y (sampled heads)", TOL["bf16"])
    _check(out["final_state"][:, hs], fs, "final_state (sampled heads)", TOL["bf16"])
    W = 4096
    pre = _span(d, 0, W)
    yp, _ = oracle_mod.forward(pre["x"], pre["raw_dt"], pre["B"], pre["C"], w.delta_init)
    _check(out["y"][:, :W], yp, "y (prefix, all heads)", TOL["bf16"])
