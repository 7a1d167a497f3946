"""Full-size workloads on the GPU, compared element by element with the oracle over
whole tensors: every head and every token of y, final_state and (where the workload
has a backward) dx, d_raw_dt, dB and dC.

The GPU side runs each workload whole, in the launch configuration bench.py times.
The oracle runs on the same seeded inputs on the host's cores; at 2M tokens it runs
four heads at a time (heads are independent), which bounds its host memory.
Bar: max|gpu - oracle| / max|oracle| <= 1e-2 (bf16 inputs) per tensor.
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


def _check(got, ref, name, tol):
    e = rel_err(got, ref)
    assert e <= tol, "%s rel err %g" % (name, e)


def _check_all(ssd, oracle_mod, name):
    """Whole workload on the GPU; whole tensors against the oracle on the same inputs."""
    from state_space_model_ssd_gb300.inputs import WORKLOADS, make_inputs
    w = WORKLOADS[name]
    d = make_inputs(w, seed=0)
    out = _run(ssd, d, w, backward=w.backward)
    y, fs = oracle_mod.forward(d["x"], d["raw_dt"], d["B"], d["C"], w.delta_init,
                               cu_seqlens=d["cu_seqlens"])
    _check(out["y"], y, "y", TOL[w.dtype])
    _check(out["final_state"], fs, "final_state", TOL[w.dtype])
    del y, fs
    if w.backward:
        g = oracle_mod.backward(d["x"], d["raw_dt"], d["B"], d["C"], d["dy"], w.delta_init,
                                cu_seqlens=d["cu_seqlens"])
        for k in ("dx", "d_raw_dt", "dB", "dC"):
            _check(out[k], g[k], k, TOL[w.dtype])


def test_mamba3_example_shape(ssd, oracle_mod):
    """Mamba-3 constructor example: 2 x 2048 tokens, 24 heads, P=64, N=128 (forward)."""
    _check_all(ssd, oracle_mod, "mamba3_2x2048")


def test_mamba28b_layer_32k(ssd, oracle_mod):
    """mamba-2.8b layer: L=32768, 80 heads, P=64, N=128, forward and backward."""
    _check_all(ssd, oracle_mod, "mamba2.8b_32k")


def test_varlen_packed_64k(ssd, oracle_mod):
    """65536 packed tokens, lengths in [512, 8192], 24 heads, forward and backward."""
    _check_all(ssd, oracle_mod, "varlen_64k")


def test_genomics_2m(ssd, oracle_mod):
    """2,097,152 tokens, 16 heads, P=N=64, delta_init -5.0, forward with final_state:
    every head, compared four heads at a time."""
    import torch
    from state_space_model_ssd_gb300.inputs import WORKLOADS, make_inputs
    w = WORKLOADS["genomics_2m"]
    d = make_inputs(w, seed=0)
    t = to_device(d, w.dtype)
    y, fs = ssd.forward(t["x"], t["raw_dt"], t["B"], t["C"], delta_init=w.delta_init,
                        chunk_size=w.chunk_size)
    del t
    torch.cuda.synchronize()
    num = {"y": 0.0, "final_state": 0.0}
    den = {"y": 0.0, "final_state": 0.0}
    for h0 in range(0, w.nheads, 4):
        hs = slice(h0, h0 + 4)
        sub = {k: np.ascontiguousarray(d[k][:, :, hs]) for k in ("x", "raw_dt")}
        yr, fr = oracle_mod.forward(sub["x"], sub["raw_dt"], d["B"], d["C"], w.delta_init)
        yg = y[:, :, hs].float().cpu().numpy()
        fg = fs[:, hs].float().cpu().numpy()
        for k, got, ref in (("y", yg, yr), ("final_state", fg, fr)):
            num[k] = max(num[k], float(np.max(np.abs(got.astype(np.float64) - ref))))
            den[k] = max(den[k], float(np.max(np.abs(ref))))
        del yr, fr, yg, fg, sub
    for k in num:
        e = num[k] / den[k]
        assert e <= TOL[w.dtype], "%s rel err %g (all heads)" % (k, e)


def _check_all_states(ssd, oracle_mod, name):
    """The workload with an initial state per sequence and an upstream final-state
    gradient: every output and gradient, d_initial_state included, over whole tensors."""
    import torch
    from state_space_model_ssd_gb300.inputs import WORKLOADS, make_inputs
    w = WORKLOADS[name]
    d = make_inputs(w, seed=0)
    nseq = w.batch if d["cu_seqlens"] is None else len(d["cu_seqlens"]) - 1
    rng = np.random.default_rng(1)
    shape = (nseq, w.nheads, w.headdim, w.dstate)
    h0 = rng.standard_normal(shape, dtype=np.float32) * np.float32(0.5)
    dhT = rng.standard_normal(shape, dtype=np.float32)
    t = to_device(d, w.dtype)
    th0, tdhT = torch.from_numpy(h0).cuda(), torch.from_numpy(dhT).cuda()
    y, fs = ssd.forward(t["x"], t["raw_dt"], t["B"], t["C"], delta_init=w.delta_init,
                        cu_seqlens=t["cu_seqlens"], initial_state=th0)
    g = ssd.backward(t["x"], t["raw_dt"], t["B"], t["C"], t["dy"], delta_init=w.delta_init,
                     cu_seqlens=t["cu_seqlens"], initial_state=th0, d_final_state=tdhT,
                     d_initial_state=True)
    out = {"y": to_np(y), "final_state": to_np(fs)}
    out.update({k: to_np(v) for k, v in g.items()})
    del t, y, fs, g
    torch.cuda.empty_cache()
    yr, fr = oracle_mod.forward(d["x"], d["raw_dt"], d["B"], d["C"], w.delta_init,
                                cu_seqlens=d["cu_seqlens"], initial_state=h0)
    _check(out["y"], yr, "y", TOL[w.dtype])
    _check(out["final_state"], fr, "final_state", TOL[w.dtype])
    del yr, fr
    r = oracle_mod.backward(d["x"], d["raw_dt"], d["B"], d["C"], d["dy"], w.delta_init,
                            cu_seqlens=d["cu_seqlens"], initial_state=h0, d_final_state=dhT)
    for k in ("dx", "d_raw_dt", "dB", "dC", "d_initial_state"):
        _check(out[k], r[k], k, TOL[w.dtype])


def test_mamba28b_layer_32k_with_states(ssd, oracle_mod):
    """mamba-2.8b layer at L=32768 with initial state and final-state gradient."""
    _check_all_states(ssd, oracle_mod, "mamba2.8b_32k")


def test_varlen_packed_64k_with_states(ssd, oracle_mod):
    """65536 packed tokens, 24 heads, with initial states and final-state gradients."""
    _check_all_states(ssd, oracle_mod, "varlen_64k")
