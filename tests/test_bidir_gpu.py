"""Bidirectional mode on the GPU (page "Mamba-2架构与LaCT并行计算技术解析" §3.1) against
the oracle's bidirectional forward and backward on the same seeded inputs: the output
[T][H][2P] (forward direction | reverse direction at the original positions), both final
states, and the gradients summed over the two directions."""

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


def _draw(seed, bsz, L, H, P, N, dtype, cu=None):
    from state_space_model_ssd_gb300.inputs import bf16_round
    rng = np.random.default_rng(seed)
    rnd = bf16_round if dtype == "bf16" else (lambda a: a)
    return {
        "x": rnd(rng.standard_normal((bsz, L, H, P), dtype=np.float32)),
        "B": rnd(rng.standard_normal((bsz, L, 1, N), dtype=np.float32) / np.float32(np.sqrt(N))),
        "C": rnd(rng.standard_normal((bsz, L, 1, N), dtype=np.float32) / np.float32(np.sqrt(N))),
        "raw_dt": rng.standard_normal((bsz, L, H), dtype=np.float32) * np.float32(0.5),
        "dy": rnd(rng.standard_normal((bsz, L, H, 2 * P), dtype=np.float32)),
        "cu_seqlens": None if cu is None else np.asarray(cu, dtype=np.int32),
    }


@pytest.mark.parametrize("dtype,bsz,L,H,P,N,lens", [
    ("bf16", 2, 700, 4, 64, 128, None),
    ("bf16", 1, 0, 2, 64, 64, [300, 0, 1, 640, 65]),
    ("f32", 1, 0, 3, 16, 32, [200, 7, 0, 333]),
    ("f32", 2, 129, 2, 8, 16, None),
])
def test_bidirectional_matches_oracle(ssd, oracle_mod, dtype, bsz, L, H, P, N, lens):
    import torch
    cu = None
    if lens is not None:
        cu = np.concatenate([[0], np.cumsum(lens)])
        L = int(cu[-1])
    d = _draw(51, bsz, L, H, P, N, dtype, cu)
    t = to_device(d, dtype)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    dy = torch.from_numpy(d["dy"]).cuda().to(tdt)
    y, ff, fr = ssd.bidirectional_forward(t["x"], t["raw_dt"], t["B"], t["C"], delta_init=-4.6,
                                          cu_seqlens=t["cu_seqlens"])
    yr, ffr, frr = oracle_mod.bidirectional_forward(d["x"], d["raw_dt"], d["B"], d["C"], -4.6,
                                                    cu_seqlens=d["cu_seqlens"])
    tol = TOL[dtype]
    assert rel_err(to_np(y), yr) <= tol
    assert rel_err(to_np(ff), ffr) <= tol
    assert rel_err(to_np(fr), frr) <= tol
    g = ssd.bidirectional_backward(t["x"], t["raw_dt"], t["B"], t["C"], dy, delta_init=-4.6,
                                   cu_seqlens=t["cu_seqlens"])
    r = oracle_mod.bidirectional_backward(d["x"], d["raw_dt"], d["B"], d["C"], d["dy"], -4.6,
                                          cu_seqlens=d["cu_seqlens"])
    for k in ("dx", "d_raw_dt", "dB", "dC"):
        e = rel_err(to_np(g[k]), r[k])
        assert e <= tol, "%s rel err %g" % (k, e)
