"""Initial state in, gradients of the initial and final states out, on the GPU, against
the fp64 oracle on the same seeded inputs (page "Mamba-2架构与LaCT并行计算技术解析"
§1.1: H may start from a carried-over state).  Bar: max|gpu - oracle| / max|oracle|
<= 1e-4 (fp32 inputs) or 1e-2 (bf16 inputs) per tensor, d_initial_state included.
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


def _draw(seed, L, H, P, N, dtype, cu=None, bsz=1, raw_shift=0.0):
    from state_space_model_ssd_gb300.inputs import bf16_round
    rng = np.random.default_rng(seed)
    rnd = bf16_round if dtype == "bf16" else (lambda a: a)
    nseq = bsz if cu is None else len(cu) - 1
    return {
        "x": rnd(rng.standard_normal((bsz, L, H, P), dtype=np.float32)),
        "B": rnd(rng.standard_normal((bsz, L, 1, N), dtype=np.float32) / np.float32(np.sqrt(N))),
        "C": rnd(rng.standard_normal((bsz, L, 1, N), dtype=np.float32) / np.float32(np.sqrt(N))),
        "raw_dt": rng.standard_normal((bsz, L, H), dtype=np.float32) * np.float32(0.5)
        + np.float32(raw_shift),
        "dy": rnd(rng.standard_normal((bsz, L, H, P), dtype=np.float32)),
        "h0": rng.standard_normal((nseq, H, P, N), dtype=np.float32) * np.float32(0.5),
        "dhT": rng.standard_normal((nseq, H, P, N), dtype=np.float32),
        "cu_seqlens": None if cu is None else np.asarray(cu, dtype=np.int32),
    }


def _check_all(ssd, oracle, d, dtype, dinit, after_forward=False):
    import torch
    t = to_device(d, dtype)
    h0 = torch.from_numpy(d["h0"]).cuda()
    dhT = torch.from_numpy(d["dhT"]).cuda()
    prob = ssd.make_problem(t["x"], t["B"], dinit, 64, t["cu_seqlens"])
    ws = torch.empty(ssd.workspace_size(prob, True), dtype=torch.uint8, device="cuda")
    y, fs = ssd.forward(t["x"], t["raw_dt"], t["B"], t["C"], delta_init=dinit,
                        cu_seqlens=t["cu_seqlens"], initial_state=h0, workspace=ws)
    yr, fr = oracle.forward(d["x"], d["raw_dt"], d["B"], d["C"], dinit,
                            cu_seqlens=d["cu_seqlens"], initial_state=d["h0"])
    tol = TOL[dtype]
    assert rel_err(to_np(y), yr) <= tol, "y"
    assert rel_err(to_np(fs), fr) <= tol, "final_state"
    g = ssd.backward(t["x"], t["raw_dt"], t["B"], t["C"], t["dy"], delta_init=dinit,
                     cu_seqlens=t["cu_seqlens"], initial_state=h0, d_final_state=dhT,
                     d_initial_state=True, workspace=ws, after_forward=after_forward)
    assert ssd.device_status(ws) == 0
    r = oracle.backward(d["x"], d["raw_dt"], d["B"], d["C"], d["dy"], dinit,
                        cu_seqlens=d["cu_seqlens"], initial_state=d["h0"],
                        d_final_state=d["dhT"])
    for k in ("dx", "d_raw_dt", "dB", "dC", "d_initial_state"):
        e = rel_err(to_np(g[k]), r[k])
        assert e <= tol, "%s rel err %g" % (k, e)
    return to_np(fs), g


def test_f32_dense_batch(ssd, oracle_mod):
    """SIMT path (fp32), two dense rows, several segments each."""
    d = _draw(31, 333, 3, 16, 32, "f32", bsz=2)
    _check_all(ssd, oracle_mod, d, "f32", -3.0)


@pytest.mark.parametrize("after_forward", [False, True])
@pytest.mark.parametrize("N", [64, 128])
def test_bf16_multi_segment(ssd, oracle_mod, monkeypatch, N, after_forward):
    """Tensor-core path, 4-chunk segments: the initial state enters the first segment's
    walk, the final-state gradient the last segment's adjoint and boundary term."""
    monkeypatch.setenv("SSD_SEGMENT_CHUNKS", "4")
    d = _draw(32, 1500, 4, 64, N, "bf16")
    _check_all(ssd, oracle_mod, d, "bf16", -4.6, after_forward=after_forward)


@pytest.mark.parametrize("dtype,P,N,H", [("f32", 16, 16, 2), ("bf16", 64, 128, 4)])
def test_packed_with_empty_sequences(ssd, oracle_mod, dtype, P, N, H):
    """Packed sequences, two of them empty: an empty sequence's final state is its initial
    state and its d_initial_state its d_final_state."""
    lens = [130, 0, 257, 1, 0, 700]
    cu = np.concatenate([[0], np.cumsum(lens)])
    d = _draw(33, int(cu[-1]), H, P, N, dtype, cu=cu)
    fs, g = _check_all(ssd, oracle_mod, d, dtype, -4.6)
    for s in (1, 4):
        assert np.array_equal(fs[s], d["h0"][s])
        assert np.array_equal(to_np(g["d_initial_state"])[s], d["dhT"][s])


def test_bf16_large_delta_items(ssd, oracle_mod, monkeypatch):
    """Heads 0-1 with delta ~ 8 (the SIMT recurrence inside the tensor-core kernels) and
    heads 2-3 at the workloads' delta, both with initial state and final-state gradient."""
    monkeypatch.setenv("SSD_SEGMENT_CHUNKS", "4")
    d = _draw(34, 900, 4, 64, 128, "bf16")
    d["raw_dt"][:, :, 0:2] += np.float32(12.6)
    _check_all(ssd, oracle_mod, d, "bf16", -4.6)


def test_split_and_continue(ssd):
    """Running the first part, then the rest from its final state, gives the whole run's
    outputs (the carried-over state), on the tensor-core path."""
    import torch
    d = _draw(35, 2000, 4, 64, 128, "bf16")
    t = to_device(d, "bf16")
    y, fs = ssd.forward(t["x"], t["raw_dt"], t["B"], t["C"], delta_init=-4.6)
    k = 1216
    part = {n: t[n][:, :k].contiguous() for n in ("x", "raw_dt", "B", "C")}
    rest = {n: t[n][:, k:].contiguous() for n in ("x", "raw_dt", "B", "C")}
    y1, f1 = ssd.forward(part["x"], part["raw_dt"], part["B"], part["C"], delta_init=-4.6)
    y2, f2 = ssd.forward(rest["x"], rest["raw_dt"], rest["B"], rest["C"], delta_init=-4.6,
                         initial_state=f1)
    assert rel_err(to_np(torch.cat([y1, y2], 1)), to_np(y)) <= TOL["bf16"]
    assert rel_err(to_np(f2), to_np(fs)) <= TOL["bf16"]


@pytest.mark.parametrize("dtype,P,N,H", [("f32", 16, 16, 2), ("bf16", 64, 64, 2)])
def test_many_segments_blocked_scans(ssd, oracle_mod, monkeypatch, dtype, P, N, H):
    """More than 128 segments (one chunk each): the scans over segments run as block
    summaries, a pass over the blocks and per-block scans, with sequences starting inside
    blocks, initial states and final-state gradients."""
    monkeypatch.setenv("SSD_SEGMENT_CHUNKS", "1")
    lens = [3000, 64, 1, 4100, 700, 0, 2000]
    cu = np.concatenate([[0], np.cumsum(lens)])
    d = _draw(36, int(cu[-1]), H, P, N, dtype, cu=cu)
    _check_all(ssd, oracle_mod, d, dtype, -4.6)


@pytest.mark.parametrize("N", [64, 128])
@pytest.mark.parametrize("k", [33, 64])
def test_bf16_long_segments(ssd, oracle_mod, monkeypatch, k, N):
    """Segments of 33 and 64 chunks (the longest the aggregate kernels take) on the
    tensor-core path (at N = 64 the two-CTA-per-SM forward walk), a ragged last segment,
    head 0 at delta ~ 8 (its head pair takes the SIMT recurrence), with initial state and
    final-state gradient."""
    monkeypatch.setenv("SSD_SEGMENT_CHUNKS", str(k))
    d = _draw(37, 9000, 4, 64, N, "bf16")
    d["raw_dt"][:, :, 0] += np.float32(12.6)
    _check_all(ssd, oracle_mod, d, "bf16", -4.6)


def test_f32_long_segments(ssd, oracle_mod, monkeypatch):
    """64-chunk segments on the SIMT path (fp32), two rows."""
    monkeypatch.setenv("SSD_SEGMENT_CHUNKS", "64")
    d = _draw(38, 5000, 2, 16, 16, "f32", bsz=2)
    _check_all(ssd, oracle_mod, d, "f32", -3.0)
