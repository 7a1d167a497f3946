"""GPU parity: the CUDA path against the fp64 oracle on identical seeded inputs.

Bar (per output tensor): max|gpu - oracle| / max|oracle| <= 1e-4 for fp32
inputs and <= 1e-2 for bf16 inputs (fp32 accumulation), gradients included.
Sizes here span several chunks and segments and end in a ragged tail; the
full-size workloads are checked in test_fullsize_gpu.py.
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


def _draw(seed, bsz, L, H, P, N, G=1, dtype="f32", cu=None, raw_shift=0.0):
    from state_space_model_ssd_gb300.inputs import bf16_round
    rng = np.random.default_rng(seed)
    rnd = (lambda a: bf16_round(a)) if dtype == "bf16" else (lambda a: a)
    d = {
        "x": rnd(rng.standard_normal((bsz, L, H, P), dtype=np.float32)),
        "B": rnd(rng.standard_normal((bsz, L, G, N), dtype=np.float32) / np.float32(np.sqrt(N))),
        "C": rnd(rng.standard_normal((bsz, L, G, N), dtype=np.float32) / np.float32(np.sqrt(N))),
        "raw_dt": (rng.standard_normal((bsz, L, H), dtype=np.float32) * np.float32(0.5)
                   + np.float32(raw_shift)),
        "dy": rnd(rng.standard_normal((bsz, L, H, P), dtype=np.float32)),
        "cu_seqlens": None if cu is None else np.asarray(cu, dtype=np.int32),
    }
    return d


def _fwd_check(ssd, oracle, d, dtype, dinit, Q=64, tol=None):
    tol = TOL[dtype] if tol is None else tol
    t = to_device(d, dtype)
    y, fs = ssd.forward(t["x"], t["raw_dt"], t["B"], t["C"], delta_init=dinit, chunk_size=Q,
                        cu_seqlens=t["cu_seqlens"])
    yr, fr = oracle.forward(d["x"], d["raw_dt"], d["B"], d["C"], dinit,
                            cu_seqlens=d["cu_seqlens"])
    ey, ef = rel_err(to_np(y), yr), rel_err(to_np(fs), fr)
    assert ey <= tol, "y rel err %g" % ey
    assert ef <= tol, "final_state rel err %g" % ef
    return to_np(y), to_np(fs)


def _bwd_check(ssd, oracle, d, dtype, dinit, Q=64, tol=None):
    tol = TOL[dtype] if tol is None else tol
    t = to_device(d, dtype)
    g = ssd.backward(t["x"], t["raw_dt"], t["B"], t["C"], t["dy"], delta_init=dinit,
                     chunk_size=Q, cu_seqlens=t["cu_seqlens"])
    r = oracle.backward(d["x"], d["raw_dt"], d["B"], d["C"], d["dy"], dinit,
                        cu_seqlens=d["cu_seqlens"])
    for k in ("dx", "d_raw_dt", "dB", "dC"):
        e = rel_err(to_np(g[k]), r[k])
        assert e <= tol, "%s rel err %g" % (k, e)


def test_tiny_f32_workload(ssd, oracle_mod):
    """The tiny fp32 workload exactly as specified (seeded recipe, seed 0)."""
    from state_space_model_ssd_gb300.inputs import WORKLOADS, make_inputs
    w = WORKLOADS["tiny_f32"]
    d = make_inputs(w, seed=0)
    _fwd_check(ssd, oracle_mod, d, "f32", w.delta_init)


@pytest.mark.parametrize("P,N", [(16, 16), (8, 128), (64, 64), (32, 8), (128, 32)])
def test_f32_forward_shapes(ssd, oracle_mod, P, N):
    d = _draw(1, 2, 333, 3, P, N)
    _fwd_check(ssd, oracle_mod, d, "f32", -4.6)


@pytest.mark.parametrize("P,N", [(16, 32), (64, 128)])
def test_f32_backward(ssd, oracle_mod, P, N):
    d = _draw(2, 1, 461, 3, P, N, raw_shift=1.0)
    _bwd_check(ssd, oracle_mod, d, "f32", -3.0)


@pytest.mark.parametrize("N", [64, 128])
def test_bf16_forward_backward(ssd, oracle_mod, N):
    d = _draw(3, 2, 650, 6, 64, N, dtype="bf16")
    _fwd_check(ssd, oracle_mod, d, "bf16", -4.6)
    _bwd_check(ssd, oracle_mod, d, "bf16", -4.6)


def test_bf16_larger_delta(ssd, oracle_mod):
    """delta ~ 0.13 per token (13x the workloads'): strong decay inside every chunk."""
    d = _draw(4, 1, 517, 4, 64, 128, dtype="bf16", raw_shift=2.0)
    _fwd_check(ssd, oracle_mod, d, "bf16", -4.0)
    _bwd_check(ssd, oracle_mod, d, "bf16", -4.0)


def test_bf16_very_large_delta(ssd, oracle_mod):
    """delta ~ 0.7 per token: the in-chunk terms of d_raw_dt dominate its sums."""
    d = _draw(4, 1, 517, 4, 64, 128, dtype="bf16", raw_shift=4.0)
    _fwd_check(ssd, oracle_mod, d, "bf16", -4.0)
    _bwd_check(ssd, oracle_mod, d, "bf16", -4.0)


def test_bf16_very_large_delta_long_segments(ssd, oracle_mod, monkeypatch):
    """delta ~ 0.7 per token with 16-chunk segments (the bench's segment length): the
    sums of d_raw_dt span a whole 1024-token segment."""
    monkeypatch.setenv("SSD_SEGMENT_CHUNKS", "16")
    d = _draw(14, 1, 2100, 2, 64, 128, dtype="bf16", raw_shift=4.0)
    _bwd_check(ssd, oracle_mod, d, "bf16", -4.0)


@pytest.mark.parametrize("N", [64, 128])
def test_bf16_memoryless_delta(ssd, oracle_mod, N):
    """delta ~ 4 per token (a chunk's delta sum ~ 250, beyond what the tensor-core
    factors carry): every work item runs the SIMT recurrence inside the tensor-core
    kernels, and the result is the oracle's, near its memoryless limit."""
    import torch
    d = _draw(15, 1, 700, 4, 64, N, dtype="bf16", raw_shift=8.0)
    t = to_device(d, "bf16")
    prob = ssd.make_problem(t["x"], t["B"], -4.0)
    assert ssd.dispatch_path(prob) == "tensor-core"
    ws = torch.empty(ssd.workspace_size(prob, True), dtype=torch.uint8, device="cuda")
    y, fs = ssd.forward(t["x"], t["raw_dt"], t["B"], t["C"], delta_init=-4.0, workspace=ws)
    assert ssd.device_status(ws) == 0
    yr, fr = oracle_mod.forward(d["x"], d["raw_dt"], d["B"], d["C"], -4.0)
    assert rel_err(to_np(y), yr) <= TOL["bf16"]
    assert rel_err(to_np(fs), fr) <= TOL["bf16"]
    g = ssd.backward(t["x"], t["raw_dt"], t["B"], t["C"], t["dy"], delta_init=-4.0,
                     workspace=ws, after_forward=True)
    assert ssd.device_status(ws) == 0
    r = oracle_mod.backward(d["x"], d["raw_dt"], d["B"], d["C"], d["dy"], -4.0)
    for k in ("dx", "d_raw_dt", "dB", "dC"):
        e = rel_err(to_np(g[k]), r[k])
        assert e <= TOL["bf16"], "%s rel err %g" % (k, e)


@pytest.mark.parametrize("packed", [False, True])
def test_bf16_mixed_delta_ranges(ssd, oracle_mod, monkeypatch, packed):
    """Heads 0-1 with delta ~ 4 everywhere, heads 2-3 with delta ~ 4 over tokens
    700..900 only, heads 4-5 at the workloads' delta: tensor-core and SIMT work items
    mix inside one call, across segments and in the head-summed dB / dC."""
    monkeypatch.setenv("SSD_SEGMENT_CHUNKS", "4")
    L, H = 1500, 6
    cu = [0, 300, 301, 1100, 1500] if packed else None
    d = _draw(16, 1, L, H, 64, 128, dtype="bf16", cu=cu)
    d["raw_dt"][:, :, 0:2] += np.float32(12.6)
    d["raw_dt"][:, 700:900, 2:4] += np.float32(12.6)
    _fwd_check(ssd, oracle_mod, d, "bf16", -4.6)
    _bwd_check(ssd, oracle_mod, d, "bf16", -4.6)


@pytest.mark.parametrize("dtype,P,N,H", [("f32", 16, 32, 3), ("bf16", 64, 128, 4),
                                         ("bf16", 64, 64, 2), ("bf16", 64, 128, 3)])
def test_packed_sequences(ssd, oracle_mod, dtype, P, N, H):
    lens = [1, 64, 130, 0, 257, 7, 128, 3, 1100, 65]
    cu = np.concatenate([[0], np.cumsum(lens)])
    d = _draw(5, 1, int(cu[-1]), H, P, N, dtype=dtype, cu=cu)
    _fwd_check(ssd, oracle_mod, d, dtype, -4.6)
    _bwd_check(ssd, oracle_mod, d, dtype, -4.6)


def test_groups(ssd, oracle_mod):
    d = _draw(6, 1, 300, 4, 16, 16, G=2)
    _fwd_check(ssd, oracle_mod, d, "f32", -2.0)
    _bwd_check(ssd, oracle_mod, d, "f32", -2.0)


def test_chunk_size_invariance(ssd, oracle_mod):
    """The chunked form is exact: every chunk length gives the oracle's result."""
    d = _draw(7, 1, 700, 2, 16, 32)
    ys = []
    for Q in (16, 32, 64, 128, 256):
        y, _ = _fwd_check(ssd, oracle_mod, d, "f32", -4.6, Q=Q)
        ys.append(y)
    for y in ys[1:]:
        assert rel_err(y, ys[0]) <= 1e-4


def test_single_token_and_exact_chunks(ssd, oracle_mod):
    for L in (1, 64, 128):
        d = _draw(8, 1, L, 2, 64, 64, dtype="bf16")
        _fwd_check(ssd, oracle_mod, d, "bf16", -4.6)
        _bwd_check(ssd, oracle_mod, d, "bf16", -4.6)


@pytest.mark.parametrize("N,H", [(64, 2), (128, 2), (64, 4)])
def test_single_token(ssd, oracle_mod, N, H):
    """One token: dB and dC are sums over heads of single terms delta_h (x_h . dy_h) C
    (or B), which for this draw nearly cancel at N = 64, H = 2."""
    d = _draw(8, 1, 1, H, 64, N, dtype="bf16")
    _fwd_check(ssd, oracle_mod, d, "bf16", -4.6)
    _bwd_check(ssd, oracle_mod, d, "bf16", -4.6)


@pytest.mark.parametrize("H,G,N,L,expect", [(2, 1, 128, 64, "tensor-core"),
                                             (24, 1, 64, 100, "tensor-core"),
                                             (3, 1, 128, 64, "tensor-core"),
                                             (6, 2, 64, 64, "tensor-core"),
                                             (2, 1, 128, 63, "simt"), (2, 1, 32, 64, "simt")])
def test_dispatch_path(ssd, H, G, N, L, expect):
    """bf16, P = 64, N in {64, 128}, chunk 64 and at least one chunk's worth of tokens take
    the tensor cores, with any number of heads per B/C group."""
    import torch
    x = torch.empty(1, L, H, 64, dtype=torch.bfloat16, device="cuda")
    B = torch.empty(1, L, G, N, dtype=torch.bfloat16, device="cuda")
    assert ssd.dispatch_path(ssd.make_problem(x, B, -4.6)) == expect


@pytest.mark.parametrize("H,G,N,packed", [(3, 1, 128, False), (6, 2, 64, False),
                                          (4, 2, 128, False), (5, 5, 64, False),
                                          (3, 1, 64, True), (6, 2, 128, True)])
def test_bf16_head_group_layouts(ssd, oracle_mod, monkeypatch, H, G, N, packed):
    """Tensor-core path with an odd number of heads per group (a group's last pair holds
    one head), several groups, and one head per group; 4-chunk segments, ragged tail."""
    monkeypatch.setenv("SSD_SEGMENT_CHUNKS", "4")
    cu = [0, 333, 334, 1000, 1300] if packed else None
    d = _draw(17, 1, 1300, H, 64, N, G=G, dtype="bf16", cu=cu)
    t = to_device(d, "bf16")
    assert ssd.dispatch_path(ssd.make_problem(t["x"], t["B"], -4.6)) == "tensor-core"
    _fwd_check(ssd, oracle_mod, d, "bf16", -4.6)
    _bwd_check(ssd, oracle_mod, d, "bf16", -4.6)


def test_long_segments_bf16(ssd, oracle_mod):
    """Several full 16-chunk segments per head plus a ragged tail (tensor-core path)."""
    d = _draw(12, 1, 4 * 1024 + 100, 2, 64, 128, dtype="bf16")
    _fwd_check(ssd, oracle_mod, d, "bf16", -4.6)


def test_empty_input(ssd):
    import torch
    x = torch.zeros(1, 0, 2, 16, device="cuda")
    B = torch.zeros(1, 0, 1, 16, device="cuda")
    y, fs = ssd.forward(x, torch.zeros(1, 0, 2, device="cuda"), B, B, delta_init=-4.6)
    assert y.shape == x.shape and torch.all(fs == 0)


def test_deterministic_forward(ssd):
    d = _draw(9, 1, 1000, 4, 64, 128, dtype="bf16")
    t = to_device(d, "bf16")
    y1, f1 = ssd.forward(t["x"], t["raw_dt"], t["B"], t["C"], delta_init=-4.6)
    y2, f2 = ssd.forward(t["x"], t["raw_dt"], t["B"], t["C"], delta_init=-4.6)
    assert bool((y1 == y2).all()) and bool((f1 == f2).all())


def test_output_base_16_byte_aligned(ssd):
    """y written through a base that is 16- but not 32-byte aligned (the walk then stores
    each 32-byte piece of a row as two 16-byte stores) equals y written to an aligned
    buffer, bit for bit."""
    import torch
    d = _draw(13, 1, 1000, 4, 64, 128, dtype="bf16")
    t = to_device(d, "bf16")
    y1, _ = ssd.forward(t["x"], t["raw_dt"], t["B"], t["C"], delta_init=-4.6)
    buf = torch.empty(t["x"].numel() + 8, dtype=torch.bfloat16, device="cuda")
    y2 = buf[8:].view(t["x"].shape)
    assert y2.data_ptr() % 32 == 16
    ssd.forward(t["x"], t["raw_dt"], t["B"], t["C"], delta_init=-4.6, out=y2)
    assert bool((y1 == y2).all())


def test_bad_cu_seqlens_reports_device_status(ssd):
    """A non-monotone cu_seqlens is caught on the device; the call returns, no hang."""
    import torch
    d = _draw(10, 1, 100, 2, 16, 16, cu=[0, 60, 40, 100])
    t = to_device(d, "f32")
    prob = ssd.make_problem(t["x"], t["B"], -4.6, 64, t["cu_seqlens"])
    ws = torch.empty(ssd.workspace_size(prob, False), dtype=torch.uint8, device="cuda")
    ssd.forward(t["x"], t["raw_dt"], t["B"], t["C"], delta_init=-4.6,
                cu_seqlens=t["cu_seqlens"], workspace=ws)
    assert ssd.device_status(ws) == 7
    good = torch.tensor([0, 40, 60, 100], dtype=torch.int32, device="cuda")
    ssd.forward(t["x"], t["raw_dt"], t["B"], t["C"], delta_init=-4.6, cu_seqlens=good,
                workspace=ws)
    assert ssd.device_status(ws) == 0


def test_launch_count_and_profiler(ssd):
    d = _draw(11, 1, 500, 2, 64, 128, dtype="bf16")
    t = to_device(d, "bf16")
    ssd.profiler.reset()
    ssd.profiler.enable(True)
    ssd.forward(t["x"], t["raw_dt"], t["B"], t["C"], delta_init=-4.6)
    n = ssd.last_launch_count()
    ssd.profiler.enable(False)
    prof = ssd.profiler.read()
    assert n >= 3
    assert sum(v[0] for v in prof.values()) == n
    assert all(v[1] > 0 for v in prof.values())


def test_profiler_only_times_the_named_kernel(ssd):
    """With a kernel name set, the profiler times that kernel's launches alone; with None
    it times every launch again."""
    d = _draw(11, 1, 500, 2, 64, 128, dtype="bf16")
    t = to_device(d, "bf16")
    try:
        ssd.profiler.only("tc_fwd_walk")
        ssd.profiler.reset()
        ssd.profiler.enable(True)
        for _ in range(2):
            ssd.forward(t["x"], t["raw_dt"], t["B"], t["C"], delta_init=-4.6)
        ssd.profiler.enable(False)
        prof = ssd.profiler.read()
        assert list(prof) == ["tc_fwd_walk"] and prof["tc_fwd_walk"][0] == 2
    finally:
        ssd.profiler.enable(False)
        ssd.profiler.only(None)
    ssd.profiler.reset()
    ssd.profiler.enable(True)
    ssd.forward(t["x"], t["raw_dt"], t["B"], t["C"], delta_init=-4.6)
    n = ssd.last_launch_count()
    ssd.profiler.enable(False)
    assert sum(v[0] for v in ssd.profiler.read().values()) == n


@pytest.mark.parametrize("dtype,P,N", [("f32", 16, 16), ("bf16", 64, 64)])
def test_many_short_sequences_with_empty_ones(ssd, oracle_mod, dtype, P, N):
    """1500 packed sequences of 0..4 tokens: every empty sequence's final state is zero
    (no segment writes it) and the rest match the oracle."""
    rng = np.random.default_rng(21)
    lens = rng.integers(0, 5, size=1500)
    lens[::5] = 0
    cu = np.concatenate([[0], np.cumsum(lens)])
    d = _draw(22, 1, int(cu[-1]), 2, P, N, dtype=dtype, cu=cu)
    t = to_device(d, dtype)
    y, fs = ssd.forward(t["x"], t["raw_dt"], t["B"], t["C"], delta_init=-4.6,
                        cu_seqlens=t["cu_seqlens"])
    yr, fr = oracle_mod.forward(d["x"], d["raw_dt"], d["B"], d["C"], -4.6,
                                cu_seqlens=d["cu_seqlens"])
    assert rel_err(to_np(y), yr) <= TOL[dtype]
    got = to_np(fs)
    assert np.all(got[lens == 0] == 0.0)
    assert rel_err(got, fr) <= TOL[dtype]
