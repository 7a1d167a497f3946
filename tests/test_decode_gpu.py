"""Single-token decode step on the GPU (ssd_decode_step through the C ABI): one token of
the recurrence of page "Mamba-2架构与LaCT并行计算技术解析" §1.1 from a carried state,
against the fp64 oracle run on that one token from the same initial state, and a run of
decode steps against the chunked forward over the same tokens."""

import numpy as np
import pytest

from helpers import TOL, rel_err, to_np

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


def _draw(seed, bsz, L, H, P, N, G, dtype):
    from state_space_model_ssd_gb300.inputs import bf16_round
    rng = np.random.default_rng(seed)
    rnd = bf16_round if dtype == "bf16" else (lambda a: a)
    return {
        "x": rnd(rng.standard_normal((bsz, L, H, P), dtype=np.float32)),
        "B": rnd(rng.standard_normal((bsz, L, G, N), dtype=np.float32) / np.float32(np.sqrt(N))),
        "C": rnd(rng.standard_normal((bsz, L, G, N), dtype=np.float32) / np.float32(np.sqrt(N))),
        "raw_dt": rng.standard_normal((bsz, L, H), dtype=np.float32) * np.float32(0.5),
        "h0": rng.standard_normal((bsz, H, P, N), dtype=np.float32) * np.float32(0.5),
    }


def _dev(a, dtype):
    import torch
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    return torch.from_numpy(np.ascontiguousarray(a)).cuda().to(tdt)


@pytest.mark.parametrize("dtype,H,P,N,G", [("bf16", 6, 64, 128, 1), ("f32", 4, 16, 32, 2),
                                           ("f32", 2, 128, 8, 1), ("bf16", 8, 32, 64, 4)])
def test_one_step_matches_oracle(ssd, oracle_mod, dtype, H, P, N, G):
    import torch
    d = _draw(41, 5, 1, H, P, N, G, dtype)
    state = torch.from_numpy(d["h0"]).cuda()
    y, s2 = ssd.decode_step(state, _dev(d["x"][:, 0], dtype), torch.from_numpy(
        np.ascontiguousarray(d["raw_dt"][:, 0])).cuda(), _dev(d["B"][:, 0], dtype),
        _dev(d["C"][:, 0], dtype), -4.6, state_out=torch.empty_like(state))
    yr, fr = oracle_mod.forward(d["x"], d["raw_dt"], d["B"], d["C"], -4.6, initial_state=d["h0"])
    assert rel_err(to_np(y), yr[:, 0]) <= TOL[dtype]
    assert rel_err(to_np(s2), fr) <= 1e-5  # the state itself stays fp32


def test_in_place_equals_out_of_place(ssd):
    import torch
    d = _draw(42, 3, 1, 4, 64, 128, 1, "bf16")
    args = (_dev(d["x"][:, 0], "bf16"),
            torch.from_numpy(np.ascontiguousarray(d["raw_dt"][:, 0])).cuda(),
            _dev(d["B"][:, 0], "bf16"), _dev(d["C"][:, 0], "bf16"), -4.6)
    s_a = torch.from_numpy(d["h0"]).cuda()
    y_a, out_a = ssd.decode_step(s_a, *args, state_out=torch.empty_like(s_a))
    s_b = torch.from_numpy(d["h0"]).cuda()
    y_b, out_b = ssd.decode_step(s_b, *args)
    assert out_b.data_ptr() == s_b.data_ptr()
    assert bool((y_a == y_b).all()) and bool((out_a == out_b).all())


@pytest.mark.parametrize("dtype,H,P,N", [("bf16", 4, 64, 128), ("f32", 2, 16, 16)])
def test_decode_loop_matches_forward(ssd, oracle_mod, dtype, H, P, N):
    """T decode steps from an initial state reproduce the chunked forward's y and final
    state over the same T tokens (and the oracle's)."""
    import torch
    T = 150
    d = _draw(43, 2, T, H, P, N, 1, dtype)
    x, B, C = _dev(d["x"], dtype), _dev(d["B"], dtype), _dev(d["C"], dtype)
    raw = torch.from_numpy(d["raw_dt"]).cuda()
    h0 = torch.from_numpy(d["h0"]).cuda()
    yf, ff = ssd.forward(x, raw, B, C, delta_init=-4.6, initial_state=h0)
    state = h0.clone()
    ys = []
    for t in range(T):
        yt, _ = ssd.decode_step(state, x[:, t].contiguous(), raw[:, t].contiguous(),
                                B[:, t].contiguous(), C[:, t].contiguous(), -4.6)
        ys.append(yt)
    yd = torch.stack(ys, 1)
    yr, fr = oracle_mod.forward(d["x"], d["raw_dt"], d["B"], d["C"], -4.6, initial_state=d["h0"])
    assert rel_err(to_np(yd), yr) <= TOL[dtype]
    assert rel_err(to_np(state), fr) <= TOL[dtype]
    assert rel_err(to_np(yd), to_np(yf)) <= TOL[dtype]
    assert rel_err(to_np(state), to_np(ff)) <= TOL[dtype]
