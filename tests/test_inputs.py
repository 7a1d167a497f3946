"""The seeded input generator: bf16 rounding and the packed-length recipe."""

import numpy as np
import torch

from state_space_model_ssd_gb300 import inputs


def test_bf16_round_matches_torch():
    rng = np.random.default_rng(0)
    a = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 3,
                        np.array([0.0, -0.0, 1.0, 1.00390625, 1.01171875, 65504.0, 1e-30],
                                 dtype=np.float32)])
    ref = torch.from_numpy(a).to(torch.bfloat16).float().numpy()
    np.testing.assert_array_equal(inputs.bf16_round(a), ref)
    bits = inputs.bf16_bits(inputs.bf16_round(a))
    np.testing.assert_array_equal(bits, torch.from_numpy(ref).to(torch.bfloat16).view(torch.int16)
                                  .numpy().view(np.uint16))


def test_packed_lengths_recipe():
    w = inputs.WORKLOADS["varlen_64k"]
    d = inputs.make_inputs(w, seed=0, with_dy=False, tokens=65536)
    cu = d["cu_seqlens"]
    lens = np.diff(cu)
    assert cu[0] == 0 and cu[-1] == 65536
    assert np.all(lens[:-1] >= 512) and np.all(lens <= 8192) and lens[-1] >= 1
    assert d["x"].shape == (1, 65536, 24, 64)


def test_deterministic_and_bf16_representable():
    w = inputs.WORKLOADS["mamba3_2x2048"]
    a = inputs.make_inputs(w, seed=0, tokens=64, with_dy=True)
    b = inputs.make_inputs(w, seed=0, tokens=64, with_dy=True)
    for k in ("x", "B", "C", "raw_dt", "dy"):
        np.testing.assert_array_equal(a[k], b[k])
    for k in ("x", "B", "C", "dy"):
        np.testing.assert_array_equal(inputs.bf16_round(a[k]), a[k])
    assert a["x"].shape == (2, 64, 24, 64) and a["B"].shape == (2, 64, 1, 128)
    assert abs(np.std(a["raw_dt"]) - 0.5) < 0.05
