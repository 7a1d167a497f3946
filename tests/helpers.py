"""Shared helpers for the GPU parity tests: move seeded inputs to the GPU, run
the oracle on the same values, and measure max|a - ref| / max|ref|."""

import numpy as np

TOL = {"f32": 1e-4, "bf16": 1e-2}


def rel_err(a, ref) -> float:
    a = np.asarray(a, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    scale = float(np.max(np.abs(ref))) if ref.size else 0.0
    if ref.size == 0:
        return 0.0
    diff = float(np.max(np.abs(a - ref)))
    return diff / scale if scale > 0 else diff


def to_device(d, dtype_name, device="cuda"):
    import torch
    tdt = torch.bfloat16 if dtype_name == "bf16" else torch.float32
    out = {}
    for k in ("x", "B", "C", "dy"):
        if k in d:
            out[k] = torch.from_numpy(np.ascontiguousarray(d[k])).to(device=device, dtype=tdt)
    out["raw_dt"] = torch.from_numpy(np.ascontiguousarray(d["raw_dt"])).to(device)
    cu = d.get("cu_seqlens")
    out["cu_seqlens"] = None if cu is None else torch.from_numpy(cu.astype(np.int32)).to(device)
    return out


def to_np(t):
    return t.detach().float().cpu().numpy()
