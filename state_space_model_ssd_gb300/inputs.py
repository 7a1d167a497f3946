"""Seeded synthetic workloads for the SSD scan.

This module only draws random numbers and rounds them to bf16; it holds none
of the scan's arithmetic.  Both the CUDA path (through ``bench.py`` and the GPU
tests) and the fp64 oracle read the tensors it returns, so the two sides see
bit-identical inputs.

Recipe (shared by every workload):

* ``numpy.random.default_rng(seed)``; draw order: sequence lengths (packed
  variable-length workloads only), X, B, C, raw_dt, dY.
* X ~ N(0, 1), B and C ~ N(0, 1) / sqrt(N), raw_dt ~ N(0, 0.5**2),
  dY ~ N(0, 1); all drawn as float32.
* For bf16 workloads X, B, C and dY are rounded to bf16 (round to nearest
  even) on the host; raw_dt stays float32.  Both consumers read the rounded
  values.
* Packed variable-length workloads draw lengths ``integers(lo, hi,
  endpoint=True)`` one at a time until they cover the total token count; the
  last one is cut so that the lengths sum to the total exactly.

The shapes follow the pages: the Mamba-3 constructor example (d_model 768,
d_state 128, headdim 64, bf16 input of shape (2, 2048, 768)) and mamba-2.8b's
d_model 2560 from "长序列 Mamba 多卡训练算力和显存怎么同时省" §三/§四; the
genomics row (16 heads, headdim 64, delta_init -5.0, 2M tokens) of the table in
"Mamba-2架构与LaCT并行计算技术解析" §3.2; chunk 64 from the same page 4 §三.
"""

from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

# Large draws are made in blocks so the float32 temporaries stay small.
_BLOCK = 1 << 24


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int           # rows of the dense batch (1 for packed input)
    seqlen: int          # tokens per row (total tokens for packed input)
    nheads: int
    headdim: int         # P
    dstate: int          # N
    chunk_size: int      # Q
    dtype: str           # "f32" or "bf16" for X, B, C, y and the gradients
    delta_init: float
    ngroups: int = 1
    varlen: Optional[tuple] = None   # (lo, hi) length range for packed input
    backward: bool = False

    @property
    def total_tokens(self) -> int:
        return self.batch * self.seqlen


WORKLOADS = {
    "tiny_f32": Workload("tiny_f32", 1, 256, 2, 16, 16, 64, "f32", -4.6),
    "mamba3_2x2048": Workload("mamba3_2x2048", 2, 2048, 24, 64, 128, 64, "bf16", -4.6),
    "mamba2.8b_32k": Workload("mamba2.8b_32k", 1, 32768, 80, 64, 128, 64, "bf16", -4.6,
                              backward=True),
    "varlen_64k": Workload("varlen_64k", 1, 65536, 24, 64, 128, 64, "bf16", -4.6,
                           varlen=(512, 8192), backward=True),
    "genomics_2m": Workload("genomics_2m", 1, 2097152, 16, 64, 64, 64, "bf16", -5.0),
}


def bf16_round(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); returns float32."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    bits = a.view(np.uint32)
    rounded = (bits + np.uint32(0x7FFF) + ((bits >> np.uint32(16)) & np.uint32(1))) \
        & np.uint32(0xFFFF0000)
    return rounded.view(np.float32)


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """The upper 16 bits of float32 values that are already bf16-representable."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    return (a.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def _normal(rng: np.random.Generator, shape, scale: float, bf16: bool) -> np.ndarray:
    out = np.empty(int(np.prod(shape)), dtype=np.float32)
    for lo in range(0, out.size, _BLOCK):
        hi = min(out.size, lo + _BLOCK)
        blk = rng.standard_normal(hi - lo, dtype=np.float32)
        if scale != 1.0:
            blk *= np.float32(scale)
        out[lo:hi] = bf16_round(blk) if bf16 else blk
    return out.reshape(shape)


def draw_lengths(rng: np.random.Generator, total: int, lo: int, hi: int) -> np.ndarray:
    lens = []
    acc = 0
    while acc < total:
        n = int(rng.integers(lo, hi, endpoint=True))
        n = min(n, total - acc)
        lens.append(n)
        acc += n
    return np.asarray(lens, dtype=np.int64)


def cu_from_lengths(lens) -> np.ndarray:
    cu = np.zeros(len(lens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(np.asarray(lens, dtype=np.int64))
    return cu


def make_inputs(w: Workload, seed: int = 0, with_dy: Optional[bool] = None,
                tokens: Optional[int] = None) -> dict:
    """Draw one workload.

    Returns a dict of float32 numpy arrays (bf16-representable for bf16
    workloads): ``x [batch, L, H, P]``, ``raw_dt [batch, L, H]``,
    ``B``/``C [batch, L, G, N]``, optionally ``dy`` like x, and ``cu_seqlens``
    (int32, ``None`` for a dense batch).  ``tokens`` overrides the row length
    (used to draw a smaller case with the same recipe).
    """
    rng = np.random.default_rng(seed)
    L = w.seqlen if tokens is None else int(tokens)
    bsz = w.batch
    cu = None
    if w.varlen is not None:
        lens = draw_lengths(rng, bsz * L, w.varlen[0], w.varlen[1])
        cu = cu_from_lengths(lens)
    bf16 = w.dtype == "bf16"
    H, P, N, G = w.nheads, w.headdim, w.dstate, w.ngroups
    out = {
        "x": _normal(rng, (bsz, L, H, P), 1.0, bf16),
        "B": _normal(rng, (bsz, L, G, N), 1.0 / np.sqrt(N), bf16),
        "C": _normal(rng, (bsz, L, G, N), 1.0 / np.sqrt(N), bf16),
        "raw_dt": _normal(rng, (bsz, L, H), 0.5, False),
        "cu_seqlens": cu,
    }
    if with_dy is None:
        with_dy = w.backward
    if with_dy:
        out["dy"] = _normal(rng, (bsz, L, H, P), 1.0, bf16)
    return out
