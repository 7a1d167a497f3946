"""fp64 CPU oracle of the SSD selective-state recurrence (ctypes wrapper).

TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT: only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference leg may
import this package.  It shares no code with the CUDA library; the recurrence
lives in ``ssd_oracle.c`` (see its header for the equations and their source,
page "Mamba-2架构与LaCT并行计算技术解析" §1.1).

Arrays use the framework's layouts: ``x [batch, L, H, P]``, ``raw_dt
[batch, L, H]``, ``B``/``C [batch, L, G, N]``; with ``cu_seqlens`` the batch
must be 1 and the tokens are packed sequences.  Everything is computed in
fp64 from the given values (bf16 inputs are passed as their exact float
values).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssd_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ssd_oracle.c into oracle/_build/liboracle.so with gcc + OpenMP."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".%d.tmp" % os.getpid()
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        dp = ctypes.POINTER(ctypes.c_double)
        lp = ctypes.POINTER(ctypes.c_int64)
        lib.ssd_oracle_forward.restype = ctypes.c_int
        lib.ssd_oracle_forward.argtypes = [
            ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            lp, dp, dp, dp, dp, ctypes.c_double, dp, dp, dp, ctypes.c_int]
        lib.ssd_oracle_backward.restype = ctypes.c_int
        lib.ssd_oracle_backward.argtypes = [
            ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            lp, dp, dp, dp, dp, ctypes.c_double, dp, dp, dp, dp, dp, dp, dp, dp, ctypes.c_int]
        lib.ssd_oracle_softplus.restype = ctypes.c_double
        lib.ssd_oracle_softplus.argtypes = [ctypes.c_double]
        lib.ssd_oracle_max_threads.restype = ctypes.c_int
        lib.ssd_oracle_max_threads.argtypes = []
        _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a: Optional[np.ndarray]):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _problem(x, raw_dt, B, C, cu_seqlens):
    x = np.asarray(x)
    if x.ndim != 4:
        raise ValueError("x must be [batch, L, H, P]")
    bsz, L, H, P = x.shape
    G, N = np.asarray(B).shape[-2:]
    T = bsz * L
    if cu_seqlens is None:
        cu = np.arange(bsz + 1, dtype=np.int64) * L
    else:
        if bsz != 1:
            raise ValueError("packed sequences need batch == 1")
        cu = np.ascontiguousarray(cu_seqlens, dtype=np.int64)
    return bsz, L, H, P, G, N, T, cu


def softplus(z: float) -> float:
    return float(_load().ssd_oracle_softplus(float(z)))


def max_threads() -> int:
    return int(_load().ssd_oracle_max_threads())


def forward(x, raw_dt, B, C, delta_init: float, cu_seqlens=None, initial_state=None,
            threads: int = 0):
    """Returns ``(y [batch, L, H, P], final_state [nseq, H, P, N])`` in fp64."""
    bsz, L, H, P, G, N, T, cu = _problem(x, raw_dt, B, C, cu_seqlens)
    nseq = len(cu) - 1
    xf, rf, bf, cf = _f64(x), _f64(raw_dt), _f64(B), _f64(C)
    h0 = None if initial_state is None else _f64(initial_state)
    if h0 is not None and h0.size != nseq * H * P * N:
        raise ValueError("initial_state must be [nseq, H, P, N]")
    y = np.zeros((bsz, L, H, P), dtype=np.float64)
    hT = np.zeros((nseq, H, P, N), dtype=np.float64)
    rc = _load().ssd_oracle_forward(
        T, H, P, N, G, nseq, cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
        _ptr(xf), _ptr(rf), _ptr(bf), _ptr(cf), float(delta_init), _ptr(h0), _ptr(y), _ptr(hT),
        int(threads))
    if rc != 0:
        raise ValueError("oracle forward rejected its arguments (code %d)" % rc)
    return y, hT


def backward(x, raw_dt, B, C, dy, delta_init: float, cu_seqlens=None, initial_state=None,
             d_final_state=None, threads: int = 0):
    """Returns a dict with ``dx, d_raw_dt, dB, dC, d_initial_state`` (fp64)."""
    bsz, L, H, P, G, N, T, cu = _problem(x, raw_dt, B, C, cu_seqlens)
    nseq = len(cu) - 1
    xf, rf, bf, cf, dyf = _f64(x), _f64(raw_dt), _f64(B), _f64(C), _f64(dy)
    h0 = None if initial_state is None else _f64(initial_state)
    dhT = None if d_final_state is None else _f64(d_final_state)
    dx = np.zeros((bsz, L, H, P), dtype=np.float64)
    draw = np.zeros((bsz, L, H), dtype=np.float64)
    dB = np.zeros((bsz, L, G, N), dtype=np.float64)
    dC = np.zeros((bsz, L, G, N), dtype=np.float64)
    dh0 = np.zeros((nseq, H, P, N), dtype=np.float64)
    rc = _load().ssd_oracle_backward(
        T, H, P, N, G, nseq, cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
        _ptr(xf), _ptr(rf), _ptr(bf), _ptr(cf), float(delta_init), _ptr(h0), _ptr(dyf),
        _ptr(dhT), _ptr(dx), _ptr(draw), _ptr(dB), _ptr(dC), _ptr(dh0), int(threads))
    if rc != 0:
        raise ValueError("oracle backward failed (code %d)" % rc)
    return {"dx": dx, "d_raw_dt": draw, "dB": dB, "dC": dC, "d_initial_state": dh0}


def _flip_sequences(a, cu_seqlens):
    """Each sequence of a [batch, L, ...] array reversed along its token axis (dense rows,
    or the packed sequences of cu_seqlens)."""
    a = np.asarray(a)
    if cu_seqlens is None:
        return np.ascontiguousarray(a[:, ::-1])
    out = np.empty_like(a)
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    for s in range(len(cu) - 1):
        out[:, cu[s]:cu[s + 1]] = a[:, cu[s]:cu[s + 1]][:, ::-1]
    return out


def bidirectional_forward(x, raw_dt, B, C, delta_init: float, cu_seqlens=None, threads: int = 0):
    """Bidirectional mode (page "Mamba-2架构与LaCT并行计算技术解析" §3.1): the scan over
    each sequence and over the sequence reversed, the reverse direction's outputs put back
    at their tokens' positions, concatenated along the last dimension.  Both directions
    read the same x, raw_dt, B, C.  Returns ``(y [batch, L, H, 2P], final_state_forward,
    final_state_reverse)`` in fp64."""
    fl = lambda a: _flip_sequences(a, cu_seqlens)  # noqa: E731
    yf, ff = forward(x, raw_dt, B, C, delta_init, cu_seqlens=cu_seqlens, threads=threads)
    yr, fr = forward(fl(x), fl(raw_dt), fl(B), fl(C), delta_init, cu_seqlens=cu_seqlens,
                     threads=threads)
    return np.concatenate([yf, fl(yr)], axis=-1), ff, fr


def bidirectional_backward(x, raw_dt, B, C, dy, delta_init: float, cu_seqlens=None,
                           threads: int = 0):
    """Gradients of sum(dy * y) for y = bidirectional_forward(...)[0], dy [batch, L, H, 2P]:
    each input's gradient is the forward direction's plus the reverse direction's put back
    at its tokens' positions."""
    fl = lambda a: _flip_sequences(a, cu_seqlens)  # noqa: E731
    P = np.asarray(x).shape[-1]
    dy = np.asarray(dy)
    gf = backward(x, raw_dt, B, C, dy[..., :P], delta_init, cu_seqlens=cu_seqlens, threads=threads)
    gr = backward(fl(x), fl(raw_dt), fl(B), fl(C), fl(dy[..., P:]), delta_init,
                  cu_seqlens=cu_seqlens, threads=threads)
    return {k: gf[k] + fl(gr[k]) for k in ("dx", "d_raw_dt", "dB", "dC")}
