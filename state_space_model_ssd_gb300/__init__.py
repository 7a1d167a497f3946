"""GB300 SSD selective-state scan: a thin Python binding over libssd.so.

Every step of the scan runs in the library's CUDA kernels; this module only
marshals arguments (shapes, dtypes, device pointers, the current CUDA stream)
and allocates outputs and workspace with torch.  There is no CPU fallback: a
missing library or a non-CUDA tensor raises.

    y, final_state = forward(x, raw_dt, B, C, delta_init=-4.6)
    grads = backward(x, raw_dt, B, C, dy, delta_init=-4.6)

Layouts: x, y, dy, dx ``[batch, L, H, P]``; raw_dt ``[batch, L, H]`` float32;
B, C ``[batch, L, G, N]``; with ``cu_seqlens`` (int32, ``[nseq + 1]``) the batch
is 1 and the tokens are packed sequences.
"""

from __future__ import annotations

import ctypes
from typing import Optional

from . import _lib
from ._lib import SSDError, check

__all__ = ["forward", "backward", "bidirectional_forward", "bidirectional_backward", "decode_step", "step_host", "step_host_size", "workspace_size",
           "dispatch_path", "make_problem", "last_launch_count", "profiler", "SSDError"]


def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.float32:
        return _lib.DTYPE_F32
    if t.dtype == torch.bfloat16:
        return _lib.DTYPE_BF16
    raise TypeError("x/B/C must be float32 or bfloat16, got %s" % t.dtype)


def make_problem(x, B, delta_init: float, chunk_size: int = 64, cu_seqlens=None) -> _lib.Problem:
    if x.dim() != 4 or B.dim() != 4:
        raise ValueError("x must be [batch, L, H, P] and B [batch, L, G, N]")
    bsz, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    nseq = 0
    if cu_seqlens is not None:
        if bsz != 1:
            raise ValueError("packed sequences need batch == 1")
        nseq = cu_seqlens.numel() - 1
    return _lib.Problem(bsz, L, H, P, N, G, int(chunk_size), nseq, float(delta_init),
                        _dtype_code(x))


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _check_tensor(t, name, dtype=None, device=None):
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if device is not None and t.device != device:
        raise ValueError("%s is on %s, expected %s" % (name, t.device, device))


def workspace_size(problem: _lib.Problem, for_backward: bool) -> int:
    n = ctypes.c_size_t(0)
    check(_lib.lib().ssd_workspace_size(ctypes.byref(problem), int(for_backward),
                                        ctypes.byref(n)), "ssd_workspace_size")
    return int(n.value)


def dispatch_path(problem: _lib.Problem, for_backward: bool = False) -> Optional[str]:
    r = _lib.lib().ssd_dispatch_path(ctypes.byref(problem), int(for_backward))
    return None if r is None else r.decode()


def last_launch_count() -> int:
    return int(_lib.lib().ssd_last_launch_count())


def _workspace(nbytes: int, device, workspace=None):
    torch = _torch()
    if workspace is not None:
        if workspace.numel() * workspace.element_size() < nbytes:
            raise ValueError("workspace too small: need %d bytes" % nbytes)
        return workspace
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def _stream(stream):
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def forward(x, raw_dt, B, C, delta_init: float, chunk_size: int = 64, cu_seqlens=None,
            final_state: bool = True, out=None, workspace=None, stream=None,
            final_state_out=None, initial_state=None):
    """Runs ssd_forward (ssd_forward_state with ``initial_state``, a float32
    ``[nseq, H, P, N]`` CUDA tensor).  Returns ``(y, final_state or None)``;
    ``final_state_out`` (float32 ``[nseq, H, P, N]``) receives the final states when given."""
    torch = _torch()
    dev = x.device
    _check_tensor(x, "x")
    _check_tensor(raw_dt, "raw_dt", torch.float32, dev)
    _check_tensor(B, "B", x.dtype, dev)
    _check_tensor(C, "C", x.dtype, dev)
    if cu_seqlens is not None:
        _check_tensor(cu_seqlens, "cu_seqlens", torch.int32, dev)
    prob = make_problem(x, B, delta_init, chunk_size, cu_seqlens)
    nseq = prob.nseq if prob.nseq > 0 else prob.batch
    y = torch.empty_like(x) if out is None else out
    fs = None
    if final_state_out is not None:
        _check_tensor(final_state_out, "final_state_out", torch.float32, dev)
        if tuple(final_state_out.shape) != (nseq, prob.nheads, prob.headdim, prob.dstate):
            raise ValueError("final_state_out must be [nseq, H, P, N]")
        fs = final_state_out
    elif final_state:
        fs = torch.empty((nseq, prob.nheads, prob.headdim, prob.dstate), dtype=torch.float32,
                         device=dev)
    if initial_state is not None:
        _check_tensor(initial_state, "initial_state", torch.float32, dev)
        if tuple(initial_state.shape) != (nseq, prob.nheads, prob.headdim, prob.dstate):
            raise ValueError("initial_state must be [nseq, H, P, N]")
    ws = _workspace(workspace_size(prob, False), dev, workspace)
    with torch.cuda.device(dev):
        st = _lib.lib().ssd_forward_state(ctypes.byref(prob), _ptr(x), _ptr(raw_dt), _ptr(B),
                                          _ptr(C), _ptr(cu_seqlens), _ptr(initial_state),
                                          _ptr(y), _ptr(fs), _ptr(ws), ws.numel(),
                                          _stream(stream))
    check(st, "ssd_forward_state")
    return y, fs


def backward(x, raw_dt, B, C, dy, delta_init: float, chunk_size: int = 64, cu_seqlens=None,
             out=None, workspace=None, stream=None, after_forward: bool = False,
             initial_state=None, d_final_state=None, d_initial_state: bool = False):
    """Runs ssd_backward_state (ssd_backward with no initial state and a zero final-state
    gradient).  ``after_forward``: the workspace holds the preceding forward on these
    inputs.  ``initial_state`` / ``d_final_state``: float32 ``[nseq, H, P, N]`` CUDA tensors
    or None.  Returns a dict ``dx, d_raw_dt, dB, dC`` and, with ``d_initial_state``,
    ``d_initial_state``."""
    torch = _torch()
    dev = x.device
    _check_tensor(x, "x")
    _check_tensor(raw_dt, "raw_dt", torch.float32, dev)
    _check_tensor(B, "B", x.dtype, dev)
    _check_tensor(C, "C", x.dtype, dev)
    _check_tensor(dy, "dy", x.dtype, dev)
    if cu_seqlens is not None:
        _check_tensor(cu_seqlens, "cu_seqlens", torch.int32, dev)
    prob = make_problem(x, B, delta_init, chunk_size, cu_seqlens)
    if out is None:
        out = {"dx": torch.empty_like(x), "d_raw_dt": torch.empty_like(raw_dt),
               "dB": torch.empty_like(B), "dC": torch.empty_like(C)}
    if after_forward and workspace is None:
        raise ValueError("after_forward needs the forward's workspace")
    nseq = prob.nseq if prob.nseq > 0 else prob.batch
    shape = (nseq, prob.nheads, prob.headdim, prob.dstate)
    for t, name in ((initial_state, "initial_state"), (d_final_state, "d_final_state")):
        if t is not None:
            _check_tensor(t, name, torch.float32, dev)
            if tuple(t.shape) != shape:
                raise ValueError("%s must be [nseq, H, P, N]" % name)
    if d_initial_state and "d_initial_state" not in out:
        out["d_initial_state"] = torch.empty(shape, dtype=torch.float32, device=dev)
    ws = _workspace(workspace_size(prob, True), dev, workspace)
    with torch.cuda.device(dev):
        st = _lib.lib().ssd_backward_state(
            ctypes.byref(prob), _ptr(x), _ptr(raw_dt), _ptr(B), _ptr(C), _ptr(cu_seqlens),
            _ptr(initial_state), _ptr(dy), _ptr(d_final_state), _ptr(out["dx"]),
            _ptr(out["d_raw_dt"]), _ptr(out["dB"]), _ptr(out["dC"]),
            _ptr(out.get("d_initial_state") if d_initial_state else None), int(after_forward),
            _ptr(ws), ws.numel(), _stream(stream))
    check(st, "ssd_backward_state")
    return out


def bidirectional_workspace_size(problem: _lib.Problem, for_backward: bool) -> int:
    n = ctypes.c_size_t(0)
    check(_lib.lib().ssd_bidirectional_workspace_size(ctypes.byref(problem), int(for_backward),
                                                      ctypes.byref(n)),
          "ssd_bidirectional_workspace_size")
    return int(n.value)


def bidirectional_forward(x, raw_dt, B, C, delta_init: float, chunk_size: int = 64,
                          cu_seqlens=None, final_state: bool = True, workspace=None,
                          stream=None):
    """Runs ssd_bidirectional_forward.  Returns ``(y [batch, L, H, 2P], final state of the
    forward direction, final state of the reverse direction)`` (None without final_state)."""
    torch = _torch()
    dev = x.device
    for t, n in ((x, "x"), (B, "B"), (C, "C")):
        _check_tensor(t, n)
    _check_tensor(raw_dt, "raw_dt", torch.float32, dev)
    if cu_seqlens is not None:
        _check_tensor(cu_seqlens, "cu_seqlens", torch.int32, dev)
    prob = make_problem(x, B, delta_init, chunk_size, cu_seqlens)
    nseq = prob.nseq if prob.nseq > 0 else prob.batch
    y = torch.empty(x.shape[:-1] + (2 * x.shape[-1],), dtype=x.dtype, device=dev)
    fs = [None, None]
    if final_state:
        fs = [torch.empty((nseq, prob.nheads, prob.headdim, prob.dstate), dtype=torch.float32,
                          device=dev) for _ in range(2)]
    ws = _workspace(bidirectional_workspace_size(prob, False), dev, workspace)
    with torch.cuda.device(dev):
        st = _lib.lib().ssd_bidirectional_forward(
            ctypes.byref(prob), _ptr(x), _ptr(raw_dt), _ptr(B), _ptr(C), _ptr(cu_seqlens),
            _ptr(y), _ptr(fs[0]), _ptr(fs[1]), _ptr(ws), ws.numel(), _stream(stream))
    check(st, "ssd_bidirectional_forward")
    return y, fs[0], fs[1]


def bidirectional_backward(x, raw_dt, B, C, dy, delta_init: float, chunk_size: int = 64,
                           cu_seqlens=None, workspace=None, stream=None):
    """Runs ssd_bidirectional_backward for dy ``[batch, L, H, 2P]``.  Returns a dict
    ``dx, d_raw_dt, dB, dC``."""
    torch = _torch()
    dev = x.device
    for t, n in ((x, "x"), (B, "B"), (C, "C"), (dy, "dy")):
        _check_tensor(t, n)
    _check_tensor(raw_dt, "raw_dt", torch.float32, dev)
    if tuple(dy.shape) != tuple(x.shape[:-1]) + (2 * x.shape[-1],) or dy.dtype != x.dtype:
        raise ValueError("dy must be [batch, L, H, 2P] in the dtype of x")
    if cu_seqlens is not None:
        _check_tensor(cu_seqlens, "cu_seqlens", torch.int32, dev)
    prob = make_problem(x, B, delta_init, chunk_size, cu_seqlens)
    out = {"dx": torch.empty_like(x), "d_raw_dt": torch.empty_like(raw_dt),
           "dB": torch.empty_like(B), "dC": torch.empty_like(C)}
    ws = _workspace(bidirectional_workspace_size(prob, True), dev, workspace)
    with torch.cuda.device(dev):
        st = _lib.lib().ssd_bidirectional_backward(
            ctypes.byref(prob), _ptr(x), _ptr(raw_dt), _ptr(B), _ptr(C), _ptr(cu_seqlens),
            _ptr(dy), _ptr(out["dx"]), _ptr(out["d_raw_dt"]), _ptr(out["dB"]), _ptr(out["dC"]),
            _ptr(ws), ws.numel(), _stream(stream))
    check(st, "ssd_bidirectional_backward")
    return out


def decode_step(state, x, raw_dt, B, C, delta_init: float, out=None, state_out=None,
                stream=None):
    """Runs ssd_decode_step for one token of every sequence of a batch: ``state``
    float32 ``[batch, H, P, N]`` (updated in place unless ``state_out`` is given), ``x``
    ``[batch, H, P]``, ``raw_dt`` float32 ``[batch, H]``, ``B``/``C`` ``[batch, G, N]``.
    Returns ``(y [batch, H, P], new state)``."""
    torch = _torch()
    dev = x.device
    _check_tensor(state, "state", torch.float32, dev)
    _check_tensor(x, "x")
    _check_tensor(raw_dt, "raw_dt", torch.float32, dev)
    _check_tensor(B, "B", x.dtype, dev)
    _check_tensor(C, "C", x.dtype, dev)
    if x.dim() != 3 or B.dim() != 3 or state.dim() != 4:
        raise ValueError("x must be [batch, H, P], B/C [batch, G, N], state [batch, H, P, N]")
    prob = make_problem(x.unsqueeze(1), B.unsqueeze(1), delta_init, 64)
    if tuple(state.shape) != (prob.batch, prob.nheads, prob.headdim, prob.dstate):
        raise ValueError("state must be [batch, H, P, N]")
    so = state if state_out is None else state_out
    y = torch.empty_like(x) if out is None else out
    with torch.cuda.device(dev):
        st = _lib.lib().ssd_decode_step(ctypes.byref(prob), _ptr(state), _ptr(so), _ptr(x),
                                        _ptr(raw_dt), _ptr(B), _ptr(C), _ptr(y),
                                        _stream(stream))
    check(st, "ssd_decode_step")
    return y, so


def step_host_size(problem: _lib.Problem) -> int:
    n = ctypes.c_size_t(0)
    check(_lib.lib().ssd_step_host_size(ctypes.byref(problem), ctypes.byref(n)),
          "ssd_step_host_size")
    return int(n.value)


def step_host(x, raw_dt, B, C, dy, delta_init: float, chunk_size: int = 64, cu_seqlens=None,
              final_state: bool = True, out=None, device_buffer=None, stream=None):
    """Runs ssd_step_host on CPU tensors (pin them for asynchronous copies): returns a dict
    ``y, final_state (or None), dx, d_raw_dt, dB, dC`` of CPU tensors (``dy=None``: the
    forward alone, no gradients), complete once ``stream`` (default: the current stream)
    has passed the call.  ``device_buffer`` is a CUDA uint8 tensor of at least
    ``step_host_size`` bytes; the current device is used."""
    torch = _torch()
    for t, name in ((x, "x"), (raw_dt, "raw_dt"), (B, "B"), (C, "C"), (dy, "dy")):
        if t is None and name == "dy":
            continue
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("%s must be a contiguous CPU tensor" % name)
    if raw_dt.dtype != torch.float32:
        raise TypeError("raw_dt must be float32")
    if cu_seqlens is not None and (cu_seqlens.is_cuda or cu_seqlens.dtype != torch.int32):
        raise ValueError("cu_seqlens must be an int32 CPU tensor")
    prob = make_problem(x, B, delta_init, chunk_size, cu_seqlens)
    nseq = prob.nseq if prob.nseq > 0 else prob.batch
    if out is None:
        pin = x.is_pinned()
        def like(t):
            return torch.empty(t.shape, dtype=t.dtype, pin_memory=pin)
        grads = dy is not None
        out = {"y": like(x), "dx": like(x) if grads else None,
               "d_raw_dt": like(raw_dt) if grads else None,
               "dB": like(B) if grads else None, "dC": like(C) if grads else None,
               "final_state": torch.empty((nseq, prob.nheads, prob.headdim, prob.dstate),
                                          dtype=torch.float32, pin_memory=pin)
               if final_state else None}
    dev = torch.device("cuda", torch.cuda.current_device())
    buf = _workspace(step_host_size(prob), dev, device_buffer)
    st = _lib.lib().ssd_step_host(ctypes.byref(prob), _ptr(x), _ptr(raw_dt), _ptr(B), _ptr(C),
                                  _ptr(cu_seqlens), _ptr(dy), _ptr(out["y"]),
                                  _ptr(out.get("final_state")), _ptr(out.get("dx")),
                                  _ptr(out.get("d_raw_dt")), _ptr(out.get("dB")),
                                  _ptr(out.get("dC")),
                                  _ptr(buf), buf.numel(), _stream(stream))
    check(st, "ssd_step_host")
    return out


def device_status(workspace, stream=None) -> int:
    v = ctypes.c_int32(0)
    check(_lib.lib().ssd_device_status(_ptr(workspace), _stream(stream), ctypes.byref(v)),
          "ssd_device_status")
    return int(v.value)


class profiler:
    """Per-kernel device time from events the library records around each launch."""

    @staticmethod
    def enable(on: bool = True) -> None:
        _lib.lib().ssd_profiler_enable(int(on))

    @staticmethod
    def only(name=None) -> None:
        """Times only the launches of kernel ``name`` (None: every kernel)."""
        _lib.lib().ssd_profiler_only(None if name is None else name.encode())

    @staticmethod
    def reset() -> None:
        _lib.lib().ssd_profiler_reset()

    @staticmethod
    def read() -> dict:
        l = _lib.lib()
        out = {}
        for i in range(l.ssd_profiler_count()):
            name = ctypes.c_char_p()
            n = ctypes.c_int64()
            ms = ctypes.c_double()
            check(l.ssd_profiler_entry(i, ctypes.byref(name), ctypes.byref(n), ctypes.byref(ms)),
                  "ssd_profiler_entry")
            out[name.value.decode()] = (int(n.value), float(ms.value))
        return out
