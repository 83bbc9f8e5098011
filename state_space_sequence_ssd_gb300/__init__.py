"""GB300 (sm_103a) Mamba-2 SSD chunked forward pass.

Thin Python binding over the C ABI of include/ssd.h.  Each function has the
name of its C entry point and only marshals arguments: torch supplies device
memory and the stream, every step of the computation runs in the library's
CUDA kernels.  Inputs must be contiguous CUDA tensors:

    x (batch, L, H, P) bf16, dt (batch, L, H) f32, A (H,) f32,
    B, C (batch, L, G, N) bf16, D (H,) f32 or None,
    init_state / final_state (batch, H, P, N) f32,
    dA_cumsum / dt_t (batch, H, nchunks, chunk_size) f32,
    chunk_states / states (batch, nchunks, H, P, N) f32.

``stream`` is a torch.cuda.Stream (default: the current stream).
"""
from __future__ import annotations

from . import _ffi

__all__ = ["ssd_chunk_cumsum", "ssd_chunk_state", "ssd_state_passing", "ssd_chunk_scan", "ssd_forward",
           "ssd_forward_noalloc", "ssd_forward_heads", "ssd_partition_heads", "ssd_forward_plan", "ssd_step",
           "ssd_step_multi", "ssd_forward_ex", "ssd_step_ex", "ssd_backward", "ssd_get_device_error", "SSDError", "library_path"]

SSDError = _ffi.SSDError
library_path = _ffi.LIB_PATH


def _torch():
    import torch
    return torch


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _need(t, name, dtype, ndim=None):
    torch = _torch()
    if t is None:
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (no CPU path exists)")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")
    return t


def _opt(t, name, dtype, ndim=None):
    return None if t is None else _need(t, name, dtype, ndim)


def ssd_chunk_cumsum(dt, A, chunk_size, dA_cumsum=None, dt_t=None, stream=None):
    """chunk_cumsum stage -> (dA_cumsum, dt_t), both (batch, H, nchunks, chunk_size) f32."""
    torch = _torch()
    _need(dt, "dt", torch.float32, 3)
    _need(A, "A", torch.float32, 1)
    b, L, H = dt.shape
    nc = -(-L // chunk_size)
    if dA_cumsum is None:
        dA_cumsum = torch.empty((b, H, nc, chunk_size), device=dt.device, dtype=torch.float32)
    if dt_t is None:
        dt_t = torch.empty((b, H, nc, chunk_size), device=dt.device, dtype=torch.float32)
    _need(dA_cumsum, "dA_cumsum", torch.float32, 4)
    _need(dt_t, "dt_t", torch.float32, 4)
    _ffi.check("ssd_chunk_cumsum", _ffi.lib().ssd_chunk_cumsum(
        _ptr(dt), _ptr(A), b, L, H, chunk_size, _ptr(dA_cumsum), _ptr(dt_t), _stream(stream)))
    return dA_cumsum, dt_t


def ssd_chunk_state(x, B, dt_t, dA_cumsum, chunk_size, chunk_states=None, stream=None):
    """First half of fwd_pass_state -> chunk_states (batch, nchunks, H, P, N) f32."""
    torch = _torch()
    _need(x, "x", torch.bfloat16, 4)
    _need(B, "B", torch.bfloat16, 4)
    _need(dt_t, "dt_t", torch.float32, 4)
    _need(dA_cumsum, "dA_cumsum", torch.float32, 4)
    b, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    nc = -(-L // chunk_size)
    if chunk_states is None:
        chunk_states = torch.empty((b, nc, H, P, N), device=x.device, dtype=torch.float32)
    _need(chunk_states, "chunk_states", torch.float32, 5)
    _ffi.check("ssd_chunk_state", _ffi.lib().ssd_chunk_state(
        _ptr(x), _ptr(B), _ptr(dt_t), _ptr(dA_cumsum), b, L, H, P, G, N, chunk_size,
        _ptr(chunk_states), _stream(stream)))
    return chunk_states


def ssd_state_passing(chunk_states, dA_cumsum, init_state, chunk_size, states=None, final_state=None,
                      want_final=True, stream=None):
    """Second half of fwd_pass_state -> (states, final_state or None)."""
    torch = _torch()
    _need(chunk_states, "chunk_states", torch.float32, 5)
    _need(dA_cumsum, "dA_cumsum", torch.float32, 4)
    _opt(init_state, "init_state", torch.float32, 4)
    b, nc, H, P, N = chunk_states.shape
    if states is None:
        states = torch.empty_like(chunk_states)
    if final_state is None and want_final:
        final_state = torch.empty((b, H, P, N), device=chunk_states.device, dtype=torch.float32)
    _need(states, "states", torch.float32, 5)
    _opt(final_state, "final_state", torch.float32, 4)
    _ffi.check("ssd_state_passing", _ffi.lib().ssd_state_passing(
        _ptr(chunk_states), _ptr(dA_cumsum), _ptr(init_state), b, nc, H, P, N, chunk_size,
        _ptr(states), _ptr(final_state), _stream(stream)))
    return states, final_state


def ssd_chunk_scan(x, B, C, dt_t, dA_cumsum, D, states, chunk_size, y=None, stream=None):
    """compute_out stage -> y (batch, L, H, P) bf16."""
    torch = _torch()
    _need(x, "x", torch.bfloat16, 4)
    _need(B, "B", torch.bfloat16, 4)
    _need(C, "C", torch.bfloat16, 4)
    _need(dt_t, "dt_t", torch.float32, 4)
    _need(dA_cumsum, "dA_cumsum", torch.float32, 4)
    _opt(D, "D", torch.float32, 1)
    _need(states, "states", torch.float32, 5)
    b, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    if y is None:
        y = torch.empty_like(x)
    _need(y, "y", torch.bfloat16, 4)
    _ffi.check("ssd_chunk_scan", _ffi.lib().ssd_chunk_scan(
        _ptr(x), _ptr(B), _ptr(C), _ptr(dt_t), _ptr(dA_cumsum), _ptr(D), _ptr(states),
        b, L, H, P, G, N, chunk_size, _ptr(y), _stream(stream)))
    return y


def ssd_forward(x, dt, A, B, C, D, init_state, chunk_size, y=None, final_state=None, want_final=True,
                stream=None):
    """Whole chunked forward pass -> (y, final_state or None)."""
    torch = _torch()
    _need(x, "x", torch.bfloat16, 4)
    _need(dt, "dt", torch.float32, 3)
    _need(A, "A", torch.float32, 1)
    _need(B, "B", torch.bfloat16, 4)
    _need(C, "C", torch.bfloat16, 4)
    _opt(D, "D", torch.float32, 1)
    _opt(init_state, "init_state", torch.float32, 4)
    b, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    if y is None:
        y = torch.empty_like(x)
    if final_state is None and want_final:
        final_state = torch.empty((b, H, P, N), device=x.device, dtype=torch.float32)
    _need(y, "y", torch.bfloat16, 4)
    _opt(final_state, "final_state", torch.float32, 4)
    _ffi.check("ssd_forward", _ffi.lib().ssd_forward(
        _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(init_state),
        b, L, H, P, G, N, chunk_size, _ptr(y), _ptr(final_state), _stream(stream)))
    return y, final_state


def ssd_backward(x, dt, A, B, C, D, init_state, dy, dfinal=None, chunk_size=256, want_dD=True, want_dinit=True,
                 stream=None):
    """Gradients through ssd_forward given dy (x's layout, bf16) and dfinal ((batch, H, P, N) f32 or None).

    Returns a dict: dx (batch, L, H, P) bf16, ddt (batch, L, H) f32, dA (H,) f32, dB and dC
    (batch, L, G, N) f32 (summed over each group's heads), dD (H,) f32 or None, dinit
    (batch, H, P, N) f32 or None."""
    torch = _torch()
    _need(x, "x", torch.bfloat16, 4)
    _need(dt, "dt", torch.float32, 3)
    _need(A, "A", torch.float32, 1)
    _need(B, "B", torch.bfloat16, 4)
    _need(C, "C", torch.bfloat16, 4)
    _opt(D, "D", torch.float32, 1)
    _opt(init_state, "init_state", torch.float32, 4)
    _need(dy, "dy", torch.bfloat16, 4)
    _opt(dfinal, "dfinal", torch.float32, 4)
    b, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    dev = x.device
    out = {"dx": torch.empty_like(x), "ddt": torch.empty((b, L, H), device=dev, dtype=torch.float32),
           "dA": torch.empty((H,), device=dev, dtype=torch.float32),
           "dB": torch.empty((b, L, G, N), device=dev, dtype=torch.float32),
           "dC": torch.empty((b, L, G, N), device=dev, dtype=torch.float32),
           "dD": torch.empty((H,), device=dev, dtype=torch.float32) if want_dD else None,
           "dinit": torch.empty((b, H, P, N), device=dev, dtype=torch.float32) if want_dinit else None}
    _ffi.check("ssd_backward", _ffi.lib().ssd_backward(
        _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(init_state), _ptr(dy), _ptr(dfinal),
        b, L, H, P, G, N, chunk_size, _ptr(out["dx"]), _ptr(out["ddt"]), _ptr(out["dA"]), _ptr(out["dB"]),
        _ptr(out["dC"]), _ptr(out["dD"]), _ptr(out["dinit"]), _stream(stream)))
    return out


def ssd_forward_heads(x, dt, A, B, C, D, init_state, chunk_size, head_begin, head_count, y=None, final_state=None,
                      want_final=True, stream=None):
    """ssd_forward over heads [head_begin, head_begin + head_count) of the full-size tensors, in place:
    only those heads' rows of y and final_state are written.  Returns (y, final_state or None)."""
    torch = _torch()
    _need(x, "x", torch.bfloat16, 4)
    _need(dt, "dt", torch.float32, 3)
    _need(A, "A", torch.float32, 1)
    _need(B, "B", torch.bfloat16, 4)
    _need(C, "C", torch.bfloat16, 4)
    _opt(D, "D", torch.float32, 1)
    _opt(init_state, "init_state", torch.float32, 4)
    b, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    if y is None:
        y = torch.empty_like(x)
    if final_state is None and want_final:
        final_state = torch.empty((b, H, P, N), device=x.device, dtype=torch.float32)
    _need(y, "y", torch.bfloat16, 4)
    _opt(final_state, "final_state", torch.float32, 4)
    _ffi.check("ssd_forward_heads", _ffi.lib().ssd_forward_heads(
        _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(init_state),
        b, L, H, P, G, N, chunk_size, int(head_begin), int(head_count), _ptr(y), _ptr(final_state), _stream(stream)))
    return y, final_state


def ssd_partition_heads(nheads, ngroups, nparts, part):
    """(head_begin, head_count) of part `part` of `nparts` for ssd_forward_heads (host only)."""
    import ctypes
    hb, hc = ctypes.c_int(0), ctypes.c_int(0)
    _ffi.check("ssd_partition_heads", _ffi.lib().ssd_partition_heads(
        int(nheads), int(ngroups), int(nparts), int(part), ctypes.addressof(hb), ctypes.addressof(hc)))
    return hb.value, hc.value


def _options(x, D, dt_bias, dt_softplus, dt_limit, z, H, P):
    """ssd_input_options from keyword arguments; D may be (H,) or (H, P) (one weight per channel)."""
    torch = _torch()
    _opt(dt_bias, "dt_bias", torch.float32, 1)
    _opt(z, "z", torch.bfloat16, x.dim())
    if dt_bias is not None and tuple(dt_bias.shape) != (H,):
        raise ValueError(f"dt_bias must have shape {(H,)}, got {tuple(dt_bias.shape)}")
    if z is not None and tuple(z.shape) != tuple(x.shape):
        raise ValueError(f"z must have x's shape {tuple(x.shape)}, got {tuple(z.shape)}")
    if D is not None:
        _need(D, "D", torch.float32)
        if tuple(D.shape) not in ((H,), (H, P)):
            raise ValueError(f"D must have shape {(H,)} or {(H, P)}, got {tuple(D.shape)}")
    o = _ffi.InputOptions()
    o.dt_bias = _ptr(dt_bias)
    o.dt_softplus = int(bool(dt_softplus))
    if dt_limit is not None:
        o.dt_limit = 1
        o.dt_min, o.dt_max = float(dt_limit[0]), float(dt_limit[1])
    o.D_per_channel = int(D is not None and D.dim() == 2)
    o.z = _ptr(z)
    return o


def ssd_forward_ex(x, dt, A, B, C, D, init_state, chunk_size, dt_bias=None, dt_softplus=False, dt_limit=None,
                   z=None, y=None, final_state=None, want_final=True, stream=None):
    """ssd_forward with a whole layer's input-side options:
    dt <- clamp(softplus(dt + dt_bias), *dt_limit) (each part optional), D of shape (H,) or (H, P)
    (one skip weight per channel), and y <- y * z * sigmoid(z) with z shaped like x.
    Returns (y, final_state or None); the state is never gated."""
    import ctypes
    torch = _torch()
    _need(x, "x", torch.bfloat16, 4)
    _need(dt, "dt", torch.float32, 3)
    _need(A, "A", torch.float32, 1)
    _need(B, "B", torch.bfloat16, 4)
    _need(C, "C", torch.bfloat16, 4)
    _opt(init_state, "init_state", torch.float32, 4)
    b, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    opts = _options(x, D, dt_bias, dt_softplus, dt_limit, z, H, P)
    if y is None:
        y = torch.empty_like(x)
    if final_state is None and want_final:
        final_state = torch.empty((b, H, P, N), device=x.device, dtype=torch.float32)
    _need(y, "y", torch.bfloat16, 4)
    _opt(final_state, "final_state", torch.float32, 4)
    _ffi.check("ssd_forward_ex", _ffi.lib().ssd_forward_ex(
        _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(init_state),
        b, L, H, P, G, N, chunk_size, ctypes.addressof(opts), _ptr(y), _ptr(final_state), _stream(stream)))
    return y, final_state


def ssd_step_ex(x, dt, A, B, C, D, state, dt_bias=None, dt_softplus=False, dt_limit=None, z=None, y=None,
                stream=None):
    """ssd_step with the input-side options of ssd_forward_ex (z shaped like x: (batch, H, P))."""
    import ctypes
    torch = _torch()
    _need(x, "x", torch.bfloat16, 3)
    _need(dt, "dt", torch.float32, 2)
    _need(A, "A", torch.float32, 1)
    _need(B, "B", torch.bfloat16, 3)
    _need(C, "C", torch.bfloat16, 3)
    _need(state, "state", torch.float32, 4)
    b, H, P = x.shape
    G, N = B.shape[1], B.shape[2]
    opts = _options(x, D, dt_bias, dt_softplus, dt_limit, z, H, P)
    if y is None:
        y = torch.empty_like(x)
    _need(y, "y", torch.bfloat16, 3)
    for name, t, shape in (("dt", dt, (b, H)), ("A", A, (H,)), ("B", B, (b, G, N)), ("C", C, (b, G, N)),
                           ("state", state, (b, H, P, N)), ("y", y, (b, H, P))):
        if tuple(t.shape) != shape:
            raise ValueError(f"{name} must have shape {shape}, got {tuple(t.shape)}")
    _ffi.check("ssd_step_ex", _ffi.lib().ssd_step_ex(
        _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(state), b, H, P, G, N,
        ctypes.addressof(opts), _ptr(y), _stream(stream)))
    return y


def ssd_forward_noalloc(x, dt, A, B, C, D, init_state, chunk_size, y, final_state=None, stream=None):
    """ssd_forward with no allocation: the library works in its fixed device
    scratch array, and the caller supplies y (and final_state, or None to skip
    it), so this call allocates nothing either.  Calls on one device share the
    scratch: overlapping calls on different streams race.  Raises SSDError
    with SSD_ERR_SCRATCH_TOO_SMALL when the workload does not fit."""
    torch = _torch()
    _need(x, "x", torch.bfloat16, 4)
    _need(dt, "dt", torch.float32, 3)
    _need(A, "A", torch.float32, 1)
    _need(B, "B", torch.bfloat16, 4)
    _need(C, "C", torch.bfloat16, 4)
    _opt(D, "D", torch.float32, 1)
    _opt(init_state, "init_state", torch.float32, 4)
    _need(y, "y", torch.bfloat16, 4)
    _opt(final_state, "final_state", torch.float32, 4)
    b, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    _ffi.check("ssd_forward_noalloc", _ffi.lib().ssd_forward_noalloc(
        _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(init_state),
        b, L, H, P, G, N, chunk_size, _ptr(y), _ptr(final_state), _stream(stream)))
    return y, final_state


def ssd_step(x, dt, A, B, C, D, state, y=None, stream=None):
    """One recurrent step for a single new token of every sequence.

    x (batch, H, P) bf16, dt (batch, H) f32, A (H,) f32, B, C (batch, G, N) bf16,
    D (H,) f32 or None, state (batch, H, P, N) f32 updated in place.  Returns y (batch, H, P) bf16."""
    torch = _torch()
    _need(x, "x", torch.bfloat16, 3)
    _need(dt, "dt", torch.float32, 2)
    _need(A, "A", torch.float32, 1)
    _need(B, "B", torch.bfloat16, 3)
    _need(C, "C", torch.bfloat16, 3)
    _opt(D, "D", torch.float32, 1)
    _need(state, "state", torch.float32, 4)
    b, H, P = x.shape
    G, N = B.shape[1], B.shape[2]
    if y is None:
        y = torch.empty_like(x)
    _need(y, "y", torch.bfloat16, 3)
    for name, t, shape in (("dt", dt, (b, H)), ("A", A, (H,)), ("B", B, (b, G, N)), ("C", C, (b, G, N)),
                           ("D", D, (H,)), ("state", state, (b, H, P, N)), ("y", y, (b, H, P))):
        if t is not None and tuple(t.shape) != shape:
            raise ValueError(f"{name} must have shape {shape}, got {tuple(t.shape)}")
    _ffi.check("ssd_step", _ffi.lib().ssd_step(
        _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(state), b, H, P, G, N, _ptr(y),
        _stream(stream)))
    return y


def ssd_step_multi(x, dt, A, B, C, D, state, y=None, stream=None):
    """K consecutive new tokens of every sequence in one call (ssd_step K times, the state kept on chip).

    x (batch, K, H, P) bf16, dt (batch, K, H) f32, A (H,) f32, B, C (batch, K, G, N) bf16,
    D (H,) f32 or None, state (batch, H, P, N) f32 updated in place.  Returns y (batch, K, H, P) bf16."""
    torch = _torch()
    _need(x, "x", torch.bfloat16, 4)
    _need(dt, "dt", torch.float32, 3)
    _need(A, "A", torch.float32, 1)
    _need(B, "B", torch.bfloat16, 4)
    _need(C, "C", torch.bfloat16, 4)
    _opt(D, "D", torch.float32, 1)
    _need(state, "state", torch.float32, 4)
    b, K, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    if y is None:
        y = torch.empty_like(x)
    _need(y, "y", torch.bfloat16, 4)
    for name, t, shape in (("dt", dt, (b, K, H)), ("A", A, (H,)), ("B", B, (b, K, G, N)), ("C", C, (b, K, G, N)),
                           ("D", D, (H,)), ("state", state, (b, H, P, N)), ("y", y, (b, K, H, P))):
        if t is not None and tuple(t.shape) != shape:
            raise ValueError(f"{name} must have shape {shape}, got {tuple(t.shape)}")
    _ffi.check("ssd_step_multi", _ffi.lib().ssd_step_multi(
        _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(state), b, K, H, P, G, N, _ptr(y),
        _stream(stream)))
    return y


def ssd_forward_plan(batch, seqlen, nheads, headdim, ngroups, dstate, chunk_size):
    """How ssd_forward splits a workload of these sizes (host-side query, nothing allocated or launched):
    {"span_chunks": chunks per span, "scan_step": spans per compute_out CTA,
     "noalloc_bytes": workspace ssd_forward_noalloc needs in its fixed scratch}."""
    import ctypes
    span, step, nb = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_ulonglong(0)
    _ffi.check("ssd_forward_plan", _ffi.lib().ssd_forward_plan(
        batch, seqlen, nheads, headdim, ngroups, dstate, chunk_size, ctypes.addressof(span), ctypes.addressof(step),
        ctypes.addressof(nb)))
    return {"span_chunks": span.value, "scan_step": step.value, "noalloc_bytes": nb.value}


def ssd_get_device_error():
    """SSD_OK (0) or SSD_ERR_TIMEOUT (5) if a bounded device wait gave up since the last read."""
    return _ffi.lib().ssd_get_device_error()
