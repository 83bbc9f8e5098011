"""CPU oracle for the Mamba-2 SSD forward pass and its gradients -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline legs of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports, loads or calls anything here, and this
package imports nothing from the product.

Two independent implementations live here:

* ``ssd_oracle.c`` -- the token-by-token fp64 recurrence (the definition), in
  plain C, threaded over (batch, head) units.  Wrapped below via ctypes.
* ``closed_form.py`` -- numpy fp64 closed forms (brute-force quadratic form,
  naive chunked form, jump formula with A = 0) used only to pin the C oracle.

Array conventions (all numpy, C-contiguous):
    x  (batch, L, H, P)   uint16 bfloat16 bit patterns
    dt (batch, L, H)      float32
    A  (H,)               float32
    B, C (batch, L, G, N) uint16 bfloat16 bit patterns
    D  (H,)               float32 or None
    init (batch, H, P, N) float32 or None
    states / chunk states (batch, nc, H, P, N); dA_cumsum (batch, H, nc, Q)
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssd_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libssd_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ssd_oracle.c with gcc into oracle/_build/libssd_oracle.so."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm", "-lpthread"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            p, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
            lib.ssd_oracle_forward.argtypes = [p] * 7 + [i64] * 7 + [p, i64, p, p, p, i32]
            f64 = ctypes.c_double
            lib.ssd_oracle_forward_opts.argtypes = ([p] * 7 + [i64] * 7 + [p, i32, i32, f64, f64, i32, p] +
                                                    [p, i64, p, p, p, i32])
            lib.ssd_oracle_chunk_states.argtypes = [p] * 4 + [i64] * 7 + [p, i64, p, i32]
            lib.ssd_oracle_chunk_scan.argtypes = [p] * 7 + [i64] * 7 + [p, i64, p, i32]
            lib.ssd_oracle_dA_cumsum.argtypes = [p, p, i64, i64, i64, i64, p, p]
            lib.ssd_oracle_state_passing.argtypes = [p, p, p] + [i64] * 6 + [p, p]
            lib.ssd_oracle_backward.argtypes = [p] * 9 + [i64] * 6 + [p, i64] + [p] * 15 + [i32]
            for f in ("ssd_oracle_forward", "ssd_oracle_forward_opts", "ssd_oracle_chunk_states", "ssd_oracle_chunk_scan",
                      "ssd_oracle_dA_cumsum", "ssd_oracle_state_passing", "ssd_oracle_backward"):
                getattr(lib, f).restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {dtype}, got {a.dtype}")
    return a


def _units(batch, nheads, units):
    if units is None:
        units = np.arange(batch * nheads, dtype=np.int64)
    units = np.ascontiguousarray(np.asarray(units, dtype=np.int64))
    if units.ndim != 1 or units.size == 0 or units.min() < 0 or units.max() >= batch * nheads:
        raise ValueError("units must be a non-empty list of b * H + h indices")
    return units


def last_threads_used() -> int:
    return _last_threads[0]


_last_threads = [0]


def forward(x, dt, A, B, C, D, init, chunk_size, units=None, want_chunk_starts=False, nthreads=0,
            dt_bias=None, dt_softplus=False, dt_limit=None, z=None):
    """Token-by-token fp64 recurrence.

    Returns dict with ``y`` (nunits, L, P), ``final`` (nunits, P, N) and,
    if requested, ``chunk_starts`` (nunits, nc, P, N): the state before each
    chunk of ``chunk_size`` tokens.  ``units`` lists b * H + h indices
    (default: all units, in order).

    Input-side options of a whole layer (none by default): ``dt_bias`` (H,)
    f32 added to dt, ``dt_softplus`` (dt <- log(1 + exp(dt))), ``dt_limit``
    = (lo, hi) clamp applied last; D of shape (H, P) gives one skip weight
    per channel; ``z`` (batch, L, H, P) bf16 bits gates y <- y z sigmoid(z).
    """
    x, B, C = _c(x, np.uint16), _c(B, np.uint16), _c(C, np.uint16)
    dt, A = _c(dt, np.float32), _c(A, np.float32)
    D, init = _c(D, np.float32), _c(init, np.float32)
    dt_bias, z = _c(dt_bias, np.float32), _c(z, np.uint16)
    b, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    nc = -(-L // chunk_size)
    u = _units(b, H, units)
    y = np.empty((u.size, L, P), np.float64)
    fin = np.empty((u.size, P, N), np.float64)
    cst = np.empty((u.size, nc, P, N), np.float64) if want_chunk_starts else None
    if D is not None and D.shape not in ((H,), (H, P)):
        raise ValueError("D must be (H,) or (H, P)")
    if z is not None and z.shape != x.shape:
        raise ValueError("z must have x's shape")
    if dt_bias is not None and dt_bias.shape != (H,):
        raise ValueError("dt_bias must be (H,)")
    plain = dt_bias is None and not dt_softplus and dt_limit is None and z is None and (D is None or D.ndim == 1)
    if plain:
        r = _load().ssd_oracle_forward(_ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(init),
                                       b, L, H, P, G, N, chunk_size, _ptr(u), u.size,
                                       _ptr(y), _ptr(fin), _ptr(cst), nthreads)
    else:
        lo, hi = (0.0, 0.0) if dt_limit is None else (float(dt_limit[0]), float(dt_limit[1]))
        r = _load().ssd_oracle_forward_opts(_ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(init),
                                            b, L, H, P, G, N, chunk_size,
                                            _ptr(dt_bias), int(bool(dt_softplus)), int(dt_limit is not None), lo, hi,
                                            int(D is not None and D.ndim == 2), _ptr(z),
                                            _ptr(u), u.size, _ptr(y), _ptr(fin), _ptr(cst), nthreads)
    if r < 0:
        raise ValueError("ssd_oracle_forward: bad arguments")
    _last_threads[0] = r
    out = {"y": y, "final": fin}
    if want_chunk_starts:
        out["chunk_starts"] = cst
    return out


def chunk_states(x, dt, A, B, chunk_size, units=None, nthreads=0):
    """Per chunk, the state reached from zero over that chunk alone: (nunits, nc, P, N)."""
    x, B = _c(x, np.uint16), _c(B, np.uint16)
    dt, A = _c(dt, np.float32), _c(A, np.float32)
    b, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    nc = -(-L // chunk_size)
    u = _units(b, H, units)
    S = np.empty((u.size, nc, P, N), np.float64)
    r = _load().ssd_oracle_chunk_states(_ptr(x), _ptr(dt), _ptr(A), _ptr(B), b, L, H, P, G, N,
                                        chunk_size, _ptr(u), u.size, _ptr(S), nthreads)
    if r < 0:
        raise ValueError("ssd_oracle_chunk_states: bad arguments")
    return S


def chunk_scan(x, dt, A, B, C, D, states, chunk_size, units=None, nthreads=0):
    """Outputs with every chunk restarted from ``states`` (batch, nc, H, P, N) f32: (nunits, L, P)."""
    x, B, C = _c(x, np.uint16), _c(B, np.uint16), _c(C, np.uint16)
    dt, A, D = _c(dt, np.float32), _c(A, np.float32), _c(D, np.float32)
    states = _c(states, np.float32)
    b, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    u = _units(b, H, units)
    y = np.empty((u.size, L, P), np.float64)
    r = _load().ssd_oracle_chunk_scan(_ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(states),
                                      b, L, H, P, G, N, chunk_size, _ptr(u), u.size, _ptr(y), nthreads)
    if r < 0:
        raise ValueError("ssd_oracle_chunk_scan: bad arguments")
    return y


def dA_cumsum(dt, A, chunk_size):
    """Inclusive in-chunk cumsum of dt*A times log2(e), and dt, both (batch, H, nc, Q) f64."""
    dt, A = _c(dt, np.float32), _c(A, np.float32)
    b, L, H = dt.shape
    nc = -(-L // chunk_size)
    cs = np.empty((b, H, nc, chunk_size), np.float64)
    dtt = np.empty((b, H, nc, chunk_size), np.float64)
    r = _load().ssd_oracle_dA_cumsum(_ptr(dt), _ptr(A), b, L, H, chunk_size, _ptr(cs), _ptr(dtt))
    if r < 0:
        raise ValueError("ssd_oracle_dA_cumsum: bad arguments")
    return cs, dtt


def state_passing(S, cs, init, chunk_size):
    """Sequential chunk hop. S (batch, nc, H, P, N) f32, cs (batch, H, nc, Q) f32, init f32 or None.

    Returns (states (batch, nc, H, P, N), final (batch, H, P, N)) in f64.
    """
    S, cs, init = _c(S, np.float32), _c(cs, np.float32), _c(init, np.float32)
    b, nc, H, P, N = S.shape
    states = np.empty(S.shape, np.float64)
    fin = np.empty((b, H, P, N), np.float64)
    r = _load().ssd_oracle_state_passing(_ptr(S), _ptr(cs), _ptr(init), b, nc, H, P, N, chunk_size,
                                         _ptr(states), _ptr(fin))
    if r < 0:
        raise ValueError("ssd_oracle_state_passing: bad arguments")
    return states, fin


def backward(x, dt, A, B, C, D, init, dy, dfinal=None, units=None, nthreads=0, scales=False):
    """Gradients of a scalar loss by the reverse-time recurrence (fp64).

    ``dy`` (batch, L, H, P) bf16 bits is dLoss/dy, ``dfinal`` (batch, H, P, N)
    f32 or None is dLoss/dfinal.  Per listed unit (b * H + h): ``dx`` (L, P),
    ``dB`` and ``dC`` (L, N) -- this head's share (a group's gradient is the
    sum over its heads) --, ``ddt`` (L,), ``dA`` and ``dD`` (this unit's share),
    ``dinit`` (P, N), and ``ddt_direct`` (L,): ddt's term <lam_t, B_t x_t^T> alone (the rest,
    ddt - ddt_direct, is A exp(dt_t A) <lam_t, state_{t-1}>).

    With ``scales``, also ``dx_s``, ``dB_s``, ``dC_s``, ``ddt_s``, ``dA_s``, ``dD_s``, ``dinit_s`` in the
    same layouts: the sum of the magnitudes of the products each gradient adds up (dx: dt sum_n |B lam|
    + |D dy|; dB: dt sum_p |lam x|; dC: sum_p |state dy|; ddt: |A| exp(dt A) sum |lam state_prev| +
    sum |lam B x|; dA: the sum over tokens of dt exp(dt A) sum |lam state_prev|; dD: sum |x dy|;
    dinit: the adjoint's terms |C_t dy_t^T| and |dfinal|, each decayed to the start as lam is).
    """
    x, B, C, dy = _c(x, np.uint16), _c(B, np.uint16), _c(C, np.uint16), _c(dy, np.uint16)
    dt, A = _c(dt, np.float32), _c(A, np.float32)
    D, init, dfinal = _c(D, np.float32), _c(init, np.float32), _c(dfinal, np.float32)
    b, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    if dy.shape != x.shape:
        raise ValueError("dy must have x's shape")
    if D is not None and D.shape != (H,):
        raise ValueError("D must be (H,)")
    u = _units(b, H, units)
    out = {"dx": np.empty((u.size, L, P)), "dB": np.empty((u.size, L, N)), "dC": np.empty((u.size, L, N)),
           "ddt": np.empty((u.size, L)), "dA": np.empty(u.size), "dD": np.empty(u.size),
           "dinit": np.empty((u.size, P, N)), "ddt_direct": np.empty((u.size, L))}
    names = ("dx", "dB", "dC", "ddt", "dA", "dD", "dinit", "ddt_direct")
    snames = ("dx_s", "dB_s", "dC_s", "ddt_s", "dA_s", "dD_s", "dinit_s")
    if scales:
        for k in snames:
            out[k] = np.empty_like(out[k[:-2]])
    r = _load().ssd_oracle_backward(_ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(init), _ptr(dy),
                                    _ptr(dfinal), b, L, H, P, G, N, _ptr(u), u.size,
                                    *[_ptr(out[k]) for k in names], *[_ptr(out.get(k)) for k in snames],
                                    nthreads)
    if r < 0:
        raise ValueError("ssd_oracle_backward: bad arguments")
    _last_threads[0] = r
    return out


def backward_full(x, dt, A, B, C, D, init, dy, dfinal=None, nthreads=0):
    """``backward`` over every unit, assembled into the inputs' layouts: dx (b, L, H, P), ddt (b, L, H),
    dB, dC (b, L, G, N) summed over each group's heads, dA, dD (H,) summed over the batch, dinit (b, H, P, N)."""
    b, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    r = backward(x, dt, A, B, C, D, init, dy, dfinal, nthreads=nthreads)
    hpg = H // G
    dB = r["dB"].reshape(b, H, L, N).reshape(b, G, hpg, L, N).sum(axis=2).transpose(0, 2, 1, 3)
    dC = r["dC"].reshape(b, H, L, N).reshape(b, G, hpg, L, N).sum(axis=2).transpose(0, 2, 1, 3)
    return {"dx": r["dx"].reshape(b, H, L, P).transpose(0, 2, 1, 3), "ddt": r["ddt"].reshape(b, H, L).transpose(0, 2, 1),
            "dB": np.ascontiguousarray(dB), "dC": np.ascontiguousarray(dC),
            "dA": r["dA"].reshape(b, H).sum(axis=0), "dD": r["dD"].reshape(b, H).sum(axis=0),
            "dinit": r["dinit"].reshape(b, H, P, N)}


def backward_terms(x, dt, A, B, C, D, init, dy, dfinal=None, nthreads=0):
    """``backward_full`` plus ``scales``: for every gradient, in its layout, the sum of the magnitudes of
    the products it adds up (see ``backward``), summed like the gradient itself (over a group's heads
    for dB and dC, over the batch for dA and dD)."""
    b, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    r = backward(x, dt, A, B, C, D, init, dy, dfinal, nthreads=nthreads, scales=True)
    hpg = H // G

    def group_sum(a):
        return np.ascontiguousarray(a.reshape(b, G, hpg, L, N).sum(axis=2).transpose(0, 2, 1, 3))

    out = {"dx": r["dx"].reshape(b, H, L, P).transpose(0, 2, 1, 3), "ddt": r["ddt"].reshape(b, H, L).transpose(0, 2, 1),
           "dB": group_sum(r["dB"]), "dC": group_sum(r["dC"]),
           "dA": r["dA"].reshape(b, H).sum(axis=0), "dD": r["dD"].reshape(b, H).sum(axis=0),
           "dinit": r["dinit"].reshape(b, H, P, N)}
    out["scales"] = {"dx": r["dx_s"].reshape(b, H, L, P).transpose(0, 2, 1, 3),
                     "ddt": r["ddt_s"].reshape(b, H, L).transpose(0, 2, 1),
                     "dB": group_sum(r["dB_s"]), "dC": group_sum(r["dC_s"]),
                     "dA": r["dA_s"].reshape(b, H).sum(axis=0), "dD": r["dD_s"].reshape(b, H).sum(axis=0),
                     "dinit": r["dinit_s"].reshape(b, H, P, N)}
    return out
