"""fp64 CPU oracle for causal linear self-attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It shares no code with the CUDA
library in ``sub_linear_memory_gb300`` and never imports it.

Two independent formulations of "Sub-Linear Memory: How to Make Performers
SLiM", section 2.1:
  * ``recurrence_forward`` / ``recurrence_backward``: the per-step prefix-sum
    recurrence, eq. (3)-(4), in plain C (``slim_oracle.c``), fp64, OpenMP over
    heads;
  * ``quadratic.forward`` / ``quadratic.backward``: the explicit quadratic form
    of eq. (2), numpy fp64;
  * ``quadratic.softmax_forward``: eq. (1), the exponential attention that the
    randomized feature map approximates;
  * ``prefill_state`` / ``decode_step``: the same recurrence in its serving
    form, one new row at a time against a carried state (C);
  * W may be one [d, M] matrix shared by every head or one per head
    ([H, d, M], dW then per head too);
  * the forward and backward also take the boundary state of rows that came
    before (``state0``) and the gradient arriving from rows that come after
    (``g0``), and return the state after the last row and the gradient with
    respect to ``state0``: a sequence cut into windows is then the same
    computation, window by window.
"""
import ctypes
import os
import subprocess
import threading

import numpy as np

from . import lm  # noqa: F401  (re-exported)
from . import orf  # noqa: F401  (re-exported)
from . import quadratic  # noqa: F401  (re-exported)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "slim_oracle.c")
_LIB = os.path.join(_HERE, "libslim_oracle.so")
_lock = threading.Lock()
_lib = None

MAP_FAVOR = 0
MAP_ELU = 1


def build(force=False):
    """Compile the C oracle with gcc (plain C99 + OpenMP; no target flags)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c99", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            lib.oracle_forward.argtypes = [dp] * 5 + [ctypes.c_long] * 3 + [ctypes.c_int] * 4
            lib.oracle_backward.argtypes = [dp] * 10 + [ctypes.c_long] * 3 + [ctypes.c_int] * 4
            lib.oracle_forward_carry.argtypes = [dp] * 7 + [ctypes.c_long] * 3 + [ctypes.c_int] * 4
            lib.oracle_backward_carry.argtypes = [dp] * 13 + [ctypes.c_long] * 3 + [ctypes.c_int] * 4
            lib.oracle_feature_map.argtypes = [dp] * 3 + [ctypes.c_long] + [ctypes.c_int] * 3
            lib.oracle_state.argtypes = [dp] * 4 + [ctypes.c_long] * 3 + [ctypes.c_int] * 4
            lib.oracle_decode.argtypes = [dp] * 6 + [ctypes.c_long] * 2 + [ctypes.c_int] * 3
            for fn in (lib.oracle_forward, lib.oracle_backward, lib.oracle_feature_map, lib.oracle_state,
                       lib.oracle_decode, lib.oracle_forward_carry, lib.oracle_backward_carry):
                fn.restype = ctypes.c_int
            lib.oracle_max_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _check_w(w, d):
    if w is not None and (np.ndim(w) != 2 or np.shape(w)[0] != d):
        raise ValueError("W must be [d, M] with d = %d, got %s" % (d, np.shape(w)))


def _as4d(x):
    x = _f64(x)
    if x.ndim == 2:
        x = x[None, None]
    if x.ndim != 4:
        raise ValueError("expected [B, H, L, d] or [L, d]")
    return x


def max_threads():
    return int(_load().oracle_max_threads())


def feature_map(x, w):
    """g applied to every row of x ([rows, d]); w None selects elu+1."""
    x = _f64(x)
    rows, d = x.reshape(-1, x.shape[-1]).shape
    _check_w(w, d)
    m = d if w is None else int(np.shape(w)[1])
    wf = None if w is None else _f64(w)
    out = np.empty((rows, m), dtype=np.float64)
    rc = _load().oracle_feature_map(_ptr(x), _ptr(wf), _ptr(out), rows, d, m,
                                     MAP_ELU if w is None else MAP_FAVOR)
    if rc:
        raise ValueError("oracle_feature_map failed (%d)" % rc)
    return out.reshape(x.shape[:-1] + (m,))


def _state_arg(st, b, h, d, m, what):
    if st is None:
        return None
    st = _f64(st)
    if st.shape != (b, h, d + 1, m):
        raise ValueError("%s must be [B, H, d + 1, M] = %s, got %s" % (what, (b, h, d + 1, m), st.shape))
    return st


def _per_head(w):
    return w is not None and np.ndim(w) == 3


def recurrence_forward(q, k, v, w, threads=0, state0=None, return_state=False):
    if _per_head(w):
        return _forward_per_head(q, k, v, w, threads, state0, return_state)
    return _recurrence_forward(q, k, v, w, threads, state0, return_state)


def _forward_per_head(q, k, v, w, threads, state0, return_state):
    """W per head ([H, d, M]): head h of every batch entry uses w[h]; each head
    is the shared-W computation with its own W."""
    q, k, v = _as4d(q), _as4d(k), _as4d(v)
    h_count = q.shape[1]
    if np.shape(w)[0] != h_count:
        raise ValueError("per-head W must be [H, d, M] with H = %d" % h_count)
    ys, states = [], []
    for h in range(h_count):
        sl = lambda t: np.ascontiguousarray(t[:, h:h + 1])
        out = _recurrence_forward(sl(q), sl(k), sl(v), w[h], threads, None if state0 is None else sl(state0),
                                  return_state)
        if return_state:
            ys.append(out[0])
            states.append(out[1])
        else:
            ys.append(out)
    y = np.concatenate(ys, axis=1)
    return (y, np.concatenate(states, axis=1)) if return_state else y


def _recurrence_forward(q, k, v, w, threads=0, state0=None, return_state=False):
    """Y = Att^lin(Q, K, V) by the per-step recurrence; arrays [B, H, L, d]
    (or [L, d]).  w None selects elu+1, else W is [d, M].

    ``state0`` ([B, H, d + 1, M], e-major like the serving state): the stacked
    prefix sums R' = [R ; S^T] of rows that came before these (default zero).
    ``return_state``: also return the state after the last row."""
    shape = np.shape(q)
    q, k, v = _as4d(q), _as4d(k), _as4d(v)
    b, h, length, d = q.shape
    _check_w(w, d)
    m = d if w is None else int(np.shape(w)[1])
    wf = None if w is None else _f64(w)
    s0 = _state_arg(state0, b, h, d, m, "state0")
    s_out = np.empty((b, h, d + 1, m), dtype=np.float64) if return_state else None
    y = np.empty_like(q)
    rc = _load().oracle_forward_carry(_ptr(q), _ptr(k), _ptr(v), _ptr(wf), _ptr(y), _ptr(s0), _ptr(s_out),
                                      b, h, length, d, m, MAP_ELU if w is None else MAP_FAVOR, int(threads))
    if rc:
        raise ValueError("oracle_forward failed (%d)" % rc)
    y = y.reshape(shape)
    return (y, s_out) if return_state else y


def recurrence_backward(q, k, v, w, dy, threads=0, want_dw=True, want_y=False, state0=None, g0=None,
                        want_gstate=False):
    if _per_head(w):
        return _backward_per_head(q, k, v, w, dy, threads, want_dw, want_y, state0, g0, want_gstate)
    return _recurrence_backward(q, k, v, w, dy, threads, want_dw, want_y, state0, g0, want_gstate)


def _backward_per_head(q, k, v, w, dy, threads, want_dw, want_y, state0, g0, want_gstate):
    """W per head ([H, d, M]): dW is per head too, [H, d, M], summed over the
    batch entries and rows of that head."""
    q, k, v, dy = _as4d(q), _as4d(k), _as4d(v), _as4d(dy)
    h_count = q.shape[1]
    if np.shape(w)[0] != h_count:
        raise ValueError("per-head W must be [H, d, M] with H = %d" % h_count)
    parts = []
    for h in range(h_count):
        sl = lambda t: None if t is None else np.ascontiguousarray(t[:, h:h + 1])
        parts.append(_recurrence_backward(sl(q), sl(k), sl(v), w[h], sl(dy), threads, want_dw, want_y,
                                          sl(state0), sl(g0), want_gstate))
    cat = lambda i: np.concatenate([p[i] for p in parts], axis=1)
    out = (cat(0), cat(1), cat(2), np.stack([p[3] for p in parts]) if want_dw else None)
    i = 4
    if want_y:
        out = out + (cat(i),)
        i += 1
    if want_gstate:
        out = out + (cat(i),)
    return out


def _recurrence_backward(q, k, v, w, dy, threads=0, want_dw=True, want_y=False, state0=None, g0=None,
                         want_gstate=False):
    """Gradients of sum(dy * Y) + sum(g0 * R'_L): returns (dq, dk, dv, dw[, y][, g_state]);
    dw is None for elu+1 or when ``want_dw`` is False.

    ``state0`` ([B, H, d + 1, M]): the state the forward started from (default
    zero).  ``g0`` (same layout, default zero): the gradient of what follows
    these rows with respect to the state R'_L after the last row.
    ``want_gstate``: also return the gradient with respect to state0."""
    shape = np.shape(q)
    q, k, v, dy = _as4d(q), _as4d(k), _as4d(v), _as4d(dy)
    b, h, length, d = q.shape
    _check_w(w, d)
    m = d if w is None else int(np.shape(w)[1])
    wf = None if w is None else _f64(w)
    s0 = _state_arg(state0, b, h, d, m, "state0")
    gin = _state_arg(g0, b, h, d, m, "g0")
    gout = np.empty((b, h, d + 1, m), dtype=np.float64) if want_gstate else None
    dq, dk, dv = np.empty_like(q), np.empty_like(q), np.empty_like(q)
    dw = np.empty((d, m), dtype=np.float64) if (w is not None and want_dw) else None
    y = np.empty_like(q) if want_y else None
    rc = _load().oracle_backward_carry(_ptr(q), _ptr(k), _ptr(v), _ptr(wf), _ptr(dy), _ptr(dq),
                                       _ptr(dk), _ptr(dv), _ptr(dw), _ptr(y), _ptr(s0), _ptr(gin), _ptr(gout),
                                       b, h, length, d, m, MAP_ELU if w is None else MAP_FAVOR, int(threads))
    if rc:
        raise ValueError("oracle_backward failed (%d)" % rc)
    out = (dq.reshape(shape), dk.reshape(shape), dv.reshape(shape), dw)
    if want_y:
        out = out + (y.reshape(shape),)
    if want_gstate:
        out = out + (gout,)
    return out


def prefill_state(k, v, w, threads=0):
    """Serving form of eq. (3)-(4): the stacked state R' = [R ; S^T] after all
    L rows of k, v ([B, H, L, d]), e-major: [B, H, d + 1, M] with
    state[e, m] = sum_j v_j[e] g(k_j)[m] for e < d and state[d, m] = sum_j g(k_j)[m]."""
    k, v = _as4d(k), _as4d(v)
    b, h, length, d = k.shape
    _check_w(w, d)
    m = d if w is None else int(np.shape(w)[1])
    wf = None if w is None else _f64(w)
    st = np.empty((b, h, d + 1, m), dtype=np.float64)
    rc = _load().oracle_state(_ptr(k), _ptr(v), _ptr(wf), _ptr(st), b, h, length, d, m,
                              MAP_ELU if w is None else MAP_FAVOR, int(threads))
    if rc:
        raise ValueError("oracle_state failed (%d)" % rc)
    return st


def decode_step(q, k, v, w, state):
    """One new row per head: q, k, v [B, H, d]; state [B, H, d + 1, M] is
    updated in place with the row's term (diagonal included), then
    y = (g(q) . R) / (g(q) . S) is returned as [B, H, d]."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    if q.ndim != 3:
        raise ValueError("q, k, v must be [B, H, d]")
    b, h, d = q.shape
    _check_w(w, d)
    m = d if w is None else int(np.shape(w)[1])
    if state.dtype != np.float64 or not state.flags.c_contiguous or state.shape != (b, h, d + 1, m):
        raise ValueError("state must be a contiguous float64 [B, H, d + 1, M] array")
    wf = None if w is None else _f64(w)
    y = np.empty((b, h, d), dtype=np.float64)
    rc = _load().oracle_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(wf), _ptr(state), _ptr(y), b, h, d, m,
                               MAP_ELU if w is None else MAP_FAVOR)
    if rc:
        raise ValueError("oracle_decode failed (%d)" % rc)
    return y


def rel_l2(x, ref):
    """Relative L2 error ||x - ref||_2 / ||ref||_2 over the whole tensor, in fp64
    (the discrepancy measure the paper uses for gradients, section 4)."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.linalg.norm((x - ref).ravel()) / np.linalg.norm(ref.ravel()))
