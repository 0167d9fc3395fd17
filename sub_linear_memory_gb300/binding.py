"""Thin ctypes binding over ``libslim_attn.so``: argument marshalling only.

Every step of the attention runs in the library's CUDA kernels; this module
checks tensor dtypes/devices/contiguity, owns the caller-side workspace (a
torch allocation, so ``torch.cuda.max_memory_allocated`` sees it) and passes
raw device pointers and the current torch stream.  There is no fallback: if
the shared library is missing, importing this module raises.
"""
import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# SLIM_ATTN_LIBRARY=debug loads the -DSLIM_DEBUG build (bounds checks; every
# call waits and reports device-side errors itself)
library_path = os.path.join(_HERE, "libslim_attn_debug.so" if os.environ.get("SLIM_ATTN_LIBRARY") == "debug"
                            else "libslim_attn.so")

if not os.path.exists(library_path):
    raise ImportError(
        os.path.basename(library_path) + " is not built (run sub_linear_memory_gb300.build.build() "
        "or __graft_entry__.build()); there is no non-CUDA fallback")

_lib = ctypes.CDLL(library_path)
_vp, _i, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t

_lib.slim_attn_fwd.argtypes = [_vp] * 5 + [_i] * 6 + [_vp]
_lib.slim_attn_fwd_f32.argtypes = _lib.slim_attn_fwd.argtypes
_lib.slim_attn_bwd.argtypes = [_vp] * 9 + [_i] * 6 + [_vp]
_lib.slim_attn_bwd_f32.argtypes = _lib.slim_attn_bwd.argtypes
_lib.slim_attn_state.argtypes = [_vp] * 4 + [_i] * 6 + [_vp]
_lib.slim_attn_state_f32.argtypes = _lib.slim_attn_state.argtypes
_lib.slim_attn_decode.argtypes = [_vp] * 6 + [_i] * 4 + [_vp]
_lib.slim_attn_decode_f32.argtypes = _lib.slim_attn_decode.argtypes
for _f in (_lib.slim_attn_fwd, _lib.slim_attn_fwd_f32, _lib.slim_attn_bwd, _lib.slim_attn_bwd_f32,
           _lib.slim_attn_state, _lib.slim_attn_state_f32, _lib.slim_attn_decode, _lib.slim_attn_decode_f32):
    _f.restype = _i
_lib.slim_attn_workspace_bytes.argtypes = [_i] * 7
_lib.slim_attn_workspace_bytes.restype = _sz
_lib.slim_attn_set_workspace.argtypes = [_vp, _sz]
_lib.slim_attn_set_workspace.restype = _i
_lib.slim_attn_set_option.argtypes = [_i, _i]
_lib.slim_attn_set_option.restype = _i
_lib.slim_attn_segments.argtypes = [_i] * 6
_lib.slim_attn_segments.restype = _i
_lib.slim_attn_sync_status.argtypes = [_vp]
_lib.slim_attn_sync_status.restype = _i
_lib.slim_attn_profile_count.argtypes = []
_lib.slim_attn_profile_count.restype = _i
_lib.slim_attn_profile_get.argtypes = [_i, ctypes.POINTER(ctypes.c_char_p),
                                       ctypes.POINTER(ctypes.c_longlong), ctypes.POINTER(ctypes.c_double)]
_lib.slim_attn_profile_get.restype = _i
_lib.slim_attn_profile_reset.argtypes = []
_lib.slim_attn_profile_reset.restype = None
_lib.slim_attn_fwd_carry.argtypes = [_vp] * 7 + [_i] * 6 + [_vp]
_lib.slim_attn_fwd_carry_f32.argtypes = _lib.slim_attn_fwd_carry.argtypes
_lib.slim_attn_bwd_carry.argtypes = [_vp] * 12 + [_i] * 6 + [_vp]
_lib.slim_attn_bwd_carry_f32.argtypes = _lib.slim_attn_bwd_carry.argtypes
for _f in (_lib.slim_attn_fwd_carry, _lib.slim_attn_fwd_carry_f32, _lib.slim_attn_bwd_carry,
           _lib.slim_attn_bwd_carry_f32):
    _f.restype = _i
_ll = ctypes.c_longlong
_lib.slim_attn_copy_rows.argtypes = [_vp, _ll, _ll, _vp, _ll, _ll, _ll, _ll, _ll, _vp]
_lib.slim_attn_copy_rows.restype = _i
_lib.slim_attn_draw_orf.argtypes = [_vp, _i, _i, _i, ctypes.c_ulonglong, ctypes.c_ulonglong, _vp]
_lib.slim_attn_draw_orf.restype = _i
class LMConfig(ctypes.Structure):
    """slim_lm_config: the multi-layer Performer language model's shape."""
    _fields_ = [("vocab", _i), ("d_model", _i), ("heads", _i), ("d_ff", _i), ("layers", _i), ("favor", _i),
                ("features", _i)]


_lib.slim_lm_param_count.argtypes = [ctypes.POINTER(LMConfig)]
_lib.slim_lm_param_count.restype = _sz
_lib.slim_lm_workspace_bytes.argtypes = [ctypes.POINTER(LMConfig), _i, _i]
_lib.slim_lm_workspace_bytes.restype = _sz
_lib.slim_lm_loss_grad.argtypes = [ctypes.POINTER(LMConfig), _vp, _vp, _vp, _i, _i, _i, _vp, _vp, _vp, _vp, _sz,
                                   _vp]
_lib.slim_lm_checkpoint_bytes.argtypes = [ctypes.POINTER(LMConfig), _i, _i, _i]
_lib.slim_lm_checkpoint_bytes.restype = _sz
_lib.slim_lm_loss_grad.restype = _i
_lib.slim_attn_noalloc_bytes.argtypes = [_i] * 6
_lib.slim_attn_noalloc_bytes.restype = _sz
_lib.slim_attn_fwd_noalloc.argtypes = _lib.slim_attn_fwd.argtypes
_lib.slim_attn_fwd_noalloc.restype = _i
_lib.slim_attn_selftest_timeout.argtypes = [ctypes.c_longlong, _vp, _vp]
_lib.slim_attn_selftest_timeout.restype = _i
_lib.slim_attn_probe_ex2.argtypes = [_i, _i, _vp, _vp]
_lib.slim_attn_probe_ex2.restype = _i
_lib.slim_status_string.argtypes = [_i]
_lib.slim_status_string.restype = ctypes.c_char_p

OPT_SEGMENTS = 1
OPT_PATH = 2
OPT_PROFILE = 3
OPT_W_PER_HEAD = 4
OPT_REUSE_STATES = 5
EXPORTED = (
    "slim_attn_fwd", "slim_attn_bwd", "slim_attn_fwd_f32", "slim_attn_bwd_f32",
    "slim_attn_state", "slim_attn_state_f32", "slim_attn_decode", "slim_attn_decode_f32",
    "slim_attn_workspace_bytes", "slim_attn_set_workspace", "slim_attn_set_option",
    "slim_attn_segments", "slim_attn_sync_status", "slim_status_string",
    "slim_attn_profile_count", "slim_attn_profile_get", "slim_attn_profile_reset",
    "slim_attn_fwd_noalloc", "slim_attn_noalloc_bytes", "slim_attn_selftest_timeout",
    "slim_attn_fwd_carry", "slim_attn_bwd_carry", "slim_attn_fwd_carry_f32", "slim_attn_bwd_carry_f32",
    "slim_attn_copy_rows", "slim_attn_draw_orf", "slim_lm_param_count", "slim_lm_workspace_bytes",
    "slim_lm_loss_grad", "slim_lm_checkpoint_bytes", "slim_attn_probe_ex2",
)


class SlimError(RuntimeError):
    def __init__(self, code, what):
        super().__init__("%s: %s" % (what, _lib.slim_status_string(code).decode()))
        self.code = code


def _check(code, what):
    if code != 0:
        raise SlimError(code, what)


_ws_lock = threading.Lock()
_ws = {}


def workspace(nbytes, device):
    """A cached torch uint8 device buffer of at least ``nbytes`` (256-B aligned)."""
    dev = torch.device(device)
    key = dev.index if dev.index is not None else torch.cuda.current_device()
    with _ws_lock:
        buf = _ws.get(key)
        if buf is None or buf.numel() < nbytes:
            buf = torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=dev)
            _ws[key] = buf
        return buf


def release_workspace():
    with _ws_lock:
        _ws.clear()
    _check(_lib.slim_attn_set_workspace(None, 0), "slim_attn_set_workspace")


def set_option(option, value):
    _check(_lib.slim_attn_set_option(option, value), "slim_attn_set_option")


def segments(B, H, L, d, M, chunk):
    return _lib.slim_attn_segments(B, H, L, d, M, chunk)


def workspace_bytes(B, H, L, d, M, chunk, is_bwd):
    return _lib.slim_attn_workspace_bytes(B, H, L, d, M, chunk, int(is_bwd))


def noalloc_bytes(B, H, L, d, M, chunk):
    return _lib.slim_attn_noalloc_bytes(B, H, L, d, M, chunk)


def selftest_timeout(limit_ns, waited=None, stream=None):
    """Launch the bounded-wait self-test (a wait on a barrier nothing arms);
    ``waited`` is an optional int64 CUDA tensor of one element that receives
    the nanoseconds the wait ran."""
    s = torch.cuda.current_stream() if stream is None else stream
    _check(_lib.slim_attn_selftest_timeout(int(limit_ns), _ptr(waited), _vp(s.cuda_stream)),
           "slim_attn_selftest_timeout")


def probe_ex2(blocks, iters, sink, stream=None):
    """Launch the exponential-unit probe: blocks * 256 * iters * 8 hardware
    2^x evaluations; ``sink`` is an fp32 CUDA tensor of blocks * 256 elements."""
    if sink.dtype != torch.float32 or not sink.is_cuda or sink.numel() < blocks * 256:
        raise ValueError("sink must be an fp32 CUDA tensor of blocks * 256 elements")
    s = torch.cuda.current_stream() if stream is None else stream
    _check(_lib.slim_attn_probe_ex2(int(blocks), int(iters), _ptr(sink), _vp(s.cuda_stream)), "slim_attn_probe_ex2")


def sync_status(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    _check(_lib.slim_attn_sync_status(_vp(s.cuda_stream)), "slim_attn_sync_status")


def profile_enable(on=True):
    set_option(OPT_PROFILE, 1 if on else 0)


def profile_reset():
    _lib.slim_attn_profile_reset()


def profile_read():
    """{kernel name: (launches, total ms)} since the last reset (waits for the GPU)."""
    out = {}
    for i in range(_lib.slim_attn_profile_count()):
        name, n, ms = ctypes.c_char_p(), ctypes.c_longlong(), ctypes.c_double()
        _check(_lib.slim_attn_profile_get(i, ctypes.byref(name), ctypes.byref(n), ctypes.byref(ms)),
               "slim_attn_profile_get")
        out[name.value.decode()] = (n.value, ms.value)
    return out


def _ptr(t):
    return None if t is None else _vp(t.data_ptr())


def _validate(q, k, v, w, extra=()):
    if q.dim() != 4:
        raise ValueError("q must be [B, H, L, d]")
    for t in (q, k, v) + tuple(extra):
        if t.shape != q.shape or t.dtype != q.dtype or t.device != q.device:
            raise ValueError("q, k, v (and dy) must share shape, dtype and device")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous [B, H, L, d]")
    if q.dtype not in (torch.bfloat16, torch.float32) or q.device.type != "cuda":
        raise ValueError("tensors must be CUDA bf16 or fp32")
    if w is not None:
        # [d, M] shared by every head, or [H, d, M] with SLIM_OPT_W_PER_HEAD set
        if w.dtype != torch.float32 or w.device != q.device or w.dim() not in (2, 3) or not w.is_contiguous():
            raise ValueError("w must be a contiguous fp32 [d, M] or [H, d, M] tensor on q's device")
        if w.shape[-2] != q.shape[3] or (w.dim() == 3 and w.shape[0] != q.shape[1]):
            raise ValueError("w must be [d, M] or [H, d, M]")
    b, h, length, d = q.shape
    m = d if w is None else w.shape[-1]
    return b, h, length, d, m


def _prepare(shape, is_bwd, device):
    nbytes = workspace_bytes(*shape, is_bwd)
    buf = workspace(nbytes, device)
    _check(_lib.slim_attn_set_workspace(_vp(buf.data_ptr()), buf.numel()), "slim_attn_set_workspace")


def _check_state(st, b, h, d, m, device, what):
    if st is None:
        return
    if st.shape != (b, h, d + 1, m) or st.dtype != torch.float32 or not st.is_contiguous() \
            or st.device != device:
        raise ValueError("%s must be a contiguous fp32 [B, H, d + 1, M] tensor on q's device" % what)


def slim_attn_fwd(q, k, v, w, chunk, y=None, state_in=None, state_out=None):
    """Y = Att^lin(Q, K, V) through the library (bf16 or fp32 I/O by q's dtype).

    ``state_in`` / ``state_out`` (fp32 [B, H, d + 1, M], optional): the
    prefix-sum state of rows before these, and a buffer for the state after
    the last row (a window of a longer sequence)."""
    b, h, length, d, m = _validate(q, k, v, w)
    if y is None:
        y = torch.empty_like(q)
    _check_state(state_in, b, h, d, m, q.device, "state_in")
    _check_state(state_out, b, h, d, m, q.device, "state_out")
    _prepare((b, h, length, d, m, chunk), False, q.device)
    stream = torch.cuda.current_stream(q.device).cuda_stream
    if state_in is None and state_out is None:
        fn = _lib.slim_attn_fwd if q.dtype == torch.bfloat16 else _lib.slim_attn_fwd_f32
        _check(fn(_ptr(q), _ptr(k), _ptr(v), _ptr(w), _ptr(y), b, h, length, d, m, chunk, _vp(stream)),
               "slim_attn_fwd")
    else:
        fn = _lib.slim_attn_fwd_carry if q.dtype == torch.bfloat16 else _lib.slim_attn_fwd_carry_f32
        _check(fn(_ptr(q), _ptr(k), _ptr(v), _ptr(w), _ptr(y), _ptr(state_in), _ptr(state_out),
                  b, h, length, d, m, chunk, _vp(stream)), "slim_attn_fwd_carry")
    return y


def slim_attn_bwd(q, k, v, w, dy, chunk, want_dw=False, out=None, state_in=None, g_in=None, g_out=None):
    """Gradients of sum(dy * Y): returns (dq, dk, dv, dw or None).

    For a window of a longer sequence: ``state_in`` is the state the forward
    started from, ``g_in`` the gradient arriving at the state after the last
    row (both fp32 [B, H, d + 1, M], optional), and ``g_out`` a buffer for the
    gradient with respect to ``state_in``."""
    b, h, length, d, m = _validate(q, k, v, w, (dy,))
    if out is None:
        dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
        dw = torch.empty(tuple(w.shape), dtype=torch.float32, device=q.device) if (want_dw and w is not None) else None
    else:
        dq, dk, dv, dw = out
    for st, what in ((state_in, "state_in"), (g_in, "g_in"), (g_out, "g_out")):
        _check_state(st, b, h, d, m, q.device, what)
    _prepare((b, h, length, d, m, chunk), True, q.device)
    stream = torch.cuda.current_stream(q.device).cuda_stream
    if state_in is None and g_in is None and g_out is None:
        fn = _lib.slim_attn_bwd if q.dtype == torch.bfloat16 else _lib.slim_attn_bwd_f32
        _check(fn(_ptr(q), _ptr(k), _ptr(v), _ptr(w), _ptr(dy), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dw),
                  b, h, length, d, m, chunk, _vp(stream)), "slim_attn_bwd")
    else:
        fn = _lib.slim_attn_bwd_carry if q.dtype == torch.bfloat16 else _lib.slim_attn_bwd_carry_f32
        _check(fn(_ptr(q), _ptr(k), _ptr(v), _ptr(w), _ptr(dy), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dw),
                  _ptr(state_in), _ptr(g_in), _ptr(g_out), b, h, length, d, m, chunk, _vp(stream)),
               "slim_attn_bwd_carry")
    return dq, dk, dv, dw


def draw_orf(n, d, m, seed, step=0, out=None, device=None):
    """n FAVOR+ projections [n, d, m] (fp32, on the device) drawn by the
    library's counter-based redraw for (seed, step)."""
    if out is None:
        dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        out = torch.empty((n, d, m), dtype=torch.float32, device=dev)
    if out.shape != (n, d, m) or out.dtype != torch.float32 or not out.is_contiguous():
        raise ValueError("out must be a contiguous fp32 [n, d, M] tensor")
    stream = torch.cuda.current_stream(out.device).cuda_stream
    _check(_lib.slim_attn_draw_orf(_ptr(out), n, d, m, seed, step, _vp(stream)), "slim_attn_draw_orf")
    return out


def copy_rows(dst, dst_row0, src, src_row0, rows, stream=None):
    """Rows [src_row0, +rows) of every head of src ([B, H, L_src, d]) into rows
    [dst_row0, +rows) of dst ([B, H, L_dst, d]); host (pinned) or device
    tensors on either side, one strided asynchronous copy on ``stream``."""
    if src.dim() != 4 or dst.dim() != 4 or src.shape[:2] != dst.shape[:2] or src.shape[3] != dst.shape[3] \
            or src.dtype != dst.dtype or not src.is_contiguous() or not dst.is_contiguous():
        raise ValueError("src and dst must be contiguous [B, H, L, d] tensors of one dtype and head shape")
    s = torch.cuda.current_stream() if stream is None else stream
    heads = src.shape[0] * src.shape[1]
    row_bytes = src.shape[3] * src.element_size()
    _check(_lib.slim_attn_copy_rows(_ptr(dst), dst.shape[2], dst_row0, _ptr(src), src.shape[2], src_row0, rows,
                                    heads, row_bytes, _vp(s.cuda_stream)), "slim_attn_copy_rows")


def slim_attn_state(k, v, w, chunk, state=None):
    """The serving state after all L rows of k, v ([B, H, L, d]): fp32
    [B, H, d + 1, M], rows e < d = sum_j v_j[e] g(k_j), row d = sum_j g(k_j)."""
    b, h, length, d, m = _validate(k, v, v, w)
    if state is None:
        state = torch.empty((b, h, d + 1, m), dtype=torch.float32, device=k.device)
    if state.shape != (b, h, d + 1, m) or state.dtype != torch.float32 or not state.is_contiguous():
        raise ValueError("state must be a contiguous fp32 [B, H, d + 1, M] tensor")
    _prepare((b, h, max(length, 1), d, m, chunk), False, k.device)
    fn = _lib.slim_attn_state if k.dtype == torch.bfloat16 else _lib.slim_attn_state_f32
    stream = torch.cuda.current_stream(k.device).cuda_stream
    _check(fn(_ptr(k), _ptr(v), _ptr(w), _ptr(state), b, h, length, d, m, chunk, _vp(stream)), "slim_attn_state")
    return state


def slim_attn_decode(q, k, v, w, state, y=None):
    """One new row per head: q, k, v [B, H, d]; ``state`` (fp32 [B, H, d + 1, M])
    takes the row's term in place; returns y [B, H, d] in q's dtype."""
    if q.dim() != 3:
        raise ValueError("q, k, v must be [B, H, d]")
    b, h, d = q.shape
    b2, h2, l2, d2, m = _validate(q.unsqueeze(2), k.unsqueeze(2), v.unsqueeze(2), w)
    if state.shape != (b, h, d + 1, m) or state.dtype != torch.float32 or not state.is_contiguous() \
            or state.device != q.device:
        raise ValueError("state must be a contiguous fp32 [B, H, d + 1, M] tensor on q's device")
    if y is None:
        y = torch.empty_like(q)
    fn = _lib.slim_attn_decode if q.dtype == torch.bfloat16 else _lib.slim_attn_decode_f32
    stream = torch.cuda.current_stream(q.device).cuda_stream
    _check(fn(_ptr(q), _ptr(k), _ptr(v), _ptr(w), _ptr(state), _ptr(y), b, h, d, m, _vp(stream)),
           "slim_attn_decode")
    return y


def raw():
    """The loaded ctypes library (for tests that call the C ABI directly)."""
    return _lib


def lm_config(vocab, d_model, heads, d_ff, layers, favor=True, features=64):
    return LMConfig(vocab, d_model, heads, d_ff, layers, 1 if favor else 0, features)


def lm_param_count(cfg):
    return _lib.slim_lm_param_count(ctypes.byref(cfg))


def lm_workspace_bytes(cfg, B, chunk):
    return _lib.slim_lm_workspace_bytes(ctypes.byref(cfg), B, chunk)


_lm_ws = {}


def lm_checkpoint_bytes(cfg, B, L, chunk):
    return _lib.slim_lm_checkpoint_bytes(ctypes.byref(cfg), B, L, chunk)


def lm_loss_grad(cfg, params, feature_w, tokens, chunk, grads=None, checkpoints=None):
    """Loss (fp64 device scalar) and gradient (fp32, params' layout) of the
    multi-layer Performer on tokens (int32 device [B, L]) by Algorithm 1 with
    slices of ``chunk`` rows.  ``checkpoints``: None (states recovered by
    subtraction) or a float32 tensor of lm_checkpoint_bytes (device, or pinned
    host to keep device memory independent of L).  The workspace is a cached
    torch allocation."""
    if tokens.dtype != torch.int32 or tokens.dim() != 2 or not tokens.is_contiguous():
        raise ValueError("tokens must be a contiguous int32 [B, L] tensor")
    b, length = tokens.shape
    n = lm_param_count(cfg)
    if n == 0 or params.numel() != n or params.dtype != torch.float32 or not params.is_contiguous():
        raise ValueError("params must be a contiguous fp32 tensor of slim_lm_param_count floats")
    if grads is None:
        grads = torch.empty_like(params)
    nbytes = lm_workspace_bytes(cfg, b, min(chunk, length))
    key = params.device.index
    buf = _lm_ws.get(key)
    if buf is None or buf.numel() < nbytes:
        buf = torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=params.device)
        _lm_ws[key] = buf
    loss = torch.empty((), dtype=torch.float64, device=params.device)
    stream = torch.cuda.current_stream(params.device).cuda_stream
    if checkpoints is not None and checkpoints.numel() * checkpoints.element_size() < lm_checkpoint_bytes(
            cfg, b, length, chunk):
        raise ValueError("checkpoints too small")
    _check(_lib.slim_lm_loss_grad(ctypes.byref(cfg), _ptr(params), _ptr(feature_w), _ptr(tokens), b, length, chunk,
                                  _ptr(grads), _ptr(loss), _ptr(checkpoints), _vp(buf.data_ptr()), buf.numel(),
                                  _vp(stream)), "slim_lm_loss_grad")
    return loss, grads


def lm_release_workspace():
    _lm_ws.clear()
