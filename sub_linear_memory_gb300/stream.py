"""Sequences kept in host memory, processed window by window on the GPU.

"Sub-Linear Memory: How to Make Performers SLiM", sections 3.2-3.3: a slice
of rows is linked to the rows before it only by the prefix-sum state at its
boundary, and to the rows after it only by the reverse (gradient) state.  The
same holds for a window of many slices, so a sequence whose Q, K, V, dY (and
Y, dQ, dK, dV) live in pinned host memory can be run through the library one
window at a time:

  forward, windows left to right: copy the window's Q, K, V in, run
  slim_attn_fwd_carry from the previous window's final state, copy Y out, and
  keep the window's incoming state in pinned host memory (the boundary
  checkpoint, (d + 1) x M floats per head);

  backward, windows right to left: copy Q, K, V, dY and the window's
  checkpoint in, run slim_attn_bwd_carry with the reverse state of the window
  after it, copy dQ, dK, dV out and pass the gradient w.r.t. the incoming
  state on to the window before.

Device memory then holds two windows of buffers (inputs of window i + 1 copy
in while window i computes and window i - 1's outputs copy out), a few states
and the library's workspace: it does not grow with L.  Copies run on streams
of their own with events ordering them against the compute stream; every
computation is a library call (this module only moves data and accumulates
the per-window dW).
"""

import torch

from . import binding


class Checkpoints:
    """Boundary states of a streamed forward: checkpoint i is the state the
    forward of window i started from (window 0 starts from zero), fp32 pinned
    host [n_windows, B, H, d + 1, M]."""

    def __init__(self, states, window, length):
        self.states = states
        self.window = window
        self.length = length


def _windows(length, window):
    return [(a, min(window, length - a)) for a in range(0, length, window)]


class _Buffers:
    """Device buffers for windows of `window` rows (double-buffered by window
    parity), plus separate buffers for a shorter last window."""

    def __init__(self, shape, dtype, device, n_in, n_out, window, last_rows):
        b, h, _, d = shape
        mk = lambda rows: [torch.empty((b, h, rows, d), dtype=dtype, device=device) for _ in range(n_in + n_out)]
        self.full = [mk(window), mk(window)]
        self.last = mk(last_rows) if last_rows != window else None
        self.n_in = n_in

    def get(self, parity, rows, is_last):
        t = self.last if (is_last and self.last is not None) else self.full[parity]
        return t[:self.n_in], t[self.n_in:]


def _check_host(*ts):
    for t in ts:
        if t.device.type != "cpu" or not t.is_pinned() or not t.is_contiguous():
            raise ValueError("streamed tensors must be contiguous pinned host [B, H, L, d] tensors")


def streamed_forward(q, k, v, w, chunk, window, y=None, ckpt=None, device=None):
    """Y for host-resident q, k, v (pinned [B, H, L, d]); returns (y, checkpoints)
    with y pinned host.  ``window`` rows per library call (a multiple of 128
    keeps the calls on whole 128-row tiles).  ``ckpt``: optional pinned fp32
    [n_windows, B, H, d + 1, M] buffer for the boundary checkpoints."""
    _check_host(q, k, v)
    b, h, length, d = q.shape
    m = d if w is None else w.shape[1]
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    if y is None:
        y = torch.empty(q.shape, dtype=q.dtype).pin_memory()
    wins = _windows(length, window)
    if ckpt is None:
        ckpt = torch.empty((len(wins), b, h, d + 1, m), dtype=torch.float32).pin_memory()
    if ckpt.shape != (len(wins), b, h, d + 1, m) or not ckpt.is_pinned():
        raise ValueError("ckpt must be a pinned fp32 [n_windows, B, H, d + 1, M] tensor")
    if wins:
        ckpt[0].zero_()  # window 0 starts from the zero state
    if not wins:
        return y, Checkpoints(ckpt, window, length)
    comp = torch.cuda.current_stream(dev)
    h2d, d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    bufs = _Buffers(q.shape, q.dtype, dev, 3, 1, window, wins[-1][1])
    states = [torch.zeros((b, h, d + 1, m), dtype=torch.float32, device=dev) for _ in range(2)]
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_read = [torch.cuda.Event() for _ in range(2)]
    h2d.wait_stream(comp)

    def load(i):
        a, rows = wins[i]
        par = i % 2
        ins, _ = bufs.get(par, rows, i == len(wins) - 1)
        if i >= 2:
            h2d.wait_event(ev_done[par])  # window i - 2 no longer reads these buffers
        for dst, src in zip(ins, (q, k, v)):
            binding.copy_rows(dst, 0, src, a, rows, stream=h2d)
        ev_in[par].record(h2d)

    load(0)
    for i, (a, rows) in enumerate(wins):
        par = i % 2
        ins, outs = bufs.get(par, rows, i == len(wins) - 1)
        if i + 1 < len(wins):
            load(i + 1)
        comp.wait_event(ev_in[par])
        if i >= 2:
            comp.wait_event(ev_read[par])  # window i - 2's Y has left this buffer
        s_in = states[i % 2] if i > 0 else None
        s_out = states[(i + 1) % 2] if i + 1 < len(wins) else None
        if i > 0:
            ckpt[i].copy_(s_in, non_blocking=True)  # the boundary checkpoint, to pinned host memory
        binding.slim_attn_fwd(ins[0], ins[1], ins[2], w, chunk, y=outs[0], state_in=s_in, state_out=s_out)
        ev_done[par].record(comp)
        d2h.wait_event(ev_done[par])
        binding.copy_rows(y, a, outs[0], 0, rows, stream=d2h)
        ev_read[par].record(d2h)
    comp.wait_stream(d2h)
    return y, Checkpoints(ckpt, window, length)


def streamed_backward(q, k, v, dy, w, chunk, ckpt, want_dw=False, out=None, device=None):
    """dQ, dK, dV (pinned host) and dW (device fp32 [d, M], summed over the
    windows, or None) for host-resident q, k, v, dy and the checkpoints of
    streamed_forward over the same q, k, v, w and window."""
    _check_host(q, k, v, dy)
    b, h, length, d = q.shape
    m = d if w is None else w.shape[1]
    if length != ckpt.length:
        raise ValueError("checkpoints belong to another sequence length")
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    if out is None:
        out = tuple(torch.empty(q.shape, dtype=q.dtype).pin_memory() for _ in range(3))
    dq, dk, dv = out
    wins = _windows(length, ckpt.window)
    want_dw = want_dw and w is not None
    dw = torch.zeros((d, m), dtype=torch.float32, device=dev) if want_dw else None
    if not wins:
        return dq, dk, dv, dw
    comp = torch.cuda.current_stream(dev)
    h2d, d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    bufs = _Buffers(q.shape, q.dtype, dev, 4, 3, ckpt.window, wins[-1][1])
    s_in = [torch.empty((b, h, d + 1, m), dtype=torch.float32, device=dev) for _ in range(2)]
    grads = [torch.zeros((b, h, d + 1, m), dtype=torch.float32, device=dev) for _ in range(2)]
    dw_win = torch.empty((d, m), dtype=torch.float32, device=dev) if want_dw else None
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_read = [torch.cuda.Event() for _ in range(2)]
    order = list(range(len(wins) - 1, -1, -1))
    h2d.wait_stream(comp)

    def load(j):
        i = order[j]
        a, rows = wins[i]
        par = j % 2
        ins, _ = bufs.get(par, rows, i == len(wins) - 1)
        if j >= 2:
            h2d.wait_event(ev_done[par])  # two windows back no longer reads these buffers
        for dst, src in zip(ins, (q, k, v, dy)):
            binding.copy_rows(dst, 0, src, a, rows, stream=h2d)
        with torch.cuda.stream(h2d):
            s_in[par].copy_(ckpt.states[i], non_blocking=True)  # the window's checkpoint comes back
        ev_in[par].record(h2d)

    load(0)
    for j, i in enumerate(order):
        a, rows = wins[i]
        par = j % 2
        ins, outs = bufs.get(par, rows, i == len(wins) - 1)
        if j + 1 < len(order):
            load(j + 1)
        comp.wait_event(ev_in[par])
        if j >= 2:
            comp.wait_event(ev_read[par])  # that window's gradients have left these buffers
        g_in = grads[j % 2] if j > 0 else None
        g_out = grads[(j + 1) % 2] if i > 0 else None
        binding.slim_attn_bwd(ins[0], ins[1], ins[2], w, ins[3], chunk, out=(outs[0], outs[1], outs[2], dw_win),
                              state_in=s_in[par] if i > 0 else None, g_in=g_in, g_out=g_out)
        if want_dw:
            dw.add_(dw_win)
        ev_done[par].record(comp)
        d2h.wait_event(ev_done[par])
        for dst, src in zip((dq, dk, dv), outs):
            binding.copy_rows(dst, a, src, 0, rows, stream=d2h)
        ev_read[par].record(d2h)
    comp.wait_stream(d2h)
    return dq, dk, dv, dw


def device_bytes(shape, dtype, window, d, m, backward=True):
    """Device bytes the window buffers and carried states of one streamed pass
    hold (the library's workspace comes on top): two windows of inputs and
    outputs, independent of the sequence length."""
    b, h = shape[0], shape[1]
    per_window = b * h * window * d * torch.empty((), dtype=dtype).element_size()
    n = (4 + 3) if backward else (3 + 1)
    return 2 * n * per_window + 4 * b * h * (d + 1) * m * 4
