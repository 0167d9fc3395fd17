"""Carried boundary states and host-resident sequences, on the GPU, against
the fp64 oracle ("Sub-Linear Memory: How to Make Performers SLiM", sections
3.2-3.3: a window of rows is linked to the rows before it only by the
prefix-sum state at its boundary and to the rows after it only by the
reverse state).

* slim_attn_fwd_carry / slim_attn_bwd_carry with a nonzero incoming state
  (the prefix sums of earlier rows) and a nonzero incoming reverse state,
  on every kernel family, with 1 and several segments per head (the last
  segment's correction by the incoming reverse state);
* the streaming driver over windows of a sequence in pinned host memory
  equals one pass of the oracle over all rows, and the device memory it holds
  does not grow with the sequence length.
Bars: relative L2 <= 2e-2 (bf16 I/O), <= 1e-4 (fp32 I/O), as everywhere.
"""
import numpy as np
import pytest
import torch

import oracle
from sub_linear_memory_gb300 import inputs

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from sub_linear_memory_gb300 import binding

    binding.set_option(binding.OPT_SEGMENTS, 0)
    binding.set_option(binding.OPT_PATH, 0)
    yield binding
    binding.set_option(binding.OPT_SEGMENTS, 0)
    binding.set_option(binding.OPT_PATH, 0)


def _np(t):
    return t.detach().to("cpu", torch.float64).numpy()


def _case(B, H, L, d, M, C, dtype, feature, seed, prior=300):
    base = inputs.WORKLOADS["tiny" if dtype == torch.float32 else "l4k"]
    wl = base.with_(B=B, H=H, L=L, d=d, M=M, chunk=C, index=600 + seed,
                    dtype="fp32" if dtype == torch.float32 else "bf16", feature=feature,
                    qk_scale=(1.0 if feature == "elu" else d ** -0.25),
                    w_kind=("none" if feature == "elu" else base.w_kind))
    q, k, v, dy, w = inputs.make_inputs(wl)
    # the incoming state: prefix sums of `prior` earlier rows of the same recipe
    _, kp, vp, _, _ = inputs.make_inputs(wl.with_(L=prior, index=700 + seed))
    wn = None if w is None else _np(w)
    kpn, vpn = _np(kp.to(dtype)), _np(vp.to(dtype))
    state0 = oracle.prefill_state(kpn, vpn, wn)
    g = torch.Generator().manual_seed(800 + seed)
    g0 = (torch.randn((B, H, d + 1, M), generator=g, dtype=torch.float64) * 0.05).numpy()
    dev = "cuda"
    t = lambda x: x.to(dev)
    return (t(q), t(k), t(v), t(dy), None if w is None else t(w), state0, g0)


def _check(name, got, ref, tol):
    err = oracle.rel_l2(got, ref)
    print("%s rel L2 %.3e (tol %.0e)" % (name, err, tol))
    assert np.isfinite(err) and err <= tol, "%s: rel L2 %.3e > %.1e" % (name, err, tol)


CASES = [
    # (B, H, L, d, M, C, dtype, feature)
    (1, 2, 700, 64, 256, 128, torch.bfloat16, "favor"),   # tensor path, two-CTA backward
    (2, 1, 1000, 64, 128, 64, torch.bfloat16, "favor"),   # tensor path, one CTA
    (1, 2, 1300, 64, 64, 256, torch.bfloat16, "favor"),
    (1, 2, 333, 64, 64, 128, torch.bfloat16, "elu"),      # tensor path, elu+1
    (1, 2, 300, 128, 128, 64, torch.bfloat16, "elu"),     # tensor forward, CUDA-core backward
    (1, 2, 250, 16, 32, 32, torch.float32, "favor"),      # CUDA-core path, fp32
    (1, 1, 200, 32, 32, 16, torch.float32, "elu"),
]


@pytest.mark.parametrize("segments", [0, 1, 3])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(str(x) for x in c[:6]) + "-" + c[7]
                         + ("-f32" if c[6] == torch.float32 else ""))
def test_carried_states_match_oracle(case, segments, lib):
    B, H, L, d, M, C, dtype, feature = case
    q, k, v, dy, w, state0, g0 = _case(B, H, L, d, M, C, dtype, feature, seed=segments)
    tol = TOL[dtype]
    dev = q.device
    s_in = torch.tensor(state0, dtype=torch.float32, device=dev)
    g_in = torch.tensor(g0, dtype=torch.float32, device=dev)
    s_out = torch.full_like(s_in, float("nan"))
    g_out = torch.full_like(s_in, float("nan"))
    lib.set_option(lib.OPT_SEGMENTS, segments)
    try:
        y = lib.slim_attn_fwd(q, k, v, w, C, state_in=s_in, state_out=s_out)
        dq, dk, dv, dw = lib.slim_attn_bwd(q, k, v, w, dy, C, want_dw=w is not None, state_in=s_in, g_in=g_in,
                                           g_out=g_out)
        lib.sync_status()
    finally:
        lib.set_option(lib.OPT_SEGMENTS, 0)
    qn, kn, vn, dyn = _np(q), _np(k), _np(v), _np(dy)
    wn = None if w is None else _np(w)
    y_ref, s_ref = oracle.recurrence_forward(qn, kn, vn, wn, state0=state0, return_state=True)
    ref = oracle.recurrence_backward(qn, kn, vn, wn, dyn, want_dw=w is not None, state0=state0, g0=g0,
                                     want_gstate=True)
    _check("Y", _np(y), y_ref, tol)
    _check("state_out", _np(s_out), s_ref, tol)
    for name, got, exp in (("dQ", dq, ref[0]), ("dK", dk, ref[1]), ("dV", dv, ref[2])):
        _check(name, _np(got), exp, tol)
    if w is not None:
        _check("dW", _np(dw), ref[3], tol)
    _check("g_out", _np(g_out), ref[4], tol)


def test_zero_rows_pass_the_states_through(lib):
    q = torch.empty((1, 2, 0, 64), dtype=torch.bfloat16, device="cuda")
    w = torch.randn(64, 128, device="cuda")
    s_in = torch.randn(1, 2, 65, 128, device="cuda")
    g_in = torch.randn(1, 2, 65, 128, device="cuda")
    s_out, g_out = torch.zeros_like(s_in), torch.zeros_like(s_in)
    lib.slim_attn_fwd(q, q, q, w, 64, state_in=s_in, state_out=s_out)
    lib.slim_attn_bwd(q, q, q, w, q, 64, state_in=s_in, g_in=g_in, g_out=g_out)
    lib.sync_status()
    assert torch.equal(s_out, s_in) and torch.equal(g_out, g_in)


def _pinned(t):
    return t.contiguous().pin_memory()


@pytest.mark.parametrize("window", [256, 384, 1000])
@pytest.mark.parametrize("M", [64, 256])
def test_streamed_windows_match_one_pass(window, M, lib):
    """A sequence in pinned host memory, run window by window (the last one
    short), equals the oracle's one pass over all rows."""
    from sub_linear_memory_gb300 import stream

    wl = inputs.WORKLOADS["l1m"].with_(B=1, H=3, L=1000, M=M, index=900 + M)
    q, k, v, dy, w = inputs.make_inputs(wl)
    qh, kh, vh, dyh = (_pinned(t) for t in (q, k, v, dy))
    wd = w.cuda()
    y, ckpt = stream.streamed_forward(qh, kh, vh, wd, wl.chunk, window)
    dq, dk, dv, dw = stream.streamed_backward(qh, kh, vh, dyh, wd, wl.chunk, ckpt, want_dw=True)
    torch.cuda.synchronize()
    lib.sync_status()
    qn, kn, vn, dyn, wn = _np(q), _np(k), _np(v), _np(dy), _np(w)
    _check("Y", _np(y), oracle.recurrence_forward(qn, kn, vn, wn), 2e-2)
    ref = oracle.recurrence_backward(qn, kn, vn, wn, dyn, want_dw=True)
    for name, got, exp in zip(("dQ", "dK", "dV", "dW"), (dq, dk, dv, dw), ref):
        _check(name, _np(got), exp, 2e-2)
    # checkpoint i is the state after the first i windows' rows
    for i in range(1, ckpt.states.shape[0]):
        rows = i * window
        exp = oracle.prefill_state(kn[:, :, :rows], vn[:, :, :rows], wn)
        _check("checkpoint %d" % i, _np(ckpt.states[i]), exp, 2e-2)


def test_streamed_device_memory_does_not_grow_with_length(lib):
    """The streamed pass holds two windows of device buffers plus states and
    the workspace: its peak device allocation is the same for a sequence four
    times longer."""
    from sub_linear_memory_gb300 import stream

    peaks = []
    for L in (1 << 15, 1 << 17):
        wl = inputs.WORKLOADS["l1m"].with_(L=L, index=950)
        q, k, v, dy, w = inputs.make_inputs(wl)
        qh, kh, vh, dyh = (_pinned(t) for t in (q, k, v, dy))
        wd = w.cuda()
        lib.release_workspace()
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        torch.cuda.reset_peak_memory_stats()
        base = torch.cuda.memory_allocated()
        y, ckpt = stream.streamed_forward(qh, kh, vh, wd, wl.chunk, 1 << 13)
        stream.streamed_backward(qh, kh, vh, dyh, wd, wl.chunk, ckpt)
        torch.cuda.synchronize()
        lib.sync_status()
        peaks.append(torch.cuda.max_memory_allocated() - base)
        del q, k, v, dy, qh, kh, vh, dyh, y, ckpt
    print("streamed peak device bytes at L = 2^15, 2^17:", peaks)
    assert peaks[1] <= peaks[0] + (1 << 20), peaks


def test_streamed_long_sequence_matches_oracle_on_sampled_heads(lib):
    """The 1M workload's head shape at L = 2^18 in pinned host memory, run in
    2^16-row windows (the bench's streamed leg at a quarter of its shortest
    length): Y, dQ, dK, dV and the last checkpoint of two heads against the
    oracle's one pass (heads are independent, so a head is an exact unit)."""
    from sub_linear_memory_gb300 import stream

    wl = inputs.WORKLOADS["l1m"].with_(L=1 << 18, index=960)
    q, k, v, dy, w = inputs.make_inputs(wl)
    qh, kh, vh, dyh = (_pinned(t) for t in (q, k, v, dy))
    wd = w.cuda()
    window = 1 << 16
    y, ckpt = stream.streamed_forward(qh, kh, vh, wd, wl.chunk, window)
    dq, dk, dv, _ = stream.streamed_backward(qh, kh, vh, dyh, wd, wl.chunk, ckpt)
    torch.cuda.synchronize()
    lib.sync_status()
    heads = [1, 6]
    sel = lambda t: _np(t[:, heads])
    qn, kn, vn, dyn, wn = sel(q), sel(k), sel(v), sel(dy), _np(w)
    _check("Y", sel(y), oracle.recurrence_forward(qn, kn, vn, wn), 2e-2)
    ref = oracle.recurrence_backward(qn, kn, vn, wn, dyn, want_dw=False)
    for name, got, exp in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
        _check(name, sel(got), exp, 2e-2)
    last = ckpt.states.shape[0] - 1
    exp = oracle.prefill_state(kn[:, :, :last * window], vn[:, :, :last * window], wn)
    _check("checkpoint %d" % last, _np(ckpt.states[last][:, heads]), exp, 2e-2)
