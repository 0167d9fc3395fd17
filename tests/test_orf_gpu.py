"""FAVOR+ projections redrawn on the device, and one W per head, against the
fp64 oracle ("Sub-Linear Memory: How to Make Performers SLiM", section 2.1:
the randomized feature map whose projection is redrawn during training).

* slim_attn_draw_orf equals the oracle's draw from the same published
  generator (Philox4x32-10, Box-Muller, positive-diagonal QR, chi_d lengths)
  to fp32 rounding, and repeats bit for bit;
* with SLIM_OPT_W_PER_HEAD, forward, backward (dW per head) and the serving
  decode use head h's own W on every kernel family, including the
  correction kernels' per-head split and carried states.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import orf
from sub_linear_memory_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from sub_linear_memory_gb300 import binding

    binding.set_option(binding.OPT_SEGMENTS, 0)
    binding.set_option(binding.OPT_PATH, 0)
    binding.set_option(binding.OPT_W_PER_HEAD, 0)
    yield binding
    binding.set_option(binding.OPT_SEGMENTS, 0)
    binding.set_option(binding.OPT_PATH, 0)
    binding.set_option(binding.OPT_W_PER_HEAD, 0)


def _np(t):
    return t.detach().to("cpu", torch.float64).numpy()


@pytest.mark.parametrize("n,d,m,seed,step", [(1, 16, 32, 1, 0), (4, 64, 256, 1234, 7), (3, 64, 100, 2**40 + 5, 2),
                                             (2, 128, 128, 99, 1), (16, 64, 64, 3, 0)])
def test_draw_matches_oracle(n, d, m, seed, step, lib):
    w = lib.draw_orf(n, d, m, seed, step)
    w2 = lib.draw_orf(n, d, m, seed, step)
    lib.sync_status()
    assert torch.equal(w, w2)  # a redraw is a pure function of (seed, step)
    ref = orf.orf_matrices(n, d, m, seed, step)
    got = _np(w)
    err = np.linalg.norm((got - ref).ravel()) / np.linalg.norm(ref.ravel())
    print("draw rel L2 %.3e, max abs %.3e" % (err, np.max(np.abs(got - ref))))
    assert err <= 1e-6
    assert np.max(np.abs(got - ref)) <= 2e-6 * np.max(np.abs(ref))


def _case(B, H, L, d, M, C, dtype, seed):
    base = inputs.WORKLOADS["tiny" if dtype == torch.float32 else "l4k"]
    wl = base.with_(B=B, H=H, L=L, d=d, M=M, chunk=C, index=1000 + seed,
                    dtype="fp32" if dtype == torch.float32 else "bf16", qk_scale=d ** -0.25)
    q, k, v, dy, _ = inputs.make_inputs(wl)
    return q.cuda(), k.cuda(), v.cuda(), dy.cuda()


PER_HEAD = [
    # (B, H, L, d, M, C, dtype)
    (2, 3, 700, 64, 256, 128, torch.bfloat16),   # tensor path, two-CTA backward
    (2, 2, 1000, 64, 128, 64, torch.bfloat16),
    (1, 4, 1300, 64, 64, 256, torch.bfloat16),
    (2, 2, 250, 16, 32, 32, torch.float32),      # CUDA-core path
]


@pytest.mark.parametrize("segments", [0, 3])
@pytest.mark.parametrize("case", PER_HEAD, ids=lambda c: "x".join(str(x) for x in c[:6])
                         + ("-f32" if c[6] == torch.float32 else ""))
def test_per_head_w_matches_oracle(case, segments, lib):
    B, H, L, d, M, C, dtype = case
    q, k, v, dy = _case(B, H, L, d, M, C, dtype, seed=segments)
    w = lib.draw_orf(H, d, M, seed=77 + segments, step=1)
    tol = 1e-4 if dtype == torch.float32 else 2e-2
    lib.set_option(lib.OPT_W_PER_HEAD, 1)
    lib.set_option(lib.OPT_SEGMENTS, segments)
    try:
        y = lib.slim_attn_fwd(q, k, v, w, C)
        dq, dk, dv, dw = lib.slim_attn_bwd(q, k, v, w, dy, C, want_dw=True)
        lib.sync_status()
    finally:
        lib.set_option(lib.OPT_W_PER_HEAD, 0)
        lib.set_option(lib.OPT_SEGMENTS, 0)
    assert dw.shape == (H, d, M)
    qn, kn, vn, dyn, wn = _np(q), _np(k), _np(v), _np(dy), _np(w)
    y_ref = oracle.recurrence_forward(qn, kn, vn, wn)
    ref = oracle.recurrence_backward(qn, kn, vn, wn, dyn, want_dw=True)
    for name, got, exp in (("Y", y, y_ref), ("dQ", dq, ref[0]), ("dK", dk, ref[1]), ("dV", dv, ref[2]),
                           ("dW", dw, ref[3])):
        err = oracle.rel_l2(_np(got), exp)
        print("%s rel L2 %.3e" % (name, err))
        assert err <= tol, (name, err)


def test_per_head_w_with_carried_states(lib):
    B, H, L, d, M, C = 1, 3, 640, 64, 128, 128
    q, k, v, dy = _case(B, H, L, d, M, C, torch.bfloat16, seed=9)
    w = lib.draw_orf(H, d, M, seed=5)
    wn = _np(w)
    g = torch.Generator().manual_seed(5)
    kp = (torch.randn((B, H, 200, d), generator=g) * d ** -0.25).to(torch.bfloat16)
    vp = torch.randn((B, H, 200, d), generator=g).to(torch.bfloat16)
    state0 = np.concatenate([oracle.prefill_state(_np(kp)[:, h:h + 1], _np(vp)[:, h:h + 1], wn[h])
                             for h in range(H)], axis=1)
    g0 = torch.randn((B, H, d + 1, M), generator=g, dtype=torch.float64).numpy() * 0.05
    s_in = torch.tensor(state0, dtype=torch.float32, device="cuda")
    g_in = torch.tensor(g0, dtype=torch.float32, device="cuda")
    s_out, g_out = torch.empty_like(s_in), torch.empty_like(s_in)
    lib.set_option(lib.OPT_W_PER_HEAD, 1)
    lib.set_option(lib.OPT_SEGMENTS, 2)
    try:
        y = lib.slim_attn_fwd(q, k, v, w, C, state_in=s_in, state_out=s_out)
        dq, dk, dv, dw = lib.slim_attn_bwd(q, k, v, w, dy, C, want_dw=True, state_in=s_in, g_in=g_in, g_out=g_out)
        lib.sync_status()
    finally:
        lib.set_option(lib.OPT_W_PER_HEAD, 0)
        lib.set_option(lib.OPT_SEGMENTS, 0)
    qn, kn, vn, dyn = _np(q), _np(k), _np(v), _np(dy)
    y_ref, s_ref = oracle.recurrence_forward(qn, kn, vn, wn, state0=state0, return_state=True)
    ref = oracle.recurrence_backward(qn, kn, vn, wn, dyn, want_dw=True, state0=state0, g0=g0, want_gstate=True)
    for name, got, exp in (("Y", y, y_ref), ("state_out", s_out, s_ref), ("dQ", dq, ref[0]), ("dK", dk, ref[1]),
                           ("dV", dv, ref[2]), ("dW", dw, ref[3]), ("g_out", g_out, ref[4])):
        err = oracle.rel_l2(_np(got), exp)
        print("%s rel L2 %.3e" % (name, err))
        assert err <= 2e-2, (name, err)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_per_head_w_serving(dtype, lib):
    """Prefill state and one decode step with each head's own W."""
    B, H, L, d, M = 2, 3, 300, 64, 128
    q, k, v, _ = _case(B, H, L + 1, d, M, 64, dtype, seed=11)
    w = lib.draw_orf(H, d, M, seed=8)
    lib.set_option(lib.OPT_W_PER_HEAD, 1)
    try:
        state = lib.slim_attn_state(k[:, :, :L].contiguous(), v[:, :, :L].contiguous(), w, 64)
        prefill = state.clone()  # the decode step below adds row L to the state in place
        y_last = lib.slim_attn_decode(q[:, :, L].contiguous(), k[:, :, L].contiguous(), v[:, :, L].contiguous(),
                                      w, state)
        lib.sync_status()
    finally:
        lib.set_option(lib.OPT_W_PER_HEAD, 0)
    qn, kn, vn, wn = _np(q), _np(k), _np(v), _np(w)
    y_ref = oracle.recurrence_forward(qn, kn, vn, wn)[:, :, L]
    tol = 1e-4 if dtype == torch.float32 else 2e-2
    assert oracle.rel_l2(_np(y_last), y_ref) <= tol
    st_ref = np.concatenate([oracle.prefill_state(kn[:, h:h + 1, :L], vn[:, h:h + 1, :L], wn[h]) for h in range(H)],
                            axis=1)
    assert oracle.rel_l2(_np(prefill), st_ref) <= tol


def test_per_head_w_full_size_l32k(lib):
    """The l32k workload at full size with one W per head redrawn on the
    device and dW per head, as the bench's per-head leg runs it: every
    output of two heads (both batch entries of each, so dW per head is
    complete) against the oracle."""
    wl = inputs.WORKLOADS["l32k"]
    q, k, v, dy, _ = (None if t is None else t.cuda() for t in inputs.make_inputs(wl))
    w = lib.draw_orf(wl.H, wl.d, wl.M, seed=2024, step=5)
    lib.set_option(lib.OPT_W_PER_HEAD, 1)
    try:
        y = lib.slim_attn_fwd(q, k, v, w, wl.chunk)
        dq, dk, dv, dw = lib.slim_attn_bwd(q, k, v, w, dy, wl.chunk, want_dw=True)
        lib.sync_status()
    finally:
        lib.set_option(lib.OPT_W_PER_HEAD, 0)
    for h in (3, 12):
        sel = lambda t: _np(t[:, h:h + 1])
        qn, kn, vn, dyn, wn = sel(q), sel(k), sel(v), sel(dy), _np(w)[h:h + 1]
        y_ref = oracle.recurrence_forward(qn, kn, vn, wn)
        ref = oracle.recurrence_backward(qn, kn, vn, wn, dyn, want_dw=True)
        for name, got, exp in (("Y", sel(y), y_ref), ("dQ", sel(dq), ref[0]), ("dK", sel(dk), ref[1]),
                               ("dV", sel(dv), ref[2]), ("dW", _np(dw)[h:h + 1], ref[3])):
            err = oracle.rel_l2(got, exp)
            print("head %d %s rel L2 %.3e" % (h, name, err))
            assert err <= 2e-2, (h, name, err)
