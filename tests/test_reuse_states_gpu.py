"""Forward-to-backward reuse of the boundary states (SLIM_OPT_REUSE_STATES)
against the fp64 oracle ("Sub-Linear Memory: How to Make Performers SLiM",
section 3.2: the forward keeps the states at the slice boundaries; section
3.3: the backward rebuilds every other state from them).

* with the option on, the backward after a matching forward runs no state
  pass of its own (the per-kernel profile shows one segment-state launch per
  forward and backward pair) and still matches the oracle on every kernel
  layout: one CTA and the two-CTA pair, elu+1, dW, one W per head;
* a backward whose k differs from the forward's, that follows another call on
  the workspace, or whose own segments differ from the forward's, recomputes
  the states and matches the oracle for its own inputs.
"""
import numpy as np
import pytest
import torch

import oracle
from sub_linear_memory_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from sub_linear_memory_gb300 import binding

    for opt in (binding.OPT_SEGMENTS, binding.OPT_PATH, binding.OPT_W_PER_HEAD, binding.OPT_REUSE_STATES):
        binding.set_option(opt, 0)
    yield binding
    for opt in (binding.OPT_SEGMENTS, binding.OPT_PATH, binding.OPT_W_PER_HEAD, binding.OPT_REUSE_STATES):
        binding.set_option(opt, 0)
    binding.profile_enable(False)


def _np(t):
    return t.detach().to("cpu", torch.float64).numpy()


def _case(B, H, L, M, feature, seed):
    wl = inputs.WORKLOADS["l4k"].with_(B=B, H=H, L=L, d=64, M=M, chunk=128, index=2000 + seed, feature=feature,
                                       w_kind="orf" if feature == "favor" else "none", qk_scale=64 ** -0.25)
    q, k, v, dy, w = (None if t is None else t.cuda() for t in inputs.make_inputs(wl))
    return q, k, v, dy, w


def _compare(got, ref, tol=2e-2):
    for name, g, r in zip(("Y", "dQ", "dK", "dV", "dW"), got, ref):
        if g is None:
            continue
        err = oracle.rel_l2(_np(g), r)
        print("%s rel L2 %.3e" % (name, err))
        assert err <= tol, (name, err)


def _profiled(lib, fn):
    lib.profile_enable(True)
    lib.profile_reset()
    try:
        out = fn()
        lib.sync_status()
        prof = lib.profile_read()
    finally:
        lib.profile_enable(False)
    return out, prof


CASES = [
    # (B, H, L, M, feature, segments, want_dw)
    (2, 2, 1000, 256, "favor", 0, False),   # two-CTA backward: it zeroes its outputs, then reduce-adds
    (1, 3, 1300, 256, "favor", 4, True),
    (2, 2, 900, 128, "favor", 3, True),     # one CTA per segment
    (1, 2, 700, 64, "favor", 0, False),
    (2, 2, 1100, 64, "elu", 5, False),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(str(x) for x in c[:4]) + "-%s-P%d%s" % (
    c[4], c[5], "-dW" if c[6] else ""))
def test_backward_reads_forward_states(case, lib):
    B, H, L, M, feature, segments, want_dw = case
    q, k, v, dy, w = _case(B, H, L, M, feature, seed=segments)
    lib.set_option(lib.OPT_SEGMENTS, segments)
    lib.set_option(lib.OPT_REUSE_STATES, 1)
    try:
        lib.slim_attn_fwd(q, k, v, w, 128)  # sizes the workspace for both calls
        lib.slim_attn_bwd(q, k, v, w, dy, 128, want_dw=want_dw)

        def step():
            y = lib.slim_attn_fwd(q, k, v, w, 128)
            return (y,) + tuple(lib.slim_attn_bwd(q, k, v, w, dy, 128, want_dw=want_dw))

        out, prof = _profiled(lib, step)
    finally:
        lib.set_option(lib.OPT_REUSE_STATES, 0)
        lib.set_option(lib.OPT_SEGMENTS, 0)
    print(prof)
    assert prof["tc_forward"][0] == 1 and prof["tc_backward"][0] == 1, prof
    assert prof["tc_segment_state"][0] == 1, prof  # the forward's, read again by the backward
    # the W image too: the backward reads the forward's, at the same workspace offset
    assert prof.get("prep_w", (0,))[0] == (1 if feature == "favor" else 0), prof
    qn, kn, vn, dyn = _np(q), _np(k), _np(v), _np(dy)
    wn = None if w is None else _np(w)
    y_ref = oracle.recurrence_forward(qn, kn, vn, wn)
    ref = oracle.recurrence_backward(qn, kn, vn, wn, dyn, want_dw=want_dw)
    _compare(out, (y_ref,) + tuple(ref[:4]))


def test_per_head_w_reuse(lib):
    B, H, L, M = 2, 3, 800, 256
    q, k, v, dy, _ = _case(B, H, L, M, "favor", seed=11)
    w = lib.draw_orf(H, 64, M, seed=21, step=2)
    lib.set_option(lib.OPT_W_PER_HEAD, 1)
    lib.set_option(lib.OPT_REUSE_STATES, 1)
    try:
        lib.slim_attn_fwd(q, k, v, w, 128)
        lib.slim_attn_bwd(q, k, v, w, dy, 128, want_dw=True)

        def step():
            y = lib.slim_attn_fwd(q, k, v, w, 128)
            return (y,) + tuple(lib.slim_attn_bwd(q, k, v, w, dy, 128, want_dw=True))

        out, prof = _profiled(lib, step)
    finally:
        lib.set_option(lib.OPT_REUSE_STATES, 0)
        lib.set_option(lib.OPT_W_PER_HEAD, 0)
    assert prof["tc_segment_state"][0] == 1, prof
    assert prof["prep_w"][0] == 1, prof
    qn, kn, vn, dyn, wn = _np(q), _np(k), _np(v), _np(dy), _np(w)
    y_ref = oracle.recurrence_forward(qn, kn, vn, wn)
    ref = oracle.recurrence_backward(qn, kn, vn, wn, dyn, want_dw=True)
    _compare(out, (y_ref,) + tuple(ref[:4]))


@pytest.mark.parametrize("between", ["other_k", "state_call", "option_cycled"])
def test_mismatch_recomputes(between, lib):
    B, H, L, M = 1, 2, 900, 256
    q, k, v, dy, w = _case(B, H, L, M, "favor", seed=31)
    k2 = (k.float() * 0.5).to(torch.bfloat16)  # another K: the backward must not take k's states
    lib.set_option(lib.OPT_REUSE_STATES, 1)
    try:
        lib.slim_attn_fwd(q, k, v, w, 128)
        lib.slim_attn_bwd(q, k, v, w, dy, 128)

        def step():
            lib.slim_attn_fwd(q, k, v, w, 128)
            kb = k
            if between == "other_k":
                kb = k2
            elif between == "state_call":
                lib.slim_attn_state(k2, v, w, 128)
            else:
                lib.set_option(lib.OPT_REUSE_STATES, 0)
                lib.set_option(lib.OPT_REUSE_STATES, 1)
            return kb, lib.slim_attn_bwd(q, kb, v, w, dy, 128)

        (kb, grads), prof = _profiled(lib, step)
    finally:
        lib.set_option(lib.OPT_REUSE_STATES, 0)
    expect = 2 if between != "state_call" else 3  # forward, (state call,) backward
    assert prof["tc_segment_state"][0] == expect, prof
    assert prof["prep_w"][0] == expect, prof  # each state pass makes its own W image
    qn, kn, vn, dyn, wn = _np(q), _np(kb), _np(v), _np(dy), _np(w)
    ref = oracle.recurrence_backward(qn, kn, vn, wn, dyn, want_dw=False)
    _compare(grads[:3], ref[:3])


def test_declined_when_segments_differ(lib):
    """40000 rows of one head at M = 256: on 152 SMs the forward plans 105
    segments of 3 tiles and the two-CTA backward 63 of 5, so the forward
    leaves no tagged states and the backward runs its own state pass."""
    B, H, L, M = 1, 1, 40000, 256
    q, k, v, dy, w = _case(B, H, L, M, "favor", seed=41)
    lib.set_option(lib.OPT_REUSE_STATES, 1)
    try:
        lib.slim_attn_fwd(q, k, v, w, 128)
        lib.slim_attn_bwd(q, k, v, w, dy, 128)

        def step():
            lib.slim_attn_fwd(q, k, v, w, 128)
            return lib.slim_attn_bwd(q, k, v, w, dy, 128)

        grads, prof = _profiled(lib, step)
    finally:
        lib.set_option(lib.OPT_REUSE_STATES, 0)
    assert prof["tc_segment_state"][0] == 2, prof
    qn, kn, vn, dyn, wn = _np(q), _np(k), _np(v), _np(dy), _np(w)
    ref = oracle.recurrence_backward(qn, kn, vn, wn, dyn, want_dw=False)
    _compare(grads[:3], ref[:3])

