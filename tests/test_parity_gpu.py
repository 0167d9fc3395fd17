"""GPU parity: the CUDA library against the fp64 oracle, element by element.

Bars (relative L2 over the whole tensor, computed in fp64, as the gradient
discrepancy of "Sub-Linear Memory: How to Make Performers SLiM", section 4):
  fp32 I/O: <= 1e-4 on Y, dQ, dK, dV and dW;
  bf16 I/O with fp32 accumulation: <= 2e-2 on the same tensors.
Small cases compare every head against the oracle; the full-size workloads
run at full size on the GPU, exactly as the benchmark calls them, and compare
every head (4k and 32k rows, with dW) or sampled (b, h) heads (the 2^20-row
and the elu+1 workload; heads are independent, so a head is an exact unit).
"""
import numpy as np
import pytest
import torch

import oracle
from sub_linear_memory_gb300 import inputs

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}


@pytest.fixture(scope="module", autouse=True)
def _lib():
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


def _wnp(w):
    return None if w is None else _np(w)


def run_library(q, k, v, w, dy, chunk, want_dw=True):
    from sub_linear_memory_gb300 import binding

    y = binding.slim_attn_fwd(q, k, v, w, chunk)
    dq, dk, dv, dw = binding.slim_attn_bwd(q, k, v, w, dy, chunk, want_dw=want_dw)
    binding.sync_status()
    return y, dq, dk, dv, dw


def check(name, got, ref, tol, floor=0.0):
    """Relative L2 error; ``floor`` bounds the denominator from below for
    gradients that vanish identically (e.g. dQ, dK at L = 1, where Y_1 = V_1)."""
    den = max(float(np.linalg.norm(np.ravel(ref))), floor)
    err = float(np.linalg.norm(np.ravel(np.asarray(got, np.float64) - ref))) / den
    print("%s rel L2 %.3e (tol %.0e)" % (name, err, tol))
    assert np.isfinite(err) and err <= tol, "%s: rel L2 %.3e > %.1e" % (name, err, tol)
    return err


def small_case(B, H, L, d, M, C, dtype, feature, seed=0):
    base = inputs.WORKLOADS["tiny" if dtype == torch.float32 else "l4k"]
    wl = base.with_(B=B, H=H, L=L, d=d, M=M, chunk=C, index=100 + seed,
                    dtype="fp32" if dtype == torch.float32 else "bf16", feature=feature,
                    qk_scale=(1.0 if feature == "elu" else d ** -0.25),
                    w_kind=("none" if feature == "elu" else base.w_kind))
    q, k, v, dy, w = inputs.make_inputs(wl)
    dev = "cuda"
    return (q.to(dev), k.to(dev), v.to(dev), dy.to(dev), None if w is None else w.to(dev))


def compare_all(q, k, v, w, dy, chunk, tol, want_dw=True):
    y, dq, dk, dv, dw = run_library(q, k, v, w, dy, chunk, want_dw)
    qn, kn, vn, dyn, wn = _np(q), _np(k), _np(v), _np(dy), _wnp(w)
    y_ref = oracle.recurrence_forward(qn, kn, vn, wn)
    dq_ref, dk_ref, dv_ref, dw_ref = oracle.recurrence_backward(qn, kn, vn, wn, dyn,
                                                                want_dw=want_dw)
    # only at L = 1 do dQ, dK vanish identically (Y_1 = V_1): there the error
    # is bounded against the size of dY instead of the zero reference
    floor = 1e-2 * float(np.linalg.norm(dyn.ravel())) if q.shape[2] == 1 else 0.0
    errs = {"Y": check("Y", _np(y), y_ref, tol)}
    errs["dQ"] = check("dQ", _np(dq), dq_ref, tol, floor)
    errs["dK"] = check("dK", _np(dk), dk_ref, tol, floor)
    errs["dV"] = check("dV", _np(dv), dv_ref, tol, floor)
    if want_dw and w is not None:
        errs["dW"] = check("dW", _np(dw), dw_ref, tol)
    return errs


SMALL = [
    # (B, H, L, d, M, C, feature)    -- several chunks + a ragged tail
    (1, 1, 256, 16, 32, 32, "favor"),      # the tiny workload, full size
    (1, 1, 250, 16, 32, 32, "favor"),      # ragged last chunk
    (1, 1, 20, 16, 32, 32, "favor"),       # L < chunk
    (1, 3, 17, 16, 16, 16, "favor"),       # one full chunk + a 1-row tail
    (2, 2, 1000, 64, 128, 64, "favor"),    # the 4k workload's head shape
    (1, 2, 700, 64, 256, 128, "favor"),    # the 32k workload's head shape
    (1, 1, 1500, 64, 64, 256, "favor"),    # the 1M workload's head shape
    (1, 2, 300, 128, 128, 64, "elu"),      # elu+1, M = d = 128
    (1, 1, 200, 32, 32, 16, "elu"),
]


def check_tiles(name, got, ref, tol):
    """Error of every 128-row tile of every head on its own, over the RMS tile
    norm of the reference: a whole tensor's norm cannot see one wrong tile
    among thousands.  (Over the tile's own norm it would flag rows whose
    exact dK is a small difference of large bf16-rounded terms; at l32k
    head 0, tile 66, that reads 0.27 for correct code.)"""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    B, H, L, d = ref.shape
    nt, full = (L + 127) // 128, L // 128
    parts = [(got[:, :, :full * 128].reshape(B, H, full, 128 * d), ref[:, :, :full * 128].reshape(B, H, full, 128 * d))]
    if full < nt:
        parts.append((got[:, :, full * 128:].reshape(B, H, 1, -1), ref[:, :, full * 128:].reshape(B, H, 1, -1)))
    num = np.concatenate([np.linalg.norm(g - r, axis=3) for g, r in parts], axis=2)
    den = np.concatenate([np.linalg.norm(r, axis=3) for _, r in parts], axis=2)
    err = num / np.sqrt(np.mean(den ** 2))
    worst = float(err.max())
    at = np.unravel_index(int(err.argmax()), err.shape)
    print("%s worst tile error / RMS tile norm %.3e at (b, h, tile) %s (tol %.2f)"
          % (name, worst, tuple(int(x) for x in at), tol))
    assert np.isfinite(worst) and worst <= tol, "%s: tile %s error %.3e of the RMS tile norm > %.2f" % (name, at, worst, tol)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["fp32", "bf16"])
@pytest.mark.parametrize("case", SMALL, ids=lambda c: "x".join(map(str, c)))
def test_small_against_oracle(case, dtype):
    B, H, L, d, M, C, feature = case
    q, k, v, dy, w = small_case(B, H, L, d, M, C, dtype, feature)
    compare_all(q, k, v, w, dy, C, TOL[dtype])


@pytest.mark.parametrize("case", SMALL, ids=lambda c: "x".join(map(str, c)))
def test_small_bf16_cuda_core_family(case, _lib):
    """The CUDA-core kernels on bf16 I/O (the tensor-core kernels take the
    supported shapes by default)."""
    B, H, L, d, M, C, feature = case
    q, k, v, dy, w = small_case(B, H, L, d, M, C, torch.bfloat16, feature)
    _lib.set_option(_lib.OPT_PATH, 1)
    try:
        compare_all(q, k, v, w, dy, C, TOL[torch.bfloat16])
    finally:
        _lib.set_option(_lib.OPT_PATH, 0)


TC_SHAPES = [
    # (B, H, L, d, M, C, feature): shapes the tensor-core forward takes
    (1, 2, 700, 64, 256, 128, "favor"),
    (2, 1, 1000, 64, 128, 64, "favor"),
    (1, 1, 1500, 64, 64, 256, "favor"),
    (1, 2, 300, 128, 128, 64, "elu"),
    (1, 1, 333, 64, 64, 128, "elu"),
    (1, 3, 128, 64, 256, 128, "favor"),   # exactly one tile
    (1, 1, 1, 64, 128, 64, "favor"),      # one row
]


@pytest.mark.parametrize("case", TC_SHAPES, ids=lambda c: "x".join(map(str, c)))
def test_tensor_core_forward_is_used_and_matches(case, _lib):
    B, H, L, d, M, C, feature = case
    q, k, v, dy, w = small_case(B, H, L, d, M, C, torch.bfloat16, feature, seed=7)
    _lib.profile_reset()
    _lib.profile_enable(True)
    try:
        y = _lib.slim_attn_fwd(q, k, v, w, C)
        _lib.sync_status()
        names = set(_lib.profile_read())
    finally:
        _lib.profile_enable(False)
    assert "tc_forward" in names, names
    y_ref = oracle.recurrence_forward(_np(q), _np(k), _np(v), _wnp(w))
    check("Y", _np(y), y_ref, TOL[torch.bfloat16])


TC_BWD_SHAPES = [
    # (B, H, L, d, M, C, feature): shapes the tensor-core backward takes
    (2, 2, 1000, 64, 128, 64, "favor"),
    (1, 1, 1500, 64, 64, 256, "favor"),
    (1, 2, 333, 64, 64, 128, "elu"),
    (1, 3, 128, 64, 128, 128, "favor"),   # exactly one tile
    (1, 2, 129, 64, 64, 128, "favor"),    # one tile + a 1-row tail
    (1, 2, 700, 64, 256, 128, "favor"),   # M = 256: a two-CTA cluster per segment
    (2, 1, 300, 64, 256, 64, "favor"),
    (1, 2, 300, 128, 128, 64, "elu"),     # elu+1 at d = 128: value columns split over a pair
    (2, 1, 1000, 128, 128, 128, "elu"),
    (1, 1, 1, 128, 128, 64, "elu"),       # one row
]


def _run_profiled(_lib, fn):
    _lib.profile_reset()
    _lib.profile_enable(True)
    try:
        out = fn()
        _lib.sync_status()
        names = set(_lib.profile_read())
    finally:
        _lib.profile_enable(False)
    return out, names


@pytest.mark.parametrize("case", TC_BWD_SHAPES, ids=lambda c: "x".join(map(str, c)))
def test_tensor_core_backward_is_used_and_matches(case, _lib):
    B, H, L, d, M, C, feature = case
    q, k, v, dy, w = small_case(B, H, L, d, M, C, torch.bfloat16, feature, seed=9)
    (dq, dk, dv, _), names = _run_profiled(_lib, lambda: _lib.slim_attn_bwd(q, k, v, w, dy, C))
    assert "tc_backward" in names, names
    qn, kn, vn, dyn, wn = _np(q), _np(k), _np(v), _np(dy), _wnp(w)
    ref = oracle.recurrence_backward(qn, kn, vn, wn, dyn, want_dw=False)
    floor = 1e-2 * float(np.linalg.norm(dyn.ravel())) if L == 1 else 0.0
    for name, got, exp in (("dQ", dq, ref[0]), ("dK", dk, ref[1]), ("dV", dv, ref[2])):
        check(name, _np(got), exp, TOL[torch.bfloat16], floor)


@pytest.mark.parametrize("M", [128, 256])
@pytest.mark.parametrize("segments", [1, 2, 3, 6])
def test_tensor_core_backward_segments(segments, M, _lib):
    """Segments > 1 exercise the correction of dK, dV by the later segments' G."""
    q, k, v, dy, w = small_case(1, 2, 1300, 64, M, 128, torch.bfloat16, "favor", seed=10)
    _lib.set_option(_lib.OPT_SEGMENTS, segments)
    try:
        (dq, dk, dv, _), names = _run_profiled(_lib, lambda: _lib.slim_attn_bwd(q, k, v, w, dy, 128))
    finally:
        _lib.set_option(_lib.OPT_SEGMENTS, 0)
    assert "tc_backward" in names
    if segments > 1:
        assert "tc_backward_fix" in names
    ref = oracle.recurrence_backward(_np(q), _np(k), _np(v), _wnp(w), _np(dy), want_dw=False)
    for name, got, exp in (("dQ", dq, ref[0]), ("dK", dk, ref[1]), ("dV", dv, ref[2])):
        check(name, _np(got), exp, TOL[torch.bfloat16])


@pytest.mark.parametrize("M", [64, 128, 256])
@pytest.mark.parametrize("segments", [1, 3])
def test_tensor_core_dw(segments, M, _lib):
    """Learnable W on the tensor path: each tile's X^T u from the backward
    kernel, plus (segments > 1) the later segments' reverse-state share."""
    q, k, v, dy, w = small_case(1, 2, 1300, 64, M, 128, torch.bfloat16, "favor", seed=12)
    _lib.set_option(_lib.OPT_SEGMENTS, segments)
    try:
        (dq, dk, dv, dw), names = _run_profiled(
            _lib, lambda: _lib.slim_attn_bwd(q, k, v, w, dy, 128, want_dw=True))
    finally:
        _lib.set_option(_lib.OPT_SEGMENTS, 0)
    assert "tc_backward" in names and "reduce_dw" in names, names
    if segments > 1:
        assert "tc_dw_fix" in names, names
    ref = oracle.recurrence_backward(_np(q), _np(k), _np(v), _wnp(w), _np(dy), want_dw=True)
    for name, got, exp in zip(("dQ", "dK", "dV", "dW"), (dq, dk, dv, dw), ref):
        check(name, _np(got), exp, TOL[torch.bfloat16])


@pytest.mark.parametrize("segments", [1, 2, 4])
def test_tensor_core_backward_elu128_segments(segments, _lib):
    """elu+1 at d = 128: segments > 1 exercise the correction of dK, dV."""
    q, k, v, dy, w = small_case(1, 2, 1100, 128, 128, 64, torch.bfloat16, "elu", seed=13)
    _lib.set_option(_lib.OPT_SEGMENTS, segments)
    try:
        (dq, dk, dv, _), names = _run_profiled(_lib, lambda: _lib.slim_attn_bwd(q, k, v, w, dy, 64))
    finally:
        _lib.set_option(_lib.OPT_SEGMENTS, 0)
    assert "tc_backward" in names, names
    if segments > 1:
        assert "tc_backward_fix" in names, names
    ref = oracle.recurrence_backward(_np(q), _np(k), _np(v), None, _np(dy), want_dw=False)
    for name, got, exp in (("dQ", dq, ref[0]), ("dK", dk, ref[1]), ("dV", dv, ref[2])):
        check(name, _np(got), exp, TOL[torch.bfloat16])


def test_tensor_core_backward_long_reversal(_lib):
    """One segment of 160 tiles: the backward removes each tile's state
    increment in turn (eq. (19)); the double-float state keeps the early
    tiles' small states exact."""
    q, k, v, dy, w = small_case(1, 1, 160 * 128, 64, 64, 128, torch.bfloat16, "favor", seed=11)
    _lib.set_option(_lib.OPT_SEGMENTS, 1)
    try:
        (dq, dk, dv, _), names = _run_profiled(_lib, lambda: _lib.slim_attn_bwd(q, k, v, w, dy, 128))
    finally:
        _lib.set_option(_lib.OPT_SEGMENTS, 0)
    assert "tc_backward" in names
    ref = oracle.recurrence_backward(_np(q), _np(k), _np(v), _wnp(w), _np(dy), want_dw=False)
    for name, got, exp in (("dQ", dq, ref[0]), ("dK", dk, ref[1]), ("dV", dv, ref[2])):
        check(name, _np(got), exp, TOL[torch.bfloat16])
    # the first tile, where the recovered state is smallest relative to the
    # total: exact reversal keeps it at the level of bf16 rounding (about
    # 6e-3 here), well inside the contract bar; rounding in the segment total
    # would show up first in this tile
    for name, got, exp in (("dQ[:128]", dq, ref[0]), ("dK[:128]", dk, ref[1])):
        check(name, _np(got)[..., :128, :], exp[..., :128, :], 1e-2)


@pytest.mark.parametrize("segments", [1, 2, 3, 5])
def test_tensor_core_segments(segments, _lib):
    q, k, v, dy, w = small_case(1, 2, 1100, 64, 256, 128, torch.bfloat16, "favor", seed=8)
    _lib.set_option(_lib.OPT_SEGMENTS, segments)
    try:
        y = _lib.slim_attn_fwd(q, k, v, w, 128)
        _lib.sync_status()
    finally:
        _lib.set_option(_lib.OPT_SEGMENTS, 0)
    y_ref = oracle.recurrence_forward(_np(q), _np(k), _np(v), _wnp(w))
    check("Y", _np(y), y_ref, TOL[torch.bfloat16])


@pytest.mark.parametrize("dtype,d,M,C", [(torch.float32, 16, 32, 16), (torch.bfloat16, 16, 32, 16),
                                         (torch.bfloat16, 64, 128, 64)],
                         ids=["fp32", "bf16", "bf16-tensor-core"])
def test_single_row(dtype, d, M, C):
    """L = 1: Y_1 = V_1, dV_1 = dY_1, and dQ = dK = dW = 0 (Y_1 does not depend
    on Q or K), so only rounding noise may remain there."""
    q, k, v, dy, w = small_case(2, 3, 1, d, M, C, dtype, "favor", seed=6)
    y, dq, dk, dv, dw = run_library(q, k, v, w, dy, C, want_dw=(d == 16))
    tol = TOL[dtype]
    check("Y", _np(y), _np(v), tol)
    check("dV", _np(dv), _np(dy), tol)
    scale = float(np.linalg.norm(_np(dy).ravel())) * (1.0 + float(np.linalg.norm(_np(w))))
    for name, t in (("dQ", dq), ("dK", dk), ("dW", dw)):
        if t is not None:
            assert float(np.linalg.norm(_np(t).ravel())) <= tol * scale, name


@pytest.mark.parametrize("segments", [1, 2, 3, 7])
def test_segment_count_does_not_change_results(segments, _lib):
    q, k, v, dy, w = small_case(1, 2, 900, 32, 64, 32, torch.float32, "favor", seed=3)
    _lib.set_option(_lib.OPT_SEGMENTS, segments)
    try:
        compare_all(q, k, v, w, dy, 32, 1e-4)
    finally:
        _lib.set_option(_lib.OPT_SEGMENTS, 0)


@pytest.mark.parametrize("chunk", [16, 32, 64, 128, 256])
def test_chunk_invariance(chunk):
    """Any slice size C gives the same attention (the paper's Algorithm 1 is
    exact for every C; section 3.4)."""
    q, k, v, dy, w = small_case(1, 2, 600, 32, 64, chunk, torch.float32, "favor", seed=4)
    compare_all(q, k, v, w, dy, chunk, 1e-4)


def test_outputs_do_not_depend_on_stale_workspace(_lib):
    q, k, v, dy, w = small_case(1, 1, 300, 16, 32, 32, torch.float32, "favor", seed=5)
    first = run_library(q, k, v, w, dy, 32)
    second = run_library(q, k, v, w, dy, 32)
    for a, b in zip(first, second):
        assert torch.equal(a, b)


@pytest.mark.parametrize("M", [64, 128, 256])
def test_long_segments_repeat_cleanly(M, _lib):
    """Many tiles per CTA and every SM busy: the 1M-row workload's head shape
    at 2^18 rows (and the same with 256 features), thirty fwd + bwd runs in a
    row.  Each must end with a clean device status (a barrier wait that gives
    up raises here) and, with 64 features, give bit-identical outputs: with
    one CTA per segment every output element is stored once and corrected at
    most once.  A forward whose load slots rotated through K, Q and V tiles
    let a consumer read a slot before its load landed about once in three
    such runs, one 128-row tile of Y wrong: far too little for the
    whole-head relative L2 bar to see."""
    wl = inputs.WORKLOADS["l1m"].with_(L=1 << 18, M=M, index=300 + M)
    q, k, v, dy, w = inputs.make_inputs(wl, device="cuda")
    first = run_library(q, k, v, w, dy, wl.chunk, want_dw=False)
    deterministic = M <= 128  # 256 features: a CTA pair adds its two partials in either order
    for _ in range(29):
        again = run_library(q, k, v, w, dy, wl.chunk, want_dw=False)
        if deterministic:
            for a, b in zip(first[:4], again[:4]):
                assert torch.equal(a, b)
    if not deterministic:
        for a, b in zip(first[:4], again[:4]):
            d = (a.float() - b.float()).norm() / b.float().norm()
            assert d <= 1e-2, float(d)


def test_elu128_forward_repeats_bit_identical(_lib):
    """elu+1 with d = M = 128 over 2^16 rows per head, every SM busy: the
    forward (whose segment-state pass puts K and V in slots of their own)
    gives bit-identical Y over twenty runs, and no run reports a device
    error.  The backward's CTA pair adds its dQ, dK shares in either order,
    so only its status is checked."""
    wl = inputs.WORKLOADS["elu16k"].with_(B=1, H=8, L=1 << 16, index=410)
    q, k, v, dy, w = inputs.make_inputs(wl, device="cuda")
    first = run_library(q, k, v, w, dy, wl.chunk, want_dw=False)
    for _ in range(19):
        again = run_library(q, k, v, w, dy, wl.chunk, want_dw=False)
        assert torch.equal(first[0], again[0])


# ---- full-size workloads: sampled heads ----------------------------------

FULL = {
    # name: (sampled (b, h) heads or None for every head, also check dW)
    "l4k": (None, True),
    "l32k": (None, True),
    "l1m": ([(0, 3)], False),
    "elu16k": ([(0, 0), (3, 11)], False),
}


@pytest.mark.parametrize("name", list(FULL))
def test_full_size_workload(name):
    wl = inputs.WORKLOADS[name]
    q, k, v, dy, w = inputs.make_inputs(wl, device="cuda")
    heads, dw_too = FULL[name]
    want_dw = dw_too and w is not None
    y, dq, dk, dv, dw = run_library(q, k, v, w, dy, wl.chunk, want_dw=want_dw)
    tol = TOL[wl.torch_dtype]
    if heads is None:
        sel = lambda t: _np(t)
    else:
        idx_b = torch.tensor([b for b, _ in heads])
        idx_h = torch.tensor([h for _, h in heads])
        sel = lambda t: _np(t[idx_b, idx_h].unsqueeze(0))
    qn, kn, vn, dyn, wn = sel(q), sel(k), sel(v), sel(dy), _wnp(w)
    # every tile on its own too: a tile read before its load landed is off
    # by about its own norm; correct bf16 tiles stay below 0.14 of the RMS
    # tile norm on these workloads
    tile_tol = 0.25 if wl.torch_dtype == torch.bfloat16 else 1e-3
    y_ref = oracle.recurrence_forward(qn, kn, vn, wn)
    check("Y", sel(y), y_ref, tol)
    check_tiles("Y", sel(y), y_ref, tile_tol)
    del y_ref
    dq_ref, dk_ref, dv_ref, dw_ref = oracle.recurrence_backward(qn, kn, vn, wn, dyn, want_dw=want_dw)
    for name, got, ref in (("dQ", dq, dq_ref), ("dK", dk, dk_ref), ("dV", dv, dv_ref)):
        check(name, sel(got), ref, tol)
        check_tiles(name, sel(got), ref, tile_tol)
    if want_dw:
        check("dW", _np(dw), dw_ref, tol)


@pytest.mark.parametrize("chunk", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("M", [128, 256])
def test_chunk_invariance_tensor_path(chunk, M, _lib):
    """Every slice size C runs on the tensor-core kernels (they work on
    128-row tiles whatever C is; the slice recurrence is exact for any C,
    section 3.4) and matches the oracle at the bf16 bar."""
    q, k, v, dy, w = small_case(1, 2, 900, 64, M, chunk, torch.bfloat16, "favor", seed=14)

    def both():
        y = _lib.slim_attn_fwd(q, k, v, w, chunk)
        return (y,) + _lib.slim_attn_bwd(q, k, v, w, dy, chunk, want_dw=True)

    (y, dq, dk, dv, dw), names = _run_profiled(_lib, both)
    assert "tc_forward" in names and "tc_backward" in names, names
    qn, kn, vn, dyn, wn = _np(q), _np(k), _np(v), _np(dy), _wnp(w)
    check("Y", _np(y), oracle.recurrence_forward(qn, kn, vn, wn), TOL[torch.bfloat16])
    ref = oracle.recurrence_backward(qn, kn, vn, wn, dyn, want_dw=True)
    for name, got, exp in zip(("dQ", "dK", "dV", "dW"), (dq, dk, dv, dw), ref):
        check(name, _np(got), exp, TOL[torch.bfloat16])


@pytest.mark.parametrize("chunk", [16, 32])
def test_small_chunks_elu128_tensor_path(chunk, _lib):
    q, k, v, dy, w = small_case(1, 2, 700, 128, 128, chunk, torch.bfloat16, "elu", seed=15)

    def both():
        y = _lib.slim_attn_fwd(q, k, v, w, chunk)
        return (y,) + _lib.slim_attn_bwd(q, k, v, w, dy, chunk)

    (y, dq, dk, dv, _), names = _run_profiled(_lib, both)
    assert "tc_forward" in names and "tc_backward" in names, names
    qn, kn, vn, dyn = _np(q), _np(k), _np(v), _np(dy)
    check("Y", _np(y), oracle.recurrence_forward(qn, kn, vn, None), TOL[torch.bfloat16])
    ref = oracle.recurrence_backward(qn, kn, vn, None, dyn, want_dw=False)
    for name, got, exp in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
        check(name, _np(got), exp, TOL[torch.bfloat16])
