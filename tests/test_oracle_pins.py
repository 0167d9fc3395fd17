"""Pins for the fp64 oracle against what the mathematics fixes (CPU only).

Source throughout: "Sub-Linear Memory: How to Make Performers SLiM",
section 2.1, eq. (1)-(4) (exponential and linear causal attention, prefix-sum
form) and section 3.3 (the gradient through a prefix sum is a backward prefix
sum).  Each test is chosen so that a plausible slip in the oracle -- a dropped
diagonal, a sign in the feature map, a transposed W, a missing normaliser
term, a wrong reverse-sweep index -- fails at least one of them.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import quadratic

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(rng, b, h, length, d, m, favor=True, qk_scale=None):
    s = d ** -0.25 if qk_scale is None else qk_scale
    q = rng.standard_normal((b, h, length, d)) * s
    k = rng.standard_normal((b, h, length, d)) * s
    v = rng.standard_normal((b, h, length, d))
    dy = rng.standard_normal((b, h, length, d))
    w = rng.standard_normal((d, m)) if favor else None
    return q, k, v, dy, w


def _val(x):
    if isinstance(x, str):
        env = {"exp": math.exp, "sqrt": math.sqrt, "log": math.log}
        try:
            return float(Fraction(x))
        except ValueError:
            return float(eval(x, {"__builtins__": {}}, env))  # closed-form fixture expression
    return float(x)


def _arr(rows):
    return np.array([[_val(x) for x in row] for row in rows], dtype=np.float64)


SHAPES = [(1, 1, 1, 4, 8), (1, 2, 9, 3, 5), (2, 1, 17, 8, 16), (1, 1, 33, 16, 32)]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("favor", [True, False])
def test_recurrence_equals_quadratic_form(shape, favor):
    """P-a: eq. (3)-(4) prefix-sum recurrence == eq. (2) quadratic form, fwd and bwd."""
    b, h, length, d, m = shape
    rng = np.random.default_rng(hash((shape, favor)) % 2**32)
    q, k, v, dy, w = _rand(rng, b, h, length, d, m if favor else d, favor)
    y_rec = oracle.recurrence_forward(q, k, v, w)
    y_quad = quadratic.forward(q, k, v, w)
    assert oracle.rel_l2(y_rec, y_quad) < 1e-12
    g_rec = oracle.recurrence_backward(q, k, v, w, dy)
    g_quad = quadratic.backward(q, k, v, w, dy)
    for a, ref in zip(g_rec, g_quad):
        if ref is None:
            assert a is None
            continue
        # L = 1 has Y_1 = V_1, so dQ = dK = 0 there: compare against the scale of the inputs
        err = np.linalg.norm((a - ref).ravel())
        assert err <= 1e-12 * max(np.linalg.norm(ref.ravel()), 1.0)


def test_backward_returns_forward_output():
    rng = np.random.default_rng(3)
    q, k, v, dy, w = _rand(rng, 1, 2, 11, 4, 8)
    *_, y = oracle.recurrence_backward(q, k, v, w, dy, want_y=True)
    assert oracle.rel_l2(y, oracle.recurrence_forward(q, k, v, w)) < 1e-14


@pytest.mark.parametrize("favor", [True, False])
def test_first_output_is_first_value(favor):
    """P-b: Y_1 = V_1 (a weighted average over one value vector)."""
    rng = np.random.default_rng(5)
    q, k, v, _, w = _rand(rng, 2, 3, 6, 4, 8 if favor else 4, favor)
    for fn in (oracle.recurrence_forward, quadratic.forward):
        y = fn(q, k, v, w)
        np.testing.assert_allclose(y[..., 0, :], v[..., 0, :], rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("favor", [True, False])
def test_constant_values_and_affine_equivariance(favor):
    """P-c: the output row is a convex combination of V_{<=l}."""
    rng = np.random.default_rng(7)
    q, k, v, _, w = _rand(rng, 1, 2, 12, 4, 8 if favor else 4, favor)
    c = np.broadcast_to(rng.standard_normal(4), v.shape).copy()
    np.testing.assert_allclose(oracle.recurrence_forward(q, k, c, w), c, rtol=1e-12, atol=1e-12)
    y = oracle.recurrence_forward(q, k, v, w)
    y2 = oracle.recurrence_forward(q, k, 2.5 * v - 1.25, w)
    np.testing.assert_allclose(y2, 2.5 * y - 1.25, rtol=1e-12, atol=1e-12)
    # inside the coordinatewise hull of the prefix of V
    lo = np.minimum.accumulate(v, axis=-2)
    hi = np.maximum.accumulate(v, axis=-2)
    assert np.all(y >= lo - 1e-12) and np.all(y <= hi + 1e-12)


def test_causality():
    """P-d: Y_l depends only on rows 1..l of Q, K, V."""
    rng = np.random.default_rng(11)
    q, k, v, _, w = _rand(rng, 1, 1, 10, 4, 8)
    y = oracle.recurrence_forward(q, k, v, w)
    cut = 6
    for t in (q, k, v):
        t2 = t.copy()
        t2[..., cut:, :] += rng.standard_normal(t2[..., cut:, :].shape)
        args = [t2 if t is x else x for x in (q, k, v)]
        y2 = oracle.recurrence_forward(*args, w)
        np.testing.assert_array_equal(y2[..., :cut, :], y[..., :cut, :])
        assert not np.allclose(y2[..., cut:, :], y[..., cut:, :])


def _fd_grad(f, x, h=1e-6):
    g = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        i = it.multi_index
        old = x[i]
        x[i] = old + h
        fp = f()
        x[i] = old - h
        fm = f()
        x[i] = old
        g[i] = (fp - fm) / (2 * h)
    return g


@pytest.mark.parametrize("favor", [True, False])
@pytest.mark.parametrize("impl", ["recurrence", "quadratic"])
def test_finite_differences(favor, impl):
    """P-e: analytic gradients of sum(dY * Y) equal central differences (fp64)."""
    rng = np.random.default_rng(13 if favor else 17)
    d, m = 3, (5 if favor else 3)
    q, k, v, dy, w = _rand(rng, 1, 1, 6, d, m, favor)
    fwd = oracle.recurrence_forward if impl == "recurrence" else quadratic.forward
    bwd = oracle.recurrence_backward if impl == "recurrence" else quadratic.backward

    def loss():
        return float(np.sum(dy * fwd(q, k, v, w)))

    dq, dk, dv, dw = bwd(q, k, v, w, dy)
    for x, g in ((q, dq), (k, dk), (v, dv)) + (((w, dw),) if favor else ()):
        fd = _fd_grad(loss, x)
        assert oracle.rel_l2(g, fd) < 1e-6


def test_value_gradient_sums_to_output_gradient():
    """P-f: the weights of each row sum to one, so sum_j dV_j = sum_l dY_l."""
    rng = np.random.default_rng(19)
    q, k, v, dy, w = _rand(rng, 1, 2, 15, 4, 8)
    _, _, dv, _ = oracle.recurrence_backward(q, k, v, w, dy)
    np.testing.assert_allclose(dv.sum(axis=-2), dy.sum(axis=-2), rtol=1e-11, atol=1e-11)


def test_zero_projection_closed_form():
    """W = 0: every feature of a row equals exp(-|x|^2/2)/sqrt(M), so
    Y_l = sum_j e^{-|K_j|^2/2} V_j / sum_j e^{-|K_j|^2/2} (no Q dependence) and
    dQ = 0 (Y is invariant to rescaling g(Q_l))."""
    rng = np.random.default_rng(23)
    q, k, v, dy, _ = _rand(rng, 1, 1, 9, 4, 8)
    w = np.zeros((4, 8))
    wk = np.exp(-0.5 * np.sum(k * k, axis=-1))[..., None]
    expect = np.cumsum(wk * v, axis=-2) / np.cumsum(wk, axis=-2)
    np.testing.assert_allclose(oracle.recurrence_forward(q, k, v, w), expect, rtol=1e-12)
    dq, _, _, _ = oracle.recurrence_backward(q, k, v, w, dy)
    assert np.max(np.abs(dq)) < 1e-12


def test_golden_elu_hand_example():
    """P-j: hand-worked elu+1 example (fixture shows the arithmetic)."""
    with open(os.path.join(GOLDEN, "elu_L3_hand.json")) as f:
        g = json.load(f)
    q, k, v, dy = (_arr(g[n]) for n in ("q", "k", "v", "dy"))
    for fwd in (oracle.recurrence_forward, quadratic.forward):
        np.testing.assert_allclose(fwd(q, k, v, None), _arr(g["y"]), rtol=0, atol=1e-14)
    for bwd in (oracle.recurrence_backward, quadratic.backward):
        dq, dk, dv, dw = bwd(q, k, v, None, dy)
        assert dw is None
        np.testing.assert_allclose(dq, _arr(g["dq"]), rtol=0, atol=1e-14)
        np.testing.assert_allclose(dk, _arr(g["dk"]), rtol=0, atol=1e-14)
        np.testing.assert_allclose(dv, _arr(g["dv"]), rtol=0, atol=1e-14)


def test_golden_favor_hand_example():
    """Hand-worked FAVOR+ features (orientation of W, the -|x|^2/2 term, 1/sqrt(M))."""
    with open(os.path.join(GOLDEN, "favor_L2_hand.json")) as f:
        g = json.load(f)
    w = _arr(g["w"])
    x = _arr(g["feature_rows"])
    np.testing.assert_allclose(oracle.feature_map(x, w), _arr(g["feature_values"]), rtol=1e-14)
    np.testing.assert_allclose(quadratic.feature_map(x, w), _arr(g["feature_values"]), rtol=1e-14)
    q, k, v = _arr(g["q"]), _arr(g["k"]), _arr(g["v"])
    for fwd in (oracle.recurrence_forward, quadratic.forward):
        np.testing.assert_allclose(fwd(q, k, v, w), _arr(g["y"]), rtol=1e-13)


def test_elu_feature_map_closed_form():
    x = np.array([[-2.0, -0.5, 0.0, 0.5, 3.0]])
    expect = np.array([[math.exp(-2.0), math.exp(-0.5), 1.0, 1.5, 4.0]])
    np.testing.assert_allclose(oracle.feature_map(x, None), expect, rtol=1e-15)
    np.testing.assert_allclose(quadratic.feature_map(x, None), expect, rtol=1e-15)


def test_favor_unbiased_for_exponential_kernel():
    """P-h: E_W[g(x).g(y)] = exp(x.y) for W with iid N(0,1) entries
    (Gaussian moment generating function with z = x + y)."""
    rng = np.random.default_rng(29)
    d, m, draws = 3, 64, 400
    x = rng.standard_normal(d) * 0.5
    y = rng.standard_normal(d) * 0.5
    est = []
    for _ in range(draws):
        w = rng.standard_normal((d, m))
        f = oracle.feature_map(np.stack([x, y]), w)
        est.append(float(f[0] @ f[1]))
    est = np.array(est)
    mean, se = est.mean(), est.std(ddof=1) / math.sqrt(draws)
    assert abs(mean - math.exp(x @ y)) < 4 * se


def test_favor_converges_to_softmax_attention():
    """P-i: with random features, Att^lin -> Att^exp as M grows (error ~ M^-1/2)."""
    rng = np.random.default_rng(31)
    d, length = 4, 16
    q = rng.standard_normal((length, d)) * 0.5
    k = rng.standard_normal((length, d)) * 0.5
    v = rng.standard_normal((length, d))
    ref = quadratic.softmax_forward(q, k, v)
    errs = []
    for m in (2 ** 6, 2 ** 11, 2 ** 16):
        e = [oracle.rel_l2(oracle.recurrence_forward(q, k, v, rng.standard_normal((d, m))), ref)
             for _ in range(4)]
        errs.append(float(np.mean(e)))
    assert errs[1] < errs[0] and errs[2] < errs[1]
    assert errs[2] < 0.03
    # 1024x more features: ~32x smaller error in expectation; allow slack for noise
    assert errs[0] / errs[2] > 8


def test_oracle_rejects_bad_arguments():
    rng = np.random.default_rng(37)
    q, k, v, _, _ = _rand(rng, 1, 1, 4, 4, 4, favor=False)
    with pytest.raises(ValueError):
        oracle.recurrence_forward(q[..., :3], k[..., :3], v[..., :3], np.zeros((4, 4)))


# ---- serving form: a carried state, one new row at a time ------------------

@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("favor", [True, False])
def test_decode_chain_equals_quadratic_form(shape, favor):
    """P-d1: decoding rows one by one from the zero state (eq. (3)-(4) per
    step, diagonal included) reproduces every row of the eq. (2) quadratic form."""
    b, h, length, d, m = shape
    rng = np.random.default_rng(7 + hash((shape, favor)) % 2**32)
    q, k, v, _, w = _rand(rng, b, h, length, d, m if favor else d, favor)
    st = np.zeros((b, h, d + 1, m if favor else d))
    ys = np.stack([oracle.decode_step(q[:, :, l], k[:, :, l], v[:, :, l], w, st) for l in range(length)], axis=2)
    assert oracle.rel_l2(ys, quadratic.forward(q, k, v, w)) < 1e-12


@pytest.mark.parametrize("favor", [True, False])
def test_prefill_state_closed_form(favor):
    """P-d2: the state after L rows is [V^T g(K) ; 1^T g(K)], computed here
    with the numpy feature map and a matmul, independently of the C loops."""
    rng = np.random.default_rng(11)
    b, h, length, d, m = 2, 2, 13, 6, 10
    _, k, v, _, w = _rand(rng, b, h, length, d, m if favor else d, favor)
    st = oracle.prefill_state(k, v, w)
    phk = quadratic.feature_map(k, w)
    ref_r = np.einsum("bhle,bhlm->bhem", v, phk)
    ref_s = phk.sum(axis=2)
    assert np.allclose(st[:, :, :d], ref_r, rtol=1e-13, atol=1e-13)
    assert np.allclose(st[:, :, d], ref_s, rtol=1e-13, atol=1e-13)
    assert np.all(oracle.prefill_state(k[:, :, :0], v[:, :, :0], w) == 0.0)


@pytest.mark.parametrize("favor", [True, False])
def test_prefill_then_decode_is_the_next_row(favor):
    """P-d3: prefill over rows < l, then one decode step with row l, gives
    Y_l of the quadratic form (the state carries exactly the rows before l)."""
    rng = np.random.default_rng(12)
    b, h, length, d, m = 1, 3, 20, 8, 16
    q, k, v, _, w = _rand(rng, b, h, length, d, m if favor else d, favor)
    y_quad = quadratic.forward(q, k, v, w)
    for l in (0, 1, 19):
        st = oracle.prefill_state(k[:, :, :l], v[:, :, :l], w)
        y = oracle.decode_step(q[:, :, l], k[:, :, l], v[:, :, l], w, st)
        assert np.allclose(y, y_quad[:, :, l], rtol=1e-12, atol=1e-12)


# ---- carried boundary states (a sequence processed window by window) -------


def _carry_case(rng, favor, length=6, prior=4, b=1, h=2):
    d, m = 3, (5 if favor else 3)
    q, k, v, dy, w = _rand(rng, b, h, length, d, m, favor)
    # a realistic incoming state: the prefix sums of a few earlier rows
    _, kp, vp, _, _ = _rand(rng, b, h, prior, d, m, favor)
    state0 = oracle.prefill_state(kp, vp, w)
    g0 = rng.standard_normal((b, h, d + 1, m)) * 0.3
    return q, k, v, dy, w, state0, g0


@pytest.mark.parametrize("favor", [True, False])
def test_carry_finite_differences(favor):
    """The backward with carried states is the gradient of
    sum(dY * Y) + sum(g0 * R'_L), where the forward starts from state0 and
    R'_L is its final state: central differences in q, k, v, W and state0."""
    rng = np.random.default_rng(41 if favor else 43)
    q, k, v, dy, w, state0, g0 = _carry_case(rng, favor)

    def loss():
        y, s_out = oracle.recurrence_forward(q, k, v, w, state0=state0, return_state=True)
        return float(np.sum(dy * y) + np.sum(g0 * s_out))

    dq, dk, dv, dw, gs = oracle.recurrence_backward(q, k, v, w, dy, state0=state0, g0=g0, want_gstate=True)
    pairs = [(q, dq), (k, dk), (v, dv), (state0, gs)] + ([(w, dw)] if favor else [])
    for x, g in pairs:
        fd = _fd_grad(loss, x)
        assert oracle.rel_l2(g, fd) < 1e-6


@pytest.mark.parametrize("favor", [True, False])
def test_carry_final_state_closed_form(favor):
    """The state after the last row is state0 plus the rows' own prefix sums:
    R'_L = state0 + sum_j [V_j ; 1] (x) g(K_j), summed here directly from the
    feature map."""
    rng = np.random.default_rng(47)
    q, k, v, _, w, state0, _ = _carry_case(rng, favor, length=9)
    _, s_out = oracle.recurrence_forward(q, k, v, w, state0=state0, return_state=True)
    phik = oracle.feature_map(k, w)  # [B, H, L, M]
    vp = np.concatenate([v, np.ones(v.shape[:-1] + (1,))], axis=-1)  # [B, H, L, d + 1]
    expect = state0 + np.einsum("bhle,bhlm->bhem", vp, phik)
    np.testing.assert_allclose(s_out, expect, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("favor", [True, False])
@pytest.mark.parametrize("cut", [1, 7, 12])
def test_windows_with_carried_states_equal_one_pass(favor, cut):
    """A sequence cut at row `cut` into two windows: the forward of the second
    starts from the first's final state, the backward of the first takes the
    second's gradient with respect to its incoming state as g0.  Outputs,
    gradients (dW summed over the windows) and the gradient with respect to
    the very first state equal one pass over all rows."""
    rng = np.random.default_rng(53 + cut)
    q, k, v, dy, w, state0, g0 = _carry_case(rng, favor, length=13)
    y_all = oracle.recurrence_forward(q, k, v, w, state0=state0)
    full = oracle.recurrence_backward(q, k, v, w, dy, state0=state0, g0=g0, want_gstate=True)
    a = lambda t: t[:, :, :cut]
    b_ = lambda t: t[:, :, cut:]
    y1, s1 = oracle.recurrence_forward(a(q), a(k), a(v), w, state0=state0, return_state=True)
    y2 = oracle.recurrence_forward(b_(q), b_(k), b_(v), w, state0=s1)
    np.testing.assert_allclose(np.concatenate([y1, y2], axis=2), y_all, rtol=1e-12, atol=1e-12)
    g2 = oracle.recurrence_backward(b_(q), b_(k), b_(v), w, b_(dy), state0=s1, g0=g0, want_gstate=True)
    g1 = oracle.recurrence_backward(a(q), a(k), a(v), w, a(dy), state0=state0, g0=g2[4], want_gstate=True)
    for i in range(3):
        np.testing.assert_allclose(np.concatenate([g1[i], g2[i]], axis=2), full[i], rtol=1e-10, atol=1e-12)
    if favor:
        np.testing.assert_allclose(g1[3] + g2[3], full[3], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(g1[4], full[4], rtol=1e-10, atol=1e-12)
