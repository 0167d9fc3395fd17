"""Quadratic-form oracle -- TEST INFRASTRUCTURE ONLY.

Plain numpy fp64, O(L^2) per head; only for small L.  Written independently
of the C recurrence in ``slim_oracle.c`` (own feature map, own backward) so
that the two can pin each other.

Source: "Sub-Linear Memory: How to Make Performers SLiM", section 2.1.
  * eq. (1), exponential (softmax) self-attention, causal:
        Y_l = sum_{j<=l} exp(Q_l.K_j) V_j / sum_{j<=l} exp(Q_l.K_j)
    (Q and K arrive already scaled, so no extra 1/sqrt(d)).
  * eq. (2), linear self-attention, first (quadratic) form:
        Y_l = sum_{j<=l} (g(Q_l).g(K_j)) V_j / sum_{j<=l} g(Q_l).g(K_j)
    The diagonal j = l is included: Y_l depends on inputs 1..l.
Feature maps (the page names a randomized positive map and an elementwise
one without printing formulas):
    FAVOR+  g(x)_m = exp(w_m.x - |x|^2/2) / sqrt(M),  w_m = column m of W (d x M)
    elu+1   g(x)_i = x_i + 1 if x_i > 0 else exp(x_i)   (M == d)
"""
import numpy as np


def feature_map(x, w):
    """g(x) along the last axis. ``w`` None selects elu+1."""
    x = np.asarray(x, dtype=np.float64)
    if w is None:
        return np.where(x > 0, x + 1.0, np.exp(np.minimum(x, 0.0)))
    w = np.asarray(w, dtype=np.float64)
    m = w.shape[1]
    return np.exp(x @ w - 0.5 * np.sum(x * x, axis=-1, keepdims=True)) / np.sqrt(m)


def feature_map_backward(x, w, phi, dphi):
    """Chain rule through g: returns (dx, dW or None).

    FAVOR+: d g_m / d x = g_m (w_m - x), d g_m / d w_m = g_m x.
    elu+1:  d g_i / d x_i = 1 if x_i > 0 else exp(x_i).
    """
    x = np.asarray(x, dtype=np.float64)
    if w is None:
        return dphi * np.where(x > 0, 1.0, np.exp(np.minimum(x, 0.0))), None
    u = phi * dphi
    dx = u @ np.asarray(w, dtype=np.float64).T - x * np.sum(u, axis=-1, keepdims=True)
    dw = x.reshape(-1, x.shape[-1]).T @ u.reshape(-1, u.shape[-1])
    return dx, dw


def _causal_weights(q, k, w):
    phiq, phik = feature_map(q, w), feature_map(k, w)
    length = q.shape[-2]
    a = np.einsum("...lm,...jm->...lj", phiq, phik) * np.tril(np.ones((length, length)))
    return phiq, phik, a


def forward(q, k, v, w):
    """Y by the explicit quadratic form; arrays [..., L, d]."""
    _, _, a = _causal_weights(q, k, w)
    num = a @ np.asarray(v, dtype=np.float64)
    den = np.sum(a, axis=-1, keepdims=True)
    return num / den


def backward(q, k, v, w, dy):
    """Gradients of sum(dy * Y) for the quadratic form, differentiated by hand.

    Y = N / D with N = A V, D = A 1 and A = tril(g(Q) g(K)^T):
        dN = dy / D,  dD = -(dy . Y) / D,
        dA = tril(dN V^T + dD 1^T),
        dg(Q) = dA g(K),  dg(K) = dA^T g(Q),  dV = A^T dN.
    Returns (dq, dk, dv, dw) with dw None for elu+1.
    """
    v = np.asarray(v, dtype=np.float64)
    dy = np.asarray(dy, dtype=np.float64)
    phiq, phik, a = _causal_weights(q, k, w)
    length = v.shape[-2]
    mask = np.tril(np.ones((length, length)))
    num = a @ v
    den = np.sum(a, axis=-1, keepdims=True)
    y = num / den
    dnum = dy / den
    dden = -np.sum(dy * y, axis=-1, keepdims=True) / den
    da = (dnum @ np.swapaxes(v, -1, -2) + dden) * mask
    dphiq = da @ phik
    dphik = np.swapaxes(da, -1, -2) @ phiq
    dv = np.swapaxes(a, -1, -2) @ dnum
    dq, dwq = feature_map_backward(q, w, phiq, dphiq)
    dk, dwk = feature_map_backward(k, w, phik, dphik)
    dw = None if w is None else dwq + dwk
    return dq, dk, dv, dw


def softmax_forward(q, k, v):
    """Causal exponential self-attention, eq. (1); max-shifted per row, which
    leaves every row's weights unchanged."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    length = q.shape[-2]
    s = q @ np.swapaxes(k, -1, -2)
    s = np.where(np.tril(np.ones((length, length))) > 0, s, -np.inf)
    s = s - np.max(s, axis=-1, keepdims=True)
    p = np.exp(s)
    return (p @ np.asarray(v, dtype=np.float64)) / np.sum(p, axis=-1, keepdims=True)
