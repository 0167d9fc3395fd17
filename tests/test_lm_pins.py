"""Pins for the multi-layer Performer oracle (oracle/lm.py, CPU only).

"Sub-Linear Memory: How to Make Performers SLiM", section 2.2 (the GPT-2
style Performer, eq. 5-10) and section 3.2 (Algorithm 1's forward: slices of
C rows, every layer's prefix-sum state carried across slice boundaries).
Each pin fixes the oracle from outside: a closed form of the loss, published
values of GeLU and of the sinusoidal embedding, the layer-norm invariants,
central differences of the loss, and the slice-by-slice forward built from
the independent C recurrence with carried states.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import lm, orf
from sub_linear_memory_gb300 import inputs

CFG = {"vocab": 11, "d_model": 8, "heads": 2, "d_ff": 12, "layers": 2, "M": 8}


def _model(seed, favor=True, cfg=CFG):
    theta = inputs.lm_init_params(cfg, seed)
    d = cfg["d_model"] // cfg["heads"]
    fw = orf.orf_matrices(cfg["layers"], d, cfg["M"], seed=seed) if favor else None
    return theta, fw


def test_gelu_and_positional_values():
    # GeLU(x) = x Phi(x): Phi(1) = 0.8413447460685429 (normal table)
    g = lm.gelu(torch.tensor([1.0, -1.0, 0.0], dtype=torch.float64)).numpy()
    np.testing.assert_allclose(g, [0.8413447460685429, -0.15865525393145707, 0.0], rtol=1e-14, atol=1e-16)
    pe = lm.positional(3, 6).numpy()
    np.testing.assert_allclose(pe[0], [0, 1, 0, 1, 0, 1], atol=1e-15)
    np.testing.assert_allclose(pe[1, 0], math.sin(1.0), rtol=1e-14)           # wavelength 10000^0
    np.testing.assert_allclose(pe[2, 3], math.cos(2.0 / 10000 ** (2 / 6)), rtol=1e-14)


def test_layer_norm_rows():
    x = torch.randn(5, 16, dtype=torch.float64) * 3 + 2
    y = lm.layer_norm(x, torch.ones(16, dtype=torch.float64), torch.zeros(16, dtype=torch.float64))
    np.testing.assert_allclose(y.mean(-1).numpy(), 0, atol=1e-14)
    var = x.var(-1, unbiased=False)
    np.testing.assert_allclose(((y ** 2).mean(-1)).numpy(), (var / (var + lm.LN_EPS)).numpy(), rtol=1e-12)


def test_uniform_logits_closed_form():
    """W_out = 0, b_out = 0: every prediction is uniform over the alphabet, so
    the loss is B (L - 1) log |Sigma| whatever the rest of the model does."""
    theta, fw = _model(1)
    p = lm.unflatten(torch.as_tensor(theta), CFG["vocab"], CFG["d_model"], CFG["d_ff"], CFG["layers"])
    p["W_out"][...] = 0
    p["b_out"][...] = 0
    tok = np.random.default_rng(2).integers(0, CFG["vocab"], size=(3, 9))
    loss = lm.loss_only(theta, tok, CFG, fw)
    assert abs(loss - 3 * 8 * math.log(CFG["vocab"])) < 1e-10


@pytest.mark.parametrize("favor", [True, False])
def test_gradient_matches_central_differences(favor):
    theta, fw = _model(3, favor)
    tok = np.random.default_rng(4).integers(0, CFG["vocab"], size=(2, 7))
    _, grad = lm.loss_and_grad(theta, tok, CFG, fw)
    rng = np.random.default_rng(5)
    idx = rng.choice(theta.size, size=40, replace=False)
    h = 1e-6
    for i in idx:
        tp, tm = theta.copy(), theta.copy()
        tp[i] += h
        tm[i] -= h
        fd = (lm.loss_only(tp, tok, CFG, fw) - lm.loss_only(tm, tok, CFG, fw)) / (2 * h)
        assert abs(fd - grad[i]) <= 1e-6 * max(1.0, abs(fd)), (i, fd, grad[i])


def _chunked_loss(theta, tok, cfg, fw, chunk):
    """Algorithm 1's forward: slices of `chunk` rows, every layer's attention
    run by the C recurrence from the layer's carried boundary state."""
    vocab, dm, heads, dff, layers = cfg["vocab"], cfg["d_model"], cfg["heads"], cfg["d_ff"], cfg["layers"]
    d = dm // heads
    p = {k: v.numpy() for k, v in lm.unflatten(torch.as_tensor(theta), vocab, dm, dff, layers).items()}
    b, length = tok.shape
    pe = lm.positional(length, dm).numpy()
    m = d if fw is None else fw.shape[-1]
    states = [np.zeros((b, heads, d + 1, m)) for _ in range(layers)]
    t = lambda a: torch.as_tensor(a)
    loss = 0.0
    for a0 in range(0, length, chunk):
        rows = slice(a0, min(a0 + chunk, length))
        x = p["E"][tok[:, rows]] + pe[rows]
        for r in range(layers):
            xb = lm.layer_norm(t(x), t(p["ln1_g_%d" % r]), t(p["ln1_b_%d" % r])).numpy()
            qkv = xb @ p["W_qkv_%d" % r]
            split = lambda z: np.ascontiguousarray(z.reshape(b, -1, heads, d).transpose(0, 2, 1, 3))
            q, k, v = (split(qkv[..., i * dm:(i + 1) * dm]) for i in range(3))
            y, states[r] = oracle.recurrence_forward(q, k, v, None if fw is None else fw[r], state0=states[r],
                                                     return_state=True)
            h = x + y.transpose(0, 2, 1, 3).reshape(b, -1, dm)
            z = lm.layer_norm(t(h), t(p["ln2_g_%d" % r]), t(p["ln2_b_%d" % r])).numpy() @ p["W1_%d" % r] + p["b1_%d" % r]
            x = h + lm.gelu(t(z)).numpy() @ p["W2_%d" % r] + p["b2_%d" % r]
        logits = x @ p["W_out"] + p["b_out"]
        nxt = min(a0 + chunk, length - 1)
        for row in range(a0, nxt):
            lg = logits[:, row - a0]
            lse = np.log(np.exp(lg - lg.max(-1, keepdims=True)).sum(-1)) + lg.max(-1)
            loss += float(np.sum(lse - lg[np.arange(b), tok[:, row + 1]]))
    return loss


@pytest.mark.parametrize("favor", [True, False])
@pytest.mark.parametrize("chunk", [1, 4, 7, 30])
def test_slice_by_slice_forward_equals_full(favor, chunk):
    theta, fw = _model(6, favor)
    tok = np.random.default_rng(7).integers(0, CFG["vocab"], size=(2, 23))
    full = lm.loss_only(theta, tok, CFG, fw)
    assert abs(_chunked_loss(theta, tok, CFG, fw, chunk) - full) <= 1e-10 * abs(full)
