"""Multi-layer Performer language model -- TEST INFRASTRUCTURE ONLY
(plain PyTorch CPU ops in fp64; gradients by autograd of the plain forward).

"Sub-Linear Memory: How to Make Performers SLiM", section 2.2 (eq. 5-10) and
section 3 (Algorithm 1).  The display equations did not survive extraction;
this is the plainest reading of the surviving text (each reading is listed in
the design notes):
  X^(0)_l = E[p_l] + PE(l)        learned token embedding E (|Sigma| x d_model)
                                  plus the sinusoidal positional embedding of
                                  position l - 1 (sin on even, cos on odd
                                  coordinates, wavelengths 10000^(2i/d_model))
  for r = 1..s (GPT-2 ordering, layer norm before each block):
    Xb = LN1(X^(r-1));  Q^(j), K^(j), V^(j) = Xb W_Q^(j), Xb W_K^(j), Xb W_V^(j)
    H  = X^(r-1) + [Att^lin(Q^(1), K^(1), V^(1)), ..., Att^lin(Q^(k), K^(k), V^(k))]
    X^(r) = H + GeLU(LN2(H) W^(1) + b^(1)) W^(2) + b^(2)
  X^(out) = X^(s) W^(out) + b^(out)
  loss = sum over l = 1..L-1 of the cross-entropy of X^(out)_l against p_{l+1}
LN(x) = (x - mean) / sqrt(var + 1e-5) * gamma + beta (biased variance, per row);
GeLU(x) = x Phi(x) with the exact normal CDF.  The attention is causal linear
attention with feature map g (FAVOR+ with a fixed random projection per layer,
shared by the layer's heads, or elu+1), computed here by its explicit
quadratic form.

Parameter layout (one flat vector, the order of ``param_shapes``) is shared
with the library's model entry point.
"""
import math

import numpy as np
import torch

LN_EPS = 1e-5


def param_shapes(vocab, d_model, d_ff, layers):
    """Names and shapes of the trainable parameters, in layout order."""
    shapes = [("E", (vocab, d_model))]
    for r in range(layers):
        shapes += [("ln1_g_%d" % r, (d_model,)), ("ln1_b_%d" % r, (d_model,)),
                   ("W_qkv_%d" % r, (d_model, 3 * d_model)),
                   ("ln2_g_%d" % r, (d_model,)), ("ln2_b_%d" % r, (d_model,)),
                   ("W1_%d" % r, (d_model, d_ff)), ("b1_%d" % r, (d_ff,)),
                   ("W2_%d" % r, (d_ff, d_model)), ("b2_%d" % r, (d_model,))]
    shapes += [("W_out", (d_model, vocab)), ("b_out", (vocab,))]
    return shapes


def unflatten(theta, vocab, d_model, d_ff, layers):
    out, off = {}, 0
    for name, shp in param_shapes(vocab, d_model, d_ff, layers):
        n = int(np.prod(shp))
        out[name] = theta[off:off + n].reshape(shp)
        off += n
    assert off == theta.numel()
    return out


def positional(length, d_model, dtype=torch.float64):
    pos = torch.arange(length, dtype=dtype)[:, None]
    i = torch.arange(0, d_model, 2, dtype=dtype)[None, :]
    ang = pos / torch.pow(torch.tensor(10000.0, dtype=dtype), i / d_model)
    pe = torch.zeros((length, d_model), dtype=dtype)
    pe[:, 0::2] = torch.sin(ang)
    pe[:, 1::2] = torch.cos(ang)
    return pe


def layer_norm(x, g, b):
    mu = x.mean(dim=-1, keepdim=True)
    var = ((x - mu) ** 2).mean(dim=-1, keepdim=True)
    return (x - mu) / torch.sqrt(var + LN_EPS) * g + b


def gelu(x):
    return x * 0.5 * (1.0 + torch.erf(x / math.sqrt(2.0)))


def features(x, w):
    """g(x) along the last axis: FAVOR+ exp(x w - |x|^2/2)/sqrt(M), or elu+1."""
    if w is None:
        return torch.where(x > 0, x + 1.0, torch.exp(x))
    m = w.shape[1]
    return torch.exp(x @ w - 0.5 * (x * x).sum(-1, keepdim=True)) / math.sqrt(m)


def linear_attention(q, k, v, w):
    """Causal linear attention, explicit quadratic form; q, k, v [..., L, d]."""
    fq, fk = features(q, w), features(k, w)
    a = torch.tril(fq @ fk.transpose(-1, -2))
    return (a @ v) / a.sum(-1, keepdim=True)


def forward_loss(theta, tokens, cfg, feature_w):
    """Loss (sum of next-token cross-entropies) of tokens [B, L] (int64)."""
    vocab, d_model, heads, d_ff, layers = cfg["vocab"], cfg["d_model"], cfg["heads"], cfg["d_ff"], cfg["layers"]
    d = d_model // heads
    p = unflatten(theta, vocab, d_model, d_ff, layers)
    b, length = tokens.shape
    x = p["E"][tokens] + positional(length, d_model)
    for r in range(layers):
        xb = layer_norm(x, p["ln1_g_%d" % r], p["ln1_b_%d" % r])
        qkv = xb @ p["W_qkv_%d" % r]
        split = lambda t: t.reshape(b, length, heads, d).transpose(1, 2)
        q, k, v = (split(qkv[..., i * d_model:(i + 1) * d_model]) for i in range(3))
        w = None if feature_w is None else feature_w[r]
        y = linear_attention(q, k, v, w).transpose(1, 2).reshape(b, length, d_model)
        h = x + y
        z = layer_norm(h, p["ln2_g_%d" % r], p["ln2_b_%d" % r]) @ p["W1_%d" % r] + p["b1_%d" % r]
        x = h + gelu(z) @ p["W2_%d" % r] + p["b2_%d" % r]
    logits = x @ p["W_out"] + p["b_out"]
    logp = torch.log_softmax(logits[:, :-1], dim=-1)
    return -logp.gather(-1, tokens[:, 1:, None]).sum()


def loss_and_grad(theta, tokens, cfg, feature_w=None):
    """(loss, d loss / d theta) in fp64 by autograd of the plain forward."""
    th = torch.as_tensor(np.asarray(theta, dtype=np.float64)).clone().requires_grad_(True)
    tok = torch.as_tensor(np.asarray(tokens, dtype=np.int64))
    fw = None if feature_w is None else torch.as_tensor(np.asarray(feature_w, dtype=np.float64))
    loss = forward_loss(th, tok, cfg, fw)
    loss.backward()
    return float(loss.detach()), th.grad.numpy().copy()


def loss_only(theta, tokens, cfg, feature_w=None):
    with torch.no_grad():
        th = torch.as_tensor(np.asarray(theta, dtype=np.float64))
        tok = torch.as_tensor(np.asarray(tokens, dtype=np.int64))
        fw = None if feature_w is None else torch.as_tensor(np.asarray(feature_w, dtype=np.float64))
        return float(forward_loss(th, tok, cfg, fw))
