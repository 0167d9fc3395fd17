"""Seeded synthetic workloads for causal linear attention.

This module holds only random-input recipes and the workload table; it holds
none of the attention arithmetic and imports neither the CUDA binding nor the
oracle, so both sides of a parity test can be fed from it.

Workloads (shapes per (batch, head); all causal):

  name        B   H        L    d    M  chunk  dtype  Q, K               W
  tiny        1   1      256   16   32     32  fp32   N(0,1)*d^-1/4      iid N(0,1)
  l4k         8   8     4096   64  128     64  bf16   N(0,1)*d^-1/4      ORF
  l32k        2  16    32768   64  256    128  bf16   N(0,1)*d^-1/4      ORF
  l1m         1   8  1048576   64   64    256  bf16   N(0,1)*d^-1/4      ORF
  elu16k      4  12    16384  128  128     64  bf16   N(0,1)             none (elu+1)

V and dY are N(0,1).  Every tensor is drawn in fp32 from its own generator
seeded with (workload seed, tensor index) in the order Q, K, V, dY, W, then
cast to the workload dtype.  ORF ("orthogonal random features"): the M
feature vectors w_m (the columns of the d x M matrix W) come in blocks of d
mutually orthogonal directions (QR of a d x d Gaussian, signs fixed by the
diagonal of R), each rescaled to the norm of an independent N(0, I_d) draw,
i.e. a chi_d length; the last block is truncated when d does not divide M.
"""
import dataclasses
import math

import torch

_SEED0 = 1234


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    index: int
    B: int
    H: int
    L: int
    d: int
    M: int
    chunk: int
    dtype: str  # "fp32" | "bf16"
    feature: str  # "favor" | "elu"
    qk_scale: float
    w_kind: str  # "iid" | "orf" | "none"

    @property
    def seed(self):
        return _SEED0 + self.index

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "fp32" else torch.bfloat16

    def with_(self, **kw):
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "tiny": Workload("tiny", 1, 1, 1, 256, 16, 32, 32, "fp32", "favor", 16 ** -0.25, "iid"),
    "l4k": Workload("l4k", 2, 8, 8, 4096, 64, 128, 64, "bf16", "favor", 64 ** -0.25, "orf"),
    "l32k": Workload("l32k", 3, 2, 16, 32768, 64, 256, 128, "bf16", "favor", 64 ** -0.25, "orf"),
    "l1m": Workload("l1m", 4, 1, 8, 1 << 20, 64, 64, 256, "bf16", "favor", 64 ** -0.25, "orf"),
    "elu16k": Workload("elu16k", 5, 4, 12, 16384, 128, 128, 64, "bf16", "elu", 1.0, "none"),
}


def _gen(seed, slot, device):
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1000003 + slot)
    return g


def gaussian(shape, seed, slot, device="cpu", scale=1.0, dtype=torch.float32):
    """N(0, scale^2) draw in fp32 from generator (seed, slot), cast to dtype."""
    x = torch.randn(shape, generator=_gen(seed, slot, device), device=device, dtype=torch.float32)
    if scale != 1.0:
        x.mul_(scale)
    return x.to(dtype)


def orf_matrix(d, m, seed, slot=4):
    """Block-orthogonal Gaussian projection W (d x M, fp32, CPU), columns = features."""
    g = _gen(seed, slot, "cpu")
    cols = []
    for _ in range(math.ceil(m / d)):
        a = torch.randn((d, d), generator=g, dtype=torch.float64)
        qm, r = torch.linalg.qr(a)
        qm = qm * torch.sign(torch.diagonal(r)).unsqueeze(0)  # unique QR
        norms = torch.linalg.vector_norm(torch.randn((d, d), generator=g, dtype=torch.float64), dim=0)
        cols.append(qm * norms.unsqueeze(0))
    return torch.cat(cols, dim=1)[:, :m].contiguous().to(torch.float32)


def iid_matrix(d, m, seed, slot=4):
    return gaussian((d, m), seed, slot, "cpu")


def make_w(wl):
    if wl.w_kind == "none":
        return None
    if wl.w_kind == "orf":
        return orf_matrix(wl.d, wl.M, wl.seed)
    return iid_matrix(wl.d, wl.M, wl.seed)


def make_inputs(wl, device="cpu", heads=None, want_dy=True):
    """Q, K, V, dY ([B, H, L, d] in the workload dtype on ``device``) and W.

    ``heads`` (optional) overrides (B, H) for reduced-size variants; the
    per-tensor generators are the same, so a reduced variant is the workload
    recipe at another size, not a slice of the full tensors.
    """
    b, h = (wl.B, wl.H) if heads is None else heads
    shape = (b, h, wl.L, wl.d)
    dt = wl.torch_dtype
    q = gaussian(shape, wl.seed, 0, device, wl.qk_scale, dt)
    k = gaussian(shape, wl.seed, 1, device, wl.qk_scale, dt)
    v = gaussian(shape, wl.seed, 2, device, 1.0, dt)
    dy = gaussian(shape, wl.seed, 3, device, 1.0, dt) if want_dy else None
    w = make_w(wl)
    if w is not None:
        w = w.to(device)
    return q, k, v, dy, w


# ---- the multi-layer Performer language model: a random initialisation ----

def lm_param_layout(cfg):
    """Names and shapes of the model's parameters, in the order of its flat
    parameter vector: E, then per layer ln1_g, ln1_b, W_qkv, ln2_g, ln2_b,
    W1, b1, W2, b2, then W_out, b_out."""
    v, dm, ff = cfg["vocab"], cfg["d_model"], cfg["d_ff"]
    out = [("E", (v, dm))]
    for r in range(cfg["layers"]):
        out += [("ln1_g", (dm,)), ("ln1_b", (dm,)), ("W_qkv", (dm, 3 * dm)), ("ln2_g", (dm,)), ("ln2_b", (dm,)),
                ("W1", (dm, ff)), ("b1", (ff,)), ("W2", (ff, dm)), ("b2", (dm,))]
    return out + [("W_out", (dm, v)), ("b_out", (v,))]


def lm_init_params(cfg, seed):
    """A random initialisation as a flat float64 numpy vector: E ~ N(0, 0.02^2)
    (as GPT-2), projections ~ N(0, 1/fan_in) with the query and key thirds of
    W_qkv times d^(-1/4) (the Performer's normaliser, d = d_model / heads),
    biases zero, layer-norm gains one."""
    import numpy as np

    rng = np.random.default_rng(seed)
    d = cfg["d_model"] // cfg["heads"]
    parts = []
    for name, shp in lm_param_layout(cfg):
        if name.endswith("_g"):
            parts.append(np.ones(shp))
        elif name.startswith("b") or name.endswith("_b"):
            parts.append(np.zeros(shp))
        elif name == "E":
            parts.append(rng.standard_normal(shp) * 0.02)
        else:
            w = rng.standard_normal(shp) / math.sqrt(shp[0])
            if name == "W_qkv":
                w[:, :2 * cfg["d_model"]] *= d ** -0.25
            parts.append(w)
    return np.concatenate([x.ravel() for x in parts])
