"""Orthogonal random features drawn from a counter-based generator -- TEST
INFRASTRUCTURE ONLY (numpy, fp64).

"Sub-Linear Memory: How to Make Performers SLiM", section 2.1, names the
randomized feature map of Performers (FAVOR+) whose projection W is redrawn
during training.  The W recipe (the one the workloads use):
  * the M feature vectors w_m (the columns of the d x M matrix W) come in
    blocks of d mutually orthogonal directions: the Q factor of a d x d
    standard Gaussian matrix G = Q R, with the signs fixed so that diag(R) > 0
    (the unique such factorisation);
  * column c of a block is rescaled to the length of an independent N(0, I_d)
    draw (a chi_d length); the last block is truncated when d does not divide M.

The Gaussians come from Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel
random numbers: as easy as 1, 2, 3", SC 2011): a 4 x 32-bit counter, a
2 x 32-bit key, ten rounds of two 32 x 32 -> 64-bit multiplies with the round
constants 0xD2511F53 and 0xCD9E8D57, the key bumped by 0x9E3779B9 and
0xBB67AE85 between rounds.  Each 32-bit output x becomes a uniform
u = (x + 1/2) / 2^32 in (0, 1) and pairs (u_a, u_b) become two Gaussians by
the Box-Muller transform: sqrt(-2 ln u_a) (cos, sin)(2 pi u_b).

Draw layout (shared with the CUDA redraw, which implements the same
published generator on its own): matrix i of a redraw `step` with a 64-bit
`seed`, block b, uses key (seed mod 2^32, seed div 2^32) and counters
(j, b, i, step mod 2^32) for j = 0, 1, ...; call j yields Gaussians
4 j .. 4 j + 3 of the block's sequence: (x0, x1) -> g[4j], g[4j+1] and
(x2, x3) -> g[4j+2], g[4j+3].  The first d*d Gaussians fill G row-major
(G[r][c] = g[r*d + c]); the next d*d give the lengths: column c's length is
the norm of (g[d*d + r*d + c], r = 0 .. d-1).
"""
import numpy as np

_M0, _M1 = 0xD2511F53, 0xCD9E8D57
_W0, _W1 = 0x9E3779B9, 0xBB67AE85
_MASK = 0xFFFFFFFF


def philox4x32_10(ctr, key):
    """Philox4x32-10 on arrays: ctr [..., 4], key [..., 2] (uint32 values in
    uint64 arrays) -> [..., 4] uint32 outputs (as uint64)."""
    c = [np.asarray(ctr[..., i], dtype=np.uint64) & _MASK for i in range(4)]
    k0 = np.asarray(key[..., 0], dtype=np.uint64) & _MASK
    k1 = np.asarray(key[..., 1], dtype=np.uint64) & _MASK
    for r in range(10):
        if r > 0:
            k0 = (k0 + _W0) & _MASK
            k1 = (k1 + _W1) & _MASK
        p0 = c[0] * np.uint64(_M0)  # exact: both factors < 2^32
        p1 = c[2] * np.uint64(_M1)
        hi0, lo0 = p0 >> np.uint64(32), p0 & _MASK
        hi1, lo1 = p1 >> np.uint64(32), p1 & _MASK
        c = [hi1 ^ c[1] ^ k0, lo1, hi0 ^ c[3] ^ k1, lo0]
    return np.stack(c, axis=-1)


def block_gaussians(seed, step, i, b, n):
    """The first n Gaussians (fp64) of block b of matrix i (n a multiple of 4)."""
    j = np.arange(n // 4, dtype=np.uint64)
    ctr = np.stack([j, np.full_like(j, b), np.full_like(j, i), np.full_like(j, step & _MASK)], axis=-1)
    key = np.array([seed & _MASK, (seed >> 32) & _MASK], dtype=np.uint64)
    x = philox4x32_10(ctr, np.broadcast_to(key, ctr.shape[:-1] + (2,)))
    u = (x.astype(np.float64) + 0.5) / 4294967296.0
    out = np.empty((n // 4, 4))
    for a, bb in ((0, 1), (2, 3)):
        rad = np.sqrt(-2.0 * np.log(u[:, a]))
        ang = 2.0 * np.pi * u[:, bb]
        out[:, a] = rad * np.cos(ang)
        out[:, bb] = rad * np.sin(ang)
    return out.reshape(-1)


def orf_matrix(d, m, seed, step=0, i=0):
    """Matrix i of a redraw: block-orthogonal W (d x m, fp64), columns = features."""
    cols = []
    for b in range((m + d - 1) // d):
        g = block_gaussians(seed, step, i, b, 2 * d * d)
        gm = g[:d * d].reshape(d, d)
        q, r = np.linalg.qr(gm)
        q = q * np.sign(np.diag(r))[None, :]  # diag(R) > 0
        lengths = np.linalg.norm(g[d * d:].reshape(d, d), axis=0)
        cols.append(q * lengths[None, :])
    return np.concatenate(cols, axis=1)[:, :m]


def orf_matrices(n, d, m, seed, step=0):
    """n independent matrices of one redraw: [n, d, m]."""
    return np.stack([orf_matrix(d, m, seed, step, i) for i in range(n)])
