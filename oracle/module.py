"""FP64 oracle of the triangle-attention module around the attention core
(test infrastructure only: only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import it).

"TurboPairFormer: Fast and Stable Protein Folding Model Training with an
Optimized Triangle Attention Kernel", Figure 6 and its worked example: a
normalization precedes the projections; each pair (i, j) of the pair tensor Z
is projected into a query, a key and a value; the score of query q and key k
in slice o adds a bias taken from pair (q, k); the attention output updates
pair (o, q).  Table 1 fixes the shapes: Z is [B, N, N, C_z]; Q, K, V, O are
[B, N_o, H, N, D] with N_o = N.

Readings where the pages are silent (also listed in the design notes):
  - the normalization is a LayerNorm over the C_z features of each pair with
    a learned scale and shift (gamma, beta), eps = 1e-5;
  - the projections are bias-free linear maps: W_in [C_z, 3 H D + H] gives
    q | k | v (head-major, D features each) | the H bias channels, and
    W_o [H D, C_z] maps the heads' outputs back to C_z;
  - no gating; the module returns W_o's output and leaves the residual
    update of Z to the caller.

Every step is written out plainly in float64; the attention core is the
core oracle (``oracle.oracle``), called on float64 arrays.
"""
from __future__ import annotations

import numpy as np

from . import oracle as core

EPS = 1e-5


def _f64(x) -> np.ndarray:
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().float().cpu().numpy()
    return np.asarray(x, dtype=np.float64)


def layernorm(z, gamma, beta):
    """x = (z - mean) / sqrt(var + eps) * gamma + beta over the last axis.
    Returns (x, xhat, rstd)."""
    mean = z.mean(axis=-1, keepdims=True)
    var = ((z - mean) ** 2).mean(axis=-1, keepdims=True)
    rstd = 1.0 / np.sqrt(var + EPS)
    xhat = (z - mean) * rstd
    return xhat * gamma + beta, xhat, rstd


def split_projection(p, H, D):
    """p [B, N, N, 3HD + H] -> q, k, v [B, N_o, H, N, D] and bias [B, H, N, N]."""
    B, N, _, _ = p.shape
    HD = H * D

    def heads(block):  # [B, i, j, H*D] -> [B, i, H, j, D]
        return block.reshape(B, N, N, H, D).transpose(0, 1, 3, 2, 4)

    q = heads(p[..., 0:HD])
    k = heads(p[..., HD:2 * HD])
    v = heads(p[..., 2 * HD:3 * HD])
    bias = p[..., 3 * HD:].transpose(0, 3, 1, 2)  # bias[b, h, q, k] = p[b, q, k, 3HD + h]
    return q, k, v, bias


def fwd(z, mask, gamma, beta, w_in, w_o, H, D):
    """out [B, N, N, C] and the intermediates, all float64."""
    z, gamma, beta, w_in, w_o = (_f64(a) for a in (z, gamma, beta, w_in, w_o))
    mask = _f64(mask)
    x, xhat, rstd = layernorm(z, gamma, beta)
    p = x @ w_in
    q, k, v, bias = split_projection(p, H, D)
    o, lse = core.fwd(q, k, v, bias, mask)
    B, N = z.shape[0], z.shape[1]
    o_flat = o.transpose(0, 1, 3, 2, 4).reshape(B, N, N, H * D)  # [B, i, j, (h, d)]
    out = o_flat @ w_o
    return {"out": out, "x": x, "xhat": xhat, "rstd": rstd, "p": p, "q": q, "k": k, "v": v, "bias": bias,
            "o": o, "lse": lse, "o_flat": o_flat}


def bwd(z, mask, gamma, beta, w_in, w_o, d_out, H, D):
    """Gradients (dz, dgamma, dbeta, dw_in, dw_o) of <out, d_out>, float64."""
    z, gamma, beta, w_in, w_o, d_out = (_f64(a) for a in (z, gamma, beta, w_in, w_o, d_out))
    f = fwd(z, mask, gamma, beta, w_in, w_o, H, D)
    B, N, _, C = z.shape
    HD = H * D
    # out = o_flat W_o
    dw_o = f["o_flat"].reshape(-1, HD).T @ d_out.reshape(-1, C)
    d_oflat = d_out @ w_o.T
    do = d_oflat.reshape(B, N, N, H, D).transpose(0, 1, 3, 2, 4)
    # attention core
    dq, dk, dv, dbias = core.bwd(f["q"], f["k"], f["v"], f["bias"], _f64(mask), do)

    def unheads(g):  # [B, i, H, j, D] -> [B, i, j, H*D]
        return g.transpose(0, 1, 3, 2, 4).reshape(B, N, N, HD)

    dp = np.concatenate([unheads(dq), unheads(dk), unheads(dv), dbias.transpose(0, 2, 3, 1)], axis=-1)
    # p = x W_in
    dw_in = f["x"].reshape(-1, C).T @ dp.reshape(-1, 3 * HD + H)
    dx = dp @ w_in.T
    # x = xhat * gamma + beta, xhat = (z - mean) * rstd
    dgamma = (dx * f["xhat"]).reshape(-1, C).sum(axis=0)
    dbeta = dx.reshape(-1, C).sum(axis=0)
    dxhat = dx * gamma
    dz = f["rstd"] * (dxhat - dxhat.mean(axis=-1, keepdims=True)
                      - f["xhat"] * (dxhat * f["xhat"]).mean(axis=-1, keepdims=True))
    return {"dz": dz, "dgamma": dgamma, "dbeta": dbeta, "dw_in": dw_in, "dw_o": dw_o}


def fwd_pairs(z, mask, gamma, beta, w_in, w_o, H, D, pairs):
    """out[b, i, j, :] for the listed (b, i, j) only, by the same steps as
    ``fwd`` restricted to what they read: query j of slice i attends over the
    pairs (i, k) of its slice, with the bias of score (j, k) taken from pair
    (j, k) (row j).  Returns [len(pairs), C] float64."""
    z, gamma, beta, w_in, w_o = (_f64(a) for a in (z, gamma, beta, w_in, w_o))
    mask = _f64(mask)
    HD = H * D
    out = []
    for (b, i, j) in pairs:
        p_i = layernorm(z[b, i], gamma, beta)[0] @ w_in          # pairs (i, k), k = 0..N-1
        p_j = layernorm(z[b, j], gamma, beta)[0] @ w_in          # pairs (j, k): the bias row
        o = np.empty(HD)
        for h in range(H):
            q = p_i[j, h * D:(h + 1) * D]
            k = p_i[:, HD + h * D:HD + (h + 1) * D]
            v = p_i[:, 2 * HD + h * D:2 * HD + (h + 1) * D]
            s = k @ q / np.sqrt(D) + p_j[:, 3 * HD + h]
            if mask is not None:
                s = s + mask[b, i]
            mx = s.max()
            if not np.isfinite(mx):
                o[h * D:(h + 1) * D] = 0.0
                continue
            e = np.exp(s - mx)
            o[h * D:(h + 1) * D] = (e / e.sum()) @ v
        out.append(o @ w_o)
    return np.stack(out)
