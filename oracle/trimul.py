"""FP64 oracle of the triangle multiplicative update, outgoing and incoming
(test infrastructure only: only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import it).

"TurboPairFormer: Fast and Stable Protein Folding Model Training with an
Optimized Triangle Attention Kernel", Figure 12 (the outgoing update: an input
stage that normalizes the pair features and forms five projections -- two
branch values, two branch gates and the output-gate logits -- with the branch
values gated and masked; a contraction of the two branch operands done
independently for every channel; an output stage of normalization, output
projection and multiplication by the sigmoid of the saved output-gate logits)
and Table 10 (shapes: N in {384, 640, 768}, 64 or 128 channels, one example,
forward plus backward, both directions).

The pages print no formulas.  Readings (also listed in the design notes):
  - both normalizations are LayerNorms over the feature axis with learned
    scale and shift, eps = 1e-5;
  - every projection is a bias-free linear map; one matrix
    W_p [C_z, 4 C_h + C_z] gives, in this column order, the branch values and
    gates a_v | a_g | b_v | b_g (C_h each) and the output-gate logits g (C_z);
  - a = m * sigmoid(a_g) * a_v and b = m * sigmoid(b_g) * b_v, with m the
    optional multiplicative pair mask [B, N, N] (1 keeps a pair);
  - outgoing: X[b, i, j, c] = sum_k a[b, i, k, c] b[b, j, k, c]
    incoming: X[b, i, j, c] = sum_k a[b, k, i, c] b[b, k, j, c]
    (edges leaving i and j, or entering them);
  - out = sigmoid(g) * (LayerNorm(X) W_o) with W_o [C_h, C_z]; the residual
    update of Z is left to the caller.

Every step is written out in float64, the contraction as an einsum of its
defining sum.
"""
from __future__ import annotations

import numpy as np

EPS = 1e-5
DIRECTIONS = ("outgoing", "incoming")


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().float().cpu().numpy()
    return np.asarray(x, dtype=np.float64)


def sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def layernorm(z, gamma, beta):
    """x = (z - mean) / sqrt(var + eps) * gamma + beta over the last axis.
    Returns (x, xhat, rstd)."""
    mean = z.mean(axis=-1, keepdims=True)
    var = ((z - mean) ** 2).mean(axis=-1, keepdims=True)
    rstd = 1.0 / np.sqrt(var + EPS)
    xhat = (z - mean) * rstd
    return xhat * gamma + beta, xhat, rstd


def layernorm_bwd(dx, xhat, rstd, gamma):
    """Gradients (dz, dgamma, dbeta) of x = xhat * gamma + beta."""
    C = dx.shape[-1]
    dgamma = (dx * xhat).reshape(-1, C).sum(axis=0)
    dbeta = dx.reshape(-1, C).sum(axis=0)
    dxh = dx * gamma
    dz = rstd * (dxh - dxh.mean(axis=-1, keepdims=True) - xhat * (dxh * xhat).mean(axis=-1, keepdims=True))
    return dz, dgamma, dbeta


def split_projection(p, Ch):
    """p [..., 4 Ch + Cz] -> a_v, a_g, b_v, b_g [..., Ch] and g [..., Cz]."""
    return p[..., 0:Ch], p[..., Ch:2 * Ch], p[..., 2 * Ch:3 * Ch], p[..., 3 * Ch:4 * Ch], p[..., 4 * Ch:]


def contract(a, b, direction):
    """The per-channel contraction over the third token k."""
    if direction == "outgoing":
        return np.einsum("bikc,bjkc->bijc", a, b, optimize=True)
    if direction == "incoming":
        return np.einsum("bkic,bkjc->bijc", a, b, optimize=True)
    raise ValueError(direction)


def fwd(z, mask, ln_in_w, ln_in_b, w_p, ln_out_w, ln_out_b, w_o, direction):
    """out [B, N, N, Cz] and the intermediates, all float64."""
    z, ln_in_w, ln_in_b, w_p, ln_out_w, ln_out_b, w_o = (
        _f64(t) for t in (z, ln_in_w, ln_in_b, w_p, ln_out_w, ln_out_b, w_o))
    Ch = w_o.shape[0]
    m = np.ones(z.shape[:3] + (1,)) if mask is None else _f64(mask)[..., None]
    x, xhat, rstd = layernorm(z, ln_in_w, ln_in_b)
    p = x @ w_p
    av, ag, bv, bg, g = split_projection(p, Ch)
    a = m * sigmoid(ag) * av
    b = m * sigmoid(bg) * bv
    X = contract(a, b, direction)
    y, yhat, rstd_out = layernorm(X, ln_out_w, ln_out_b)
    u = y @ w_o
    out = sigmoid(g) * u
    return {"out": out, "x": x, "xhat": xhat, "rstd": rstd, "p": p, "m": m, "a": a, "b": b, "X": X, "y": y,
            "yhat": yhat, "rstd_out": rstd_out, "u": u}


def bwd(z, mask, ln_in_w, ln_in_b, w_p, ln_out_w, ln_out_b, w_o, d_out, direction):
    """Gradients of <out, d_out> with respect to z and every parameter."""
    f = fwd(z, mask, ln_in_w, ln_in_b, w_p, ln_out_w, ln_out_b, w_o, direction)
    ln_in_w, w_p, ln_out_w, w_o, d_out = (_f64(t) for t in (ln_in_w, w_p, ln_out_w, w_o, d_out))
    Ch, Cz = w_o.shape
    av, ag, bv, bg, g = split_projection(f["p"], Ch)
    m = f["m"]
    # out = sigmoid(g) * u,  u = y W_o
    sg = sigmoid(g)
    du = d_out * sg
    dg = d_out * f["u"] * sg * (1.0 - sg)
    dw_o = f["y"].reshape(-1, Ch).T @ du.reshape(-1, Cz)
    dy = du @ w_o.T
    dX, dln_out_w, dln_out_b = layernorm_bwd(dy, f["yhat"], f["rstd_out"], ln_out_w)
    # the contraction
    a, b = f["a"], f["b"]
    if direction == "outgoing":
        da = np.einsum("bijc,bjkc->bikc", dX, b, optimize=True)
        db = np.einsum("bijc,bikc->bjkc", dX, a, optimize=True)
    else:
        da = np.einsum("bijc,bkjc->bkic", dX, b, optimize=True)
        db = np.einsum("bijc,bkic->bkjc", dX, a, optimize=True)
    # a = m sigmoid(a_g) a_v, b likewise
    sa, sb = sigmoid(ag), sigmoid(bg)
    dav = da * m * sa
    dag = da * m * av * sa * (1.0 - sa)
    dbv = db * m * sb
    dbg = db * m * bv * sb * (1.0 - sb)
    dp = np.concatenate([dav, dag, dbv, dbg, dg], axis=-1)
    # p = x W_p
    dw_p = f["x"].reshape(-1, Cz).T @ dp.reshape(-1, dp.shape[-1])
    dx = dp @ w_p.T
    dz, dln_in_w, dln_in_b = layernorm_bwd(dx, f["xhat"], f["rstd"], ln_in_w)
    return {"dz": dz, "dln_in_w": dln_in_w, "dln_in_b": dln_in_b, "dw_p": dw_p, "dln_out_w": dln_out_w,
            "dln_out_b": dln_out_b, "dw_o": dw_o, "out": f["out"]}


def fwd_pairs(z, mask, ln_in_w, ln_in_b, w_p, ln_out_w, ln_out_b, w_o, direction, pairs):
    """out[b, i, j, :] for the listed (b, i, j) only, by the same steps as
    ``fwd`` restricted to the pairs they read: outgoing X[b, i, j] needs rows
    i and j of the branch operands (pairs (i, k) and (j, k)), incoming needs
    columns i and j (pairs (k, i) and (k, j)); the gate needs pair (i, j).
    Returns [len(pairs), C_z] float64."""
    z, ln_in_w, ln_in_b, w_p, ln_out_w, ln_out_b, w_o = (
        _f64(t) for t in (z, ln_in_w, ln_in_b, w_p, ln_out_w, ln_out_b, w_o))
    mask = _f64(mask)
    Ch = w_o.shape[0]

    def branch_line(b, t):
        """a and b of the N pairs on line t: row t (outgoing) or column t (incoming)."""
        zl = z[b, t] if direction == "outgoing" else z[b, :, t]
        ml = np.ones(zl.shape[0]) if mask is None else (mask[b, t] if direction == "outgoing" else mask[b, :, t])
        x, _, _ = layernorm(zl, ln_in_w, ln_in_b)
        av, ag, bv, bg, _ = split_projection(x @ w_p, Ch)
        return ml[:, None] * sigmoid(ag) * av, ml[:, None] * sigmoid(bg) * bv

    out = []
    for (b, i, j) in pairs:
        a_i, _ = branch_line(b, i)
        _, b_j = branch_line(b, j)
        X = (a_i * b_j).sum(axis=0)                      # sum over the third token k
        y, _, _ = layernorm(X, ln_out_w, ln_out_b)
        x_ij, _, _ = layernorm(z[b, i, j], ln_in_w, ln_in_b)
        g = split_projection(x_ij @ w_p, Ch)[4]
        out.append(sigmoid(g) * (y @ w_o))
    return np.stack(out)
