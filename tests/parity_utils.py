"""Shared helpers for the GPU parity tests: run the CUDA path through the C
ABI binding and compare with the FP64 oracle on the same seeded inputs."""
from __future__ import annotations

import numpy as np
import torch

from oracle import oracle as O
from protein_folding_triangle_gb300 import synthetic as S
from protein_folding_triangle_gb300 import triattn as T

# Tolerances on relative RMSE (RMSE / RMS of the FP64 value).
TOL_O = 4e-3
TOL_GRAD = 1e-2

# Bound on |sum_c dz[m, c]| relative to sum_c |dz[m, c]| for the BF16 dz of
# a LayerNorm backward (exactly zero in exact arithmetic):
#  - rounding each FP32 element once to BF16 (round to nearest) moves it by
#    at most 2^-8 of its magnitude, so the rounded sum moves by at most
#    2^-8 sum |dz32| <= 2^-8 sum |dz| / (1 - 2^-8);
#  - the FP32 sum itself, rstd (sum g - C mean(g) - mean(g xhat) sum xhat),
#    is not zero after rounding: the FP32 mean of g is off by at most about
#    (C/32 + 6) 2^-24 sum |g| (per-lane runs, then a 32-lane butterfly),
#    sum xhat by C 4 2^-24 max|xhat| (FP32 mean and rstd of the row), and
#    each element carries three FP32 roundings.  With sum |dz32| close to
#    rstd sum |g| (g is not nearly in the span of 1 and xhat) that is far
#    below 2^-16 sum |dz32|, which the bound allows on top.
LN_ROW_SUM_BOUND = (2.0 ** -8 + 2.0 ** -16) / (1.0 - 2.0 ** -8)


def rel_rmse(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.sqrt(np.mean(ref ** 2))
    return float(np.sqrt(np.mean((got - ref) ** 2)) / max(den, 1e-300))


def to_dev(x: dict, device="cuda") -> dict:
    return {k: (None if v is None else v.to(device).contiguous()) for k, v in x.items()}


def gpu_fwd_bwd(xd: dict, compensate: bool = True, workspace=None):
    o, lse, resid = T.tri_attn_fwd(xd["q"], xd["k"], xd["v"], xd["bias"], xd["mask"], save_residual=True)
    dq, dk, dv, db = T.tri_attn_bwd(xd["q"], xd["k"], xd["v"], xd["bias"], xd["mask"], o,
                                    resid if compensate else None, lse, xd["do"], workspace=workspace)
    torch.cuda.synchronize()
    status = T.device_status()
    assert status == T.OK, f"device status {T.STATUS[status]}"
    return {"o": o, "lse": lse, "resid": resid, "dq": dq, "dk": dk, "dv": dv, "dbias": db}


def cpu64(t):
    return t.detach().float().cpu().double().numpy()


def oracle_full(x: dict):
    o, lse = O.fwd(x["q"], x["k"], x["v"], x["bias"], x["mask"])
    dq, dk, dv, db = O.bwd(x["q"], x["k"], x["v"], x["bias"], x["mask"], x["do"])
    return {"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv, "dbias": db}


def compare_full(out: dict, ref: dict) -> dict:
    errs = {}
    for name in ("o", "dq", "dk", "dv", "dbias"):
        errs[name] = rel_rmse(cpu64(out[name]), ref[name])
    lg = cpu64(out["lse"])
    fin = np.isfinite(ref["lse"])
    errs["lse_maxabs"] = float(np.abs(lg[fin] - ref["lse"][fin]).max()) if fin.any() else 0.0
    errs["lse_inf_match"] = bool(np.all(np.isneginf(lg[~fin]))) if (~fin).any() else True
    return errs


def head_inputs(x: dict, b: int, h: int):
    """(q, k, v, bias, mask, dO) of head (b, h) alone, every outer slice (so
    that the oracle converts only this head's data to FP64)."""
    sl = (slice(b, b + 1), slice(None), slice(h, h + 1))
    mask = None if x["mask"] is None else x["mask"][b:b + 1].contiguous()
    return (x["q"][sl].contiguous(), x["k"][sl].contiguous(), x["v"][sl].contiguous(),
            x["bias"][b:b + 1, h:h + 1].contiguous(), mask, x["do"][sl].contiguous())


def sample_indices(w: S.Workload, n_slices: int, n_rows: int, seed: int = 1234, all_heads: bool = False):
    rng = np.random.default_rng(seed)
    slices = []
    for _ in range(n_slices):
        slices.append((int(rng.integers(w.B)), int(rng.integers(w.No)), int(rng.integers(w.H))))
    heads = [(int(rng.integers(w.B)), int(rng.integers(w.H)))]
    if all_heads:
        heads = [(b, h) for b in range(w.B) for h in range(w.H)]
    rows = sorted(set(int(r) for r in rng.integers(0, w.N, size=n_rows)))
    return slices, heads, rows


def compare_sampled(x: dict, out: dict, w: S.Workload, n_slices=3, n_rows=8, seed=1234, all_heads=False) -> dict:
    """Compare the GPU result with the oracle on sampled slices (all of O,
    lse, dQ, dK, dV there) and on sampled query rows of dbias (every slice
    contributes to those rows) of one sampled head, or of every head."""
    slices, heads, rows = sample_indices(w, n_slices, n_rows, seed, all_heads)
    acc = {k: ([], []) for k in ("o", "dq", "dk", "dv", "dbias")}
    lse_err = 0.0
    for (b, o_, h) in slices:
        r = O.slice_(*head_inputs(x, b, h), 0, o_, 0)
        for name in ("o", "dq", "dk", "dv"):
            acc[name][0].append(cpu64(out[name][b, o_, h]).ravel())
            acc[name][1].append(r[name].ravel())
        lg = cpu64(out["lse"][b, o_, h])
        fin = np.isfinite(r["lse"])
        if fin.any():
            lse_err = max(lse_err, float(np.abs(lg[fin] - r["lse"][fin]).max()))
    for (b, h) in heads:
        r = O.rows(*head_inputs(x, b, h), 0, 0, rows)
        acc["dbias"][0].append(cpu64(out["dbias"][b, h][rows]).ravel())
        acc["dbias"][1].append(r["dbias"].ravel())
    errs = {name: rel_rmse(np.concatenate(g), np.concatenate(rf)) for name, (g, rf) in acc.items()}
    errs["lse_maxabs"] = lse_err
    return errs
