"""Pins of the FP64 oracle to things other than itself (CPU only).

The oracle (oracle/triattn_oracle.c) states triangular attention from its
definition in "TurboPairFormer" (Abstract, Figure 1(a), Table 1, Figure 6).
These tests tie it to:
  * an independent library route: torch's scaled_dot_product_attention in
    FP64 with the bias + mask as an additive attention mask, and torch
    autograd through it for all four gradients;
  * central finite differences of sum(dO * O) on tiny inputs;
  * closed forms (uniform softmax) and invariants that the mathematics fixes
    (rows of P sum to 1, per-row bias shift, zero row-sum of dS, dbias is the
    sum over slices of dS, sum_k dV = sum_q dO, masked keys get zero dK/dV,
    K-shift invariance, permutation equivariance);
  * the index structure of the Figure 6 worked example.
A last group plants mistakes in a copy of the oracle source and checks that
the pins above catch each one.
"""
import json
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import oracle as O

HERE = os.path.dirname(os.path.abspath(__file__))


def rand_problem(B, No, H, N, D, seed, mask="none", bias_std=1.0, Nq=None):
    rng = np.random.default_rng(seed)
    Nq = N if Nq is None else Nq
    q = rng.standard_normal((B, No, H, Nq, D))
    k = rng.standard_normal((B, No, H, N, D))
    v = rng.standard_normal((B, No, H, N, D))
    do = rng.standard_normal((B, No, H, Nq, D))
    bias = rng.standard_normal((B, H, Nq, N)) * bias_std
    m = None
    if mask == "random":
        drop = rng.random((B, No, N)) < 0.3
        drop[..., 0] = False  # keep one key per slice
        m = np.where(drop, -np.inf, 0.0)
    elif mask == "tail":
        m = np.zeros((B, No, N))
        m[..., N - max(1, N // 4):] = -np.inf
    return q, k, v, do, bias, m


def torch_reference(q, k, v, bias, mask, do):
    """FP64 torch SDPA (library routine) + autograd: O and the four grads."""
    tq, tk, tv, tb = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v, bias))
    am = tb[:, None]                                   # [B,1,H,Nq,Nk]
    if mask is not None:
        am = am + torch.tensor(mask)[:, :, None, None, :]  # [B,No,1,1,Nk]
    out = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=am)
    out.backward(torch.tensor(do))
    return (out.detach().numpy(), tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy(), tb.grad.numpy())


def rel_err(a, b):
    a, b = np.asarray(a), np.asarray(b)
    return float(np.sqrt(np.mean((a - b) ** 2)) / max(np.sqrt(np.mean(b ** 2)), 1e-300))


SHAPES = [
    (1, 3, 2, 5, 4, "none"),
    (2, 4, 1, 7, 2, "random"),
    (1, 6, 3, 6, 8, "tail"),
    (1, 5, 2, 9, 16, "random"),
    (1, 1, 2, 12, 32, "none"),
]


@pytest.mark.parametrize("shape", SHAPES)
def test_matches_torch_sdpa_and_autograd(shape):
    B, No, H, N, D, mk = shape
    q, k, v, do, bias, m = rand_problem(B, No, H, N, D, seed=sum(shape[:5]), mask=mk)
    o, lse = O.fwd(q, k, v, bias, m)
    dq, dk, dv, db = O.bwd(q, k, v, bias, m, do)
    ro, rdq, rdk, rdv, rdb = torch_reference(q, k, v, bias, m, do)
    for name, a, b in [("o", o, ro), ("dq", dq, rdq), ("dk", dk, rdk), ("dv", dv, rdv), ("dbias", db, rdb)]:
        assert rel_err(a, b) < 1e-12, name
    # lse through the library logsumexp of the library-built scores
    s = torch.einsum("bohqd,bohkd->bohqk", torch.tensor(q), torch.tensor(k)) / np.sqrt(D)
    s = s + torch.tensor(bias)[:, None]
    if m is not None:
        s = s + torch.tensor(m)[:, :, None, None, :]
    assert np.allclose(lse, torch.logsumexp(s, dim=-1).numpy(), rtol=0, atol=1e-12)


def test_plain_sdpa_special_case():
    """N_o = 1, zero bias, no mask: the method is plain scaled dot-product attention."""
    q, k, v, do, _, _ = rand_problem(1, 1, 3, 10, 8, seed=5)
    bias = np.zeros((1, 3, 10, 10))
    o, _ = O.fwd(q, k, v, bias, None)
    ref = F.scaled_dot_product_attention(*(torch.tensor(x) for x in (q, k, v))).numpy()
    assert np.abs(o - ref).max() < 1e-13


@pytest.mark.parametrize("shape", [(1, 3, 1, 3, 2, "none"), (1, 2, 2, 4, 3, "random"), (1, 3, 1, 5, 4, "tail")])
def test_finite_differences(shape):
    B, No, H, N, D, mk = shape
    q, k, v, do, bias, m = rand_problem(B, No, H, N, D, seed=11 + N, mask=mk)
    grads = O.bwd(q, k, v, bias, m, do)
    eps = 1e-6

    def loss(qq, kk, vv, bb):
        o, _ = O.fwd(qq, kk, vv, bb, m)
        return float(np.sum(o * do))

    args = [q, k, v, bias]
    for ai, g in enumerate((grads[0], grads[1], grads[2], grads[3])):
        num = np.zeros_like(args[ai])
        it = np.nditer(args[ai], flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            plus = [a.copy() for a in args]
            minus = [a.copy() for a in args]
            plus[ai][idx] += eps
            minus[ai][idx] -= eps
            num[idx] = (loss(*plus) - loss(*minus)) / (2 * eps)
        err = np.abs(num - g).max() / max(np.abs(g).max(), 1e-12)
        assert err < 1e-7, (ai, err)


def test_rows_of_p_sum_to_one():
    q, k, _, _, bias, m = rand_problem(1, 4, 2, 9, 4, seed=3, mask="random")
    v = np.ones_like(k)
    o, _ = O.fwd(q, k, v, bias, m)
    assert np.abs(o - 1.0).max() < 1e-14


def test_uniform_softmax_closed_form():
    """q = 0 and bias = 0: every unmasked key gets weight 1/n, lse = log n."""
    _, k, v, _, _, m = rand_problem(1, 3, 2, 8, 4, seed=4, mask="random")
    q = np.zeros((1, 3, 2, 8, 4))
    bias = np.zeros((1, 2, 8, 8))
    o, lse = O.fwd(q, k, v, bias, m)
    keep = np.isfinite(m)  # [B,No,N]
    for o_ in range(3):
        n = keep[0, o_].sum()
        mean_v = v[0, o_][:, keep[0, o_]].mean(axis=1)  # [H,D]
        assert np.abs(o[0, o_] - mean_v[:, None, :]).max() < 1e-14
        assert np.abs(lse[0, o_] - np.log(n)).max() < 1e-14


def test_per_row_bias_shift():
    q, k, v, do, bias, m = rand_problem(1, 3, 2, 7, 4, seed=6, mask="tail")
    c = np.random.default_rng(0).standard_normal((1, 2, 7, 1)) * 3
    o1, l1 = O.fwd(q, k, v, bias, m)
    o2, l2 = O.fwd(q, k, v, bias + c, m)
    assert np.abs(o1 - o2).max() < 1e-13
    assert np.abs((l2 - l1) - np.broadcast_to(c[:, None, :, :, 0], l1.shape)).max() < 1e-12
    g1 = O.bwd(q, k, v, bias, m, do)
    g2 = O.bwd(q, k, v, bias + c, m, do)
    for a, b in zip(g1, g2):
        assert np.abs(a - b).max() < 1e-12


def test_ds_zero_row_sum_and_dbias_is_sum_over_slices():
    B, No, H, N, D = 1, 5, 2, 6, 4
    q, k, v, do, bias, m = rand_problem(B, No, H, N, D, seed=7, mask="random")
    _, _, _, db = O.bwd(q, k, v, bias, m, do)
    assert np.abs(db.sum(axis=-1)).max() < 1e-13
    acc = np.zeros_like(db)
    for b in range(B):
        for o_ in range(No):
            for h in range(H):
                r = O.slice_(q, k, v, bias, m, do, b, o_, h)
                assert np.abs(r["ds"].sum(axis=-1)).max() < 1e-13
                acc[b, h] += r["ds"]
    assert np.abs(acc - db).max() < 1e-13


def test_dv_column_sum_equals_do_sum():
    q, k, v, do, bias, m = rand_problem(2, 3, 2, 7, 4, seed=8, mask="random")
    _, _, dv, _ = O.bwd(q, k, v, bias, m, do)
    assert np.abs(dv.sum(axis=3) - do.sum(axis=3)).max() < 1e-12


def test_masked_keys_have_zero_grads_and_no_influence():
    q, k, v, do, bias, m = rand_problem(1, 3, 2, 8, 4, seed=9, mask="tail")
    dq, dk, dv, db = O.bwd(q, k, v, bias, m, do)
    masked = ~np.isfinite(m)  # [B,No,N]
    for o_ in range(3):
        assert np.all(dk[0, o_][:, masked[0, o_]] == 0.0)
        assert np.all(dv[0, o_][:, masked[0, o_]] == 0.0)
    # dbias columns of keys masked in every slice are exactly zero
    always = masked.all(axis=1)[0]
    assert np.all(db[0][:, :, always] == 0.0)
    k2, v2 = k.copy(), v.copy()
    k2[masked[:, :, None, :].repeat(2, axis=2)] = 7.0
    v2[masked[:, :, None, :].repeat(2, axis=2)] = -3.0
    o1, _ = O.fwd(q, k, v, bias, m)
    o2, _ = O.fwd(q, k2, v2, bias, m)
    assert np.abs(o1 - o2).max() == 0.0


def test_key_shift_invariance():
    q, k, v, _, bias, m = rand_problem(1, 3, 2, 7, 4, seed=10, mask="random")
    c = np.random.default_rng(1).standard_normal((1, 3, 2, 1, 4))
    o1, _ = O.fwd(q, k, v, bias, m)
    o2, _ = O.fwd(q, k + c, v, bias, m)
    assert np.abs(o1 - o2).max() < 1e-13


def test_permutation_equivariance():
    B, No, H, N, D = 1, 4, 2, 6, 4
    q, k, v, do, bias, m = rand_problem(B, No, H, N, D, seed=12, mask="random")
    perm = np.random.default_rng(2).permutation(N)
    o1, l1 = O.fwd(q, k, v, bias, m)
    g1 = O.bwd(q, k, v, bias, m, do)
    P = lambda x, ax: np.take(x, perm, axis=ax)
    o2, l2 = O.fwd(P(q, 3), P(k, 3), P(v, 3), P(P(bias, 2), 3), P(m, 2))
    g2 = O.bwd(P(q, 3), P(k, 3), P(v, 3), P(P(bias, 2), 3), P(m, 2), P(do, 3))
    assert np.abs(P(o1, 3) - o2).max() < 1e-13
    assert np.abs(P(l1, 3) - l2).max() < 1e-13
    for a, b, axes in zip(g1, g2, [(3,), (3,), (3,), (2, 3)]):
        ap = a
        for ax in axes:
            ap = P(ap, ax)
        assert np.abs(ap - b).max() < 1e-12


def test_fully_masked_row_convention():
    q, k, v, do, bias, _ = rand_problem(1, 3, 2, 5, 4, seed=13)
    m = np.zeros((1, 3, 5))
    m[0, 1, :] = -np.inf  # slice 1: every key masked
    o, lse = O.fwd(q, k, v, bias, m)
    dq, dk, dv, db = O.bwd(q, k, v, bias, m, do)
    assert np.all(o[0, 1] == 0) and np.all(np.isneginf(lse[0, 1]))
    assert np.all(dq[0, 1] == 0) and np.all(dk[0, 1] == 0) and np.all(dv[0, 1] == 0)
    assert np.all(np.isfinite(db))
    # other slices are untouched by the empty one
    m2 = np.zeros((1, 3, 5))
    o2, _ = O.fwd(q, k, v, bias, m2)
    assert np.abs(o[0, [0, 2]] - o2[0, [0, 2]]).max() == 0.0


def test_worked_example_fig6_index_structure():
    """Figure 6: with seven tokens and one head, the bias of pair (4, 6)
    enters the score of query 4 and key 6 in every slice.  Perturbing it
    changes only output rows q = 4, in all seven slices, and its gradient is
    the sum over slices of dS[o, 4, 6]."""
    ex = json.load(open(os.path.join(HERE, "golden", "worked_example_fig6.json")))
    N, H = ex["tokens"], ex["heads"]
    qi, ki = ex["bias_pair"]
    q, k, v, do, bias, _ = rand_problem(1, N, H, N, 4, seed=14)
    o1, _ = O.fwd(q, k, v, bias, None)
    b2 = bias.copy()
    b2[0, 0, qi, ki] += 0.5
    o2, _ = O.fwd(q, k, v, b2, None)
    changed = np.abs(o2 - o1).max(axis=-1)[0, :, 0]  # [No, N]
    assert np.all(changed[:, qi] > 0), "row q=4 must change in every slice"
    others = np.delete(changed, qi, axis=1)
    assert np.all(others == 0.0)
    _, _, _, db = O.bwd(q, k, v, bias, None, do)
    ds_sum = sum(O.slice_(q, k, v, bias, None, do, 0, o_, 0)["ds"][qi, ki] for o_ in range(N))
    assert abs(db[0, 0, qi, ki] - ds_sum) < 1e-14
    # the score of the example's slice o=2 really is the (q=4, k=6) entry: a
    # one-hot V on key 6 reads out P[4, 6] of slice 2 at output row 4
    v1 = np.zeros_like(v)
    v1[0, ex["outer"], 0, ki, 0] = 1.0
    o3, lse = O.fwd(q, k, v1, bias, None)
    s = q[0, ex["outer"], 0, qi] @ k[0, ex["outer"], 0, ki] / 2.0 + bias[0, 0, qi, ki]
    assert abs(o3[0, ex["outer"], 0, qi, 0] - np.exp(s - lse[0, ex["outer"], 0, qi])) < 1e-14


def test_rows_subset_matches_full():
    q, k, v, do, bias, m = rand_problem(1, 4, 2, 10, 4, seed=15, mask="random")
    o, lse = O.fwd(q, k, v, bias, m)
    dq, _, _, db = O.bwd(q, k, v, bias, m, do)
    sel = [0, 3, 9]
    r = O.rows(q, k, v, bias, m, do, 0, 1, sel)
    assert np.abs(r["o"] - o[0, :, 1][:, sel]).max() < 1e-14
    assert np.abs(r["lse"] - lse[0, :, 1][:, sel]).max() < 1e-14
    assert np.abs(r["dq"] - dq[0, :, 1][:, sel]).max() < 1e-14
    assert np.abs(r["dbias"] - db[0, 1][sel]).max() < 1e-13


# --------------------------------------------------------------------------
# Planted mistakes: each edit of the oracle source must be caught by a pin.
# --------------------------------------------------------------------------
MUTATIONS = {
    "drop_bias": ("double sc = dot * scale + bias_bh[(size_t)q * Nk + k];", "double sc = dot * scale;"),
    "drop_mask": ("if (mask_bo) sc += mask_bo[k];", ";"),
    "no_scale": ("const double scale = 1.0 / sqrt((double)D);\n  for (int q = 0; q < Nq; ++q) {",
                 "const double scale = 1.0;\n  for (int q = 0; q < Nq; ++q) {"),
    "delta_sign": ("dSrow[kk] = Prow[kk] * (dp - delta[qq]);", "dSrow[kk] = Prow[kk] * (dp + delta[qq]);"),
    "dk_transposed_operand": ("dK[(size_t)kk * D + d] += dSrow[kk] * Q[(size_t)qq * D + d] * scale;",
                              "dK[(size_t)kk * D + d] += dSrow[kk] * K[(size_t)kk * D + d] * scale;"),
    "dv_uses_ds": ("dV[(size_t)kk * D + d] += Prow[kk] * G[(size_t)qq * D + d];",
                   "dV[(size_t)kk * D + d] += dSrow[kk] * G[(size_t)qq * D + d];"),
    "dbias_last_slice_only": ("dB[(size_t)qq * Nk + kk] += dSrow[kk];", "dB[(size_t)qq * Nk + kk] = dSrow[kk];"),
    "bias_transposed": ("bias_bh[(size_t)q * Nk + k]", "bias_bh[(size_t)k * Nk + q]"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name):
    old, new = MUTATIONS[name]
    src = O.source_text()
    assert old in src, f"mutation anchor missing for {name}"
    lib = O.load_variant(O.compile_variant(src.replace(old, new, 1), name))
    caught = []
    # the last shape has many more slices than threads, so every thread sums
    # several slices of one head into dbias
    for shape in SHAPES[:3] + [(1, 40, 1, 5, 4, "random")]:
        B, No, H, N, D, mk = shape
        q, k, v, do, bias, m = rand_problem(B, No, H, N, D, seed=sum(shape[:5]), mask=mk)
        o, _ = O.fwd(q, k, v, bias, m, lib=lib)
        dq, dk, dv, db = O.bwd(q, k, v, bias, m, do, lib=lib)
        ro, rdq, rdk, rdv, rdb = torch_reference(q, k, v, bias, m, do)
        errs = [rel_err(a, b) for a, b in [(o, ro), (dq, rdq), (dk, rdk), (dv, rdv), (db, rdb)]]
        caught.append(max(errs) > 1e-6)
    assert any(caught), f"planted mistake {name} was not caught"
