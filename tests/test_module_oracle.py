"""Pins of the FP64 module oracle (oracle/module.py): LayerNorm, projections
into q, k, v and the pair bias, the attention core, and the output
projection, forward and backward ("TurboPairFormer", Figure 6).

The oracle is checked against things other than itself: FP64 torch autograd
of an independently written module, central finite differences, the
LayerNorm's invariances, and the dependency structure of the worked example
(which pairs an output pair depends on).
"""
import numpy as np
import pytest
import torch

from oracle import module as M

pytestmark = pytest.mark.filterwarnings("ignore::UserWarning")


def make(B, N, C, H, D, seed, masked=False):
    g = np.random.default_rng(seed)
    z = g.standard_normal((B, N, N, C))
    gamma = 1.0 + 0.1 * g.standard_normal(C)
    beta = 0.1 * g.standard_normal(C)
    w_in = g.standard_normal((C, 3 * H * D + H)) / np.sqrt(C)
    w_o = g.standard_normal((H * D, C)) / np.sqrt(H * D)
    mask = None
    if masked:
        mask = np.zeros((B, N, N))
        mask[:, :, N - 1] = -np.inf
        mask[:, 0, 1] = -np.inf
    return z, mask, gamma, beta, w_in, w_o


def torch_module(z, mask, gamma, beta, w_in, w_o, H, D):
    """The module written directly in torch (float64), for autograd."""
    B, N, _, C = z.shape
    x = torch.nn.functional.layer_norm(z, (C,), gamma, beta, eps=1e-5)
    p = x @ w_in
    HD = H * D
    q = p[..., :HD].reshape(B, N, N, H, D)             # [b, o, q, h, d]
    k = p[..., HD:2 * HD].reshape(B, N, N, H, D)       # [b, o, k, h, d]
    v = p[..., 2 * HD:3 * HD].reshape(B, N, N, H, D)
    bias = p[..., 3 * HD:]                             # [b, q, k, h]: pair (q, k)
    s = torch.einsum("boqhd,bokhd->bohqk", q, k) / np.sqrt(D) + bias.permute(0, 3, 1, 2)[:, None]
    if mask is not None:
        s = s + mask[:, :, None, None, :]
    a = torch.softmax(s, dim=-1)
    o = torch.einsum("bohqk,bokhd->boqhd", a, v).reshape(B, N, N, HD)
    return o @ w_o


@pytest.mark.parametrize("shape,masked", [((1, 6, 8, 2, 4), False), ((2, 5, 6, 3, 2), True)])
def test_module_matches_torch_autograd(shape, masked):
    B, N, C, H, D = shape
    z, mask, gamma, beta, w_in, w_o = make(B, N, C, H, D, seed=N + C, masked=masked)
    g = np.random.default_rng(7)
    d_out = g.standard_normal((B, N, N, C))
    f = M.fwd(z, mask, gamma, beta, w_in, w_o, H, D)
    gr = M.bwd(z, mask, gamma, beta, w_in, w_o, d_out, H, D)
    tz, tg, tb, twi, two = (torch.tensor(a, requires_grad=True) for a in (z, gamma, beta, w_in, w_o))
    tm = None if mask is None else torch.tensor(mask)
    out = torch_module(tz, tm, tg, tb, twi, two, H, D)
    out.backward(torch.tensor(d_out))
    np.testing.assert_allclose(f["out"], out.detach().numpy(), rtol=1e-10, atol=1e-11)
    for name, t in (("dz", tz), ("dgamma", tg), ("dbeta", tb), ("dw_in", twi), ("dw_o", two)):
        np.testing.assert_allclose(gr[name], t.grad.numpy(), rtol=1e-8, atol=1e-10, err_msg=name)


def test_module_finite_differences():
    B, N, C, H, D = 1, 4, 5, 2, 3
    z, mask, gamma, beta, w_in, w_o = make(B, N, C, H, D, seed=3, masked=True)
    d_out = np.random.default_rng(11).standard_normal((B, N, N, C))
    gr = M.bwd(z, mask, gamma, beta, w_in, w_o, d_out, H, D)

    def loss(z_, gamma_, beta_, w_in_, w_o_):
        return float((M.fwd(z_, mask, gamma_, beta_, w_in_, w_o_, H, D)["out"] * d_out).sum())

    args = [z, gamma, beta, w_in, w_o]
    names = ["dz", "dgamma", "dbeta", "dw_in", "dw_o"]
    rng = np.random.default_rng(5)
    eps = 1e-6
    for a_i, name in enumerate(names):
        for _ in range(6):
            idx = tuple(int(rng.integers(s)) for s in args[a_i].shape)
            plus = [a.copy() for a in args]
            minus = [a.copy() for a in args]
            plus[a_i][idx] += eps
            minus[a_i][idx] -= eps
            fd = (loss(*plus) - loss(*minus)) / (2 * eps)
            assert abs(fd - gr[name][idx]) <= 1e-6 * max(1.0, abs(fd)), (name, idx, fd, gr[name][idx])


def test_layernorm_closed_forms_and_pair_shift_invariance():
    """xhat has zero mean and variance var / (var + eps) per pair; adding a
    constant to all features of one pair leaves the module output unchanged
    (the LayerNorm removes it)."""
    B, N, C, H, D = 1, 5, 8, 2, 4
    z, mask, gamma, beta, w_in, w_o = make(B, N, C, H, D, seed=1)
    x, xhat, rstd = M.layernorm(z, gamma, beta)
    np.testing.assert_allclose(xhat.mean(-1), 0.0, atol=1e-12)
    # mean(xhat^2) = var / (var + eps) = 1 - eps * rstd^2
    np.testing.assert_allclose((xhat ** 2).mean(-1), 1.0 - 1e-5 * rstd[..., 0] ** 2, rtol=1e-12)
    base = M.fwd(z, mask, gamma, beta, w_in, w_o, H, D)["out"]
    z2 = z.copy()
    z2[0, 2, 3, :] += 7.5
    shifted = M.fwd(z2, mask, gamma, beta, w_in, w_o, H, D)["out"]
    np.testing.assert_allclose(shifted, base, rtol=1e-10, atol=1e-12)


def test_worked_example_dependency_structure():
    """Figure 6: the output of pair (o, q) = (2, 4) depends on the pairs of
    slice 2 (its query (2, 4) and the keys / values (2, k)) and on the bias
    pairs (4, k) of query 4, and on no other pair."""
    B, N, C, H, D = 1, 7, 6, 2, 3
    z, mask, gamma, beta, w_in, w_o = make(B, N, C, H, D, seed=9)
    base = M.fwd(z, mask, gamma, beta, w_in, w_o, H, D)["out"][0, 2, 4]
    for i in range(N):
        for j in range(N):
            z2 = z.copy()
            z2[0, i, j, :] += np.linspace(-1.0, 1.0, C)
            changed = np.abs(M.fwd(z2, mask, gamma, beta, w_in, w_o, H, D)["out"][0, 2, 4] - base).max() > 1e-12
            assert changed == (i == 2 or i == 4), (i, j)


def test_planted_mistake_in_projection_split_is_caught():
    """A plausible mistake -- taking the bias from pair (k, q) instead of
    (q, k) -- must fail the autograd comparison above."""
    B, N, C, H, D = 1, 5, 6, 2, 3
    z, mask, gamma, beta, w_in, w_o = make(B, N, C, H, D, seed=4)
    orig = M.split_projection

    def wrong(p, H_, D_):
        q, k, v, bias = orig(p, H_, D_)
        return q, k, v, bias.transpose(0, 1, 3, 2)

    M.split_projection = wrong
    try:
        bad = M.fwd(z, mask, gamma, beta, w_in, w_o, H, D)["out"]
    finally:
        M.split_projection = orig
    tz, tg, tb, twi, two = (torch.tensor(a) for a in (z, gamma, beta, w_in, w_o))
    ref = torch_module(tz, None, tg, tb, twi, two, H, D).numpy()
    assert np.abs(bad - ref).max() > 1e-3


def test_fwd_pairs_matches_full_forward():
    """The per-pair forward used for sampled full-size checks gives the full
    forward's values at the listed pairs (masked slices included)."""
    B, N, C, H, D = 2, 6, 8, 2, 3
    z, mask, gamma, beta, w_in, w_o = make(B, N, C, H, D, seed=13, masked=True)
    full = M.fwd(z, mask, gamma, beta, w_in, w_o, H, D)["out"]
    pairs = [(0, 1, 4), (1, 5, 0), (1, 2, 2), (0, 0, 5)]
    got = M.fwd_pairs(z, mask, gamma, beta, w_in, w_o, H, D, pairs)
    for r, (b, i, j) in enumerate(pairs):
        np.testing.assert_allclose(got[r], full[b, i, j], rtol=1e-12, atol=1e-13)
