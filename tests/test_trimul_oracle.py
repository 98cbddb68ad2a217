"""Pins of the FP64 oracle of the triangle multiplicative update
(oracle/trimul.py; "TurboPairFormer", Figure 12 and Table 10).

Checked against things other than itself: FP64 torch autograd of an
independently written update, central finite differences, the contraction
written as explicit loops, the identity that relates the two directions
(the incoming contraction of Z is the outgoing contraction of the
pair-transposed Z), which pairs each output pair depends on, and the
isolation of masked pairs.
"""
import itertools

import numpy as np
import pytest
import torch

from oracle import trimul as TM


def make(B, N, Cz, Ch, seed, masked=False):
    g = np.random.default_rng(seed)
    z = g.standard_normal((B, N, N, Cz))
    ln_in_w = 1.0 + 0.1 * g.standard_normal(Cz)
    ln_in_b = 0.1 * g.standard_normal(Cz)
    w_p = g.standard_normal((Cz, 4 * Ch + Cz)) / np.sqrt(Cz)
    ln_out_w = 1.0 + 0.1 * g.standard_normal(Ch)
    ln_out_b = 0.1 * g.standard_normal(Ch)
    w_o = g.standard_normal((Ch, Cz)) / np.sqrt(Ch)
    mask = None
    if masked:
        mask = (g.random((B, N, N)) > 0.2).astype(np.float64)
    return z, mask, ln_in_w, ln_in_b, w_p, ln_out_w, ln_out_b, w_o


def torch_update(z, mask, ln_in_w, ln_in_b, w_p, ln_out_w, ln_out_b, w_o, direction):
    """The update written directly in torch (float64), for autograd."""
    Ch, Cz = w_o.shape
    x = torch.nn.functional.layer_norm(z, (Cz,), ln_in_w, ln_in_b, eps=1e-5)
    p = x @ w_p
    m = torch.ones_like(z[..., :1]) if mask is None else mask[..., None]
    a = m * torch.sigmoid(p[..., Ch:2 * Ch]) * p[..., :Ch]
    b = m * torch.sigmoid(p[..., 3 * Ch:4 * Ch]) * p[..., 2 * Ch:3 * Ch]
    if direction == "outgoing":
        X = torch.einsum("bikc,bjkc->bijc", a, b)
    else:
        X = torch.einsum("bkic,bkjc->bijc", a, b)
    y = torch.nn.functional.layer_norm(X, (Ch,), ln_out_w, ln_out_b, eps=1e-5)
    return torch.sigmoid(p[..., 4 * Ch:]) * (y @ w_o)


PARAMS = ("z", "ln_in_w", "ln_in_b", "w_p", "ln_out_w", "ln_out_b", "w_o")
GRADS = ("dz", "dln_in_w", "dln_in_b", "dw_p", "dln_out_w", "dln_out_b", "dw_o")


@pytest.mark.parametrize("direction", TM.DIRECTIONS)
@pytest.mark.parametrize("shape,masked", [((1, 5, 6, 4), False), ((2, 4, 8, 3), True)])
def test_matches_torch_autograd(direction, shape, masked):
    B, N, Cz, Ch = shape
    z, mask, *w = make(B, N, Cz, Ch, seed=N * Cz + Ch, masked=masked)
    d_out = np.random.default_rng(2).standard_normal((B, N, N, Cz))
    f = TM.fwd(z, mask, *w, direction)
    gr = TM.bwd(z, mask, *w, d_out, direction)
    ts = [torch.tensor(a, requires_grad=True) for a in [z] + w]
    tm = None if mask is None else torch.tensor(mask)
    out = torch_update(ts[0], tm, *ts[1:], direction)
    out.backward(torch.tensor(d_out))
    np.testing.assert_allclose(f["out"], out.detach().numpy(), rtol=1e-10, atol=1e-12)
    for name, t in zip(GRADS, ts):
        np.testing.assert_allclose(gr[name], t.grad.numpy(), rtol=1e-8, atol=1e-10, err_msg=name)


@pytest.mark.parametrize("direction", TM.DIRECTIONS)
def test_finite_differences(direction):
    B, N, Cz, Ch = 1, 4, 4, 3
    z, mask, *w = make(B, N, Cz, Ch, seed=7, masked=True)
    d_out = np.random.default_rng(3).standard_normal((B, N, N, Cz))
    gr = TM.bwd(z, mask, *w, d_out, direction)
    args = [z] + w

    def loss(*a):
        return float((TM.fwd(a[0], mask, *a[1:], direction)["out"] * d_out).sum())

    rng = np.random.default_rng(9)
    eps = 1e-6
    for i, name in enumerate(GRADS):
        for _ in range(5):
            idx = tuple(int(rng.integers(s)) for s in args[i].shape)
            plus = [a.copy() for a in args]
            minus = [a.copy() for a in args]
            plus[i][idx] += eps
            minus[i][idx] -= eps
            fd = (loss(*plus) - loss(*minus)) / (2 * eps)
            assert abs(fd - gr[name][idx]) <= 1e-6 * max(1.0, abs(fd)), (name, idx, fd, gr[name][idx])


def test_contraction_matches_explicit_loops():
    rng = np.random.default_rng(4)
    B, N, C = 2, 4, 3
    a = rng.standard_normal((B, N, N, C))
    b = rng.standard_normal((B, N, N, C))
    out = TM.contract(a, b, "outgoing")
    inc = TM.contract(a, b, "incoming")
    for bb, i, j, c in itertools.product(range(B), range(N), range(N), range(C)):
        so = si = 0.0
        for k in range(N):
            so += a[bb, i, k, c] * b[bb, j, k, c]   # edges i->k and j->k
            si += a[bb, k, i, c] * b[bb, k, j, c]   # edges k->i and k->j
        assert abs(out[bb, i, j, c] - so) < 1e-12
        assert abs(inc[bb, i, j, c] - si) < 1e-12


def test_incoming_is_outgoing_of_the_transposed_pairs():
    """Swapping the two token axes of Z (and of the mask) turns one direction
    into the other: the incoming contraction of Z equals the outgoing
    contraction of the swapped Z, pair for pair (sum_k a[k,i] b[k,j] =
    sum_k a'[i,k] b'[j,k] with a'[r,s] = a[s,r]), and so does the projected
    u = LayerNorm(X) W_o.  The output gate is not part of the identity: it
    reads pair (i, j) of its own input."""
    B, N, Cz, Ch = 1, 6, 5, 4
    z, mask, *w = make(B, N, Cz, Ch, seed=11, masked=True)
    swap = lambda t: None if t is None else np.swapaxes(t, 1, 2)  # noqa: E731
    inc = TM.fwd(z, mask, *w, "incoming")
    out_t = TM.fwd(swap(z), swap(mask), *w, "outgoing")
    np.testing.assert_allclose(inc["X"], out_t["X"], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(inc["u"], out_t["u"], rtol=1e-12, atol=1e-12)
    # and the directions really differ on generic inputs
    assert np.abs(inc["X"] - TM.fwd(z, mask, *w, "outgoing")["X"]).max() > 1e-3


@pytest.mark.parametrize("direction", TM.DIRECTIONS)
def test_dependency_structure(direction):
    """Outgoing: output pair (i, j) depends on the pairs of rows i and j
    (edges leaving i and j); incoming: on the pairs of columns i and j."""
    B, N, Cz, Ch = 1, 5, 4, 3
    z, mask, *w = make(B, N, Cz, Ch, seed=5)
    i, j = 1, 3
    base = TM.fwd(z, mask, *w, direction)["out"][0, i, j]
    for r, s in itertools.product(range(N), range(N)):
        z2 = z.copy()
        z2[0, r, s] += np.linspace(-1.0, 1.0, Cz)
        changed = np.abs(TM.fwd(z2, mask, *w, direction)["out"][0, i, j] - base).max() > 1e-12
        hit = (r in (i, j)) if direction == "outgoing" else (s in (i, j))
        assert changed == hit, (r, s)


@pytest.mark.parametrize("direction", TM.DIRECTIONS)
def test_masked_pair_only_reaches_its_own_gate(direction):
    """A masked pair contributes nothing to the contraction: changing it
    changes only its own output pair (through the output gate)."""
    B, N, Cz, Ch = 1, 5, 4, 3
    z, _, *w = make(B, N, Cz, Ch, seed=6)
    mask = np.ones((B, N, N))
    mask[0, 2, 4] = 0.0
    base = TM.fwd(z, mask, *w, direction)["out"]
    z2 = z.copy()
    z2[0, 2, 4] += 3.0 * np.linspace(-1.0, 1.0, Cz)
    diff = np.abs(TM.fwd(z2, mask, *w, direction)["out"] - base).max(axis=-1)[0]
    assert diff[2, 4] > 1e-6
    diff[2, 4] = 0.0
    assert diff.max() < 1e-12


def test_planted_mistake_swapped_branches_is_caught():
    """Taking a from the b columns (a plausible slip in the column order) must
    fail the autograd comparison."""
    B, N, Cz, Ch = 1, 4, 5, 3
    z, mask, *w = make(B, N, Cz, Ch, seed=8)
    orig = TM.split_projection

    def wrong(p, Ch_):
        av, ag, bv, bg, g = orig(p, Ch_)
        return bv, bg, av, ag, g

    TM.split_projection = wrong
    try:
        bad = TM.fwd(z, mask, *w, "outgoing")["out"]
    finally:
        TM.split_projection = orig
    ref = torch_update(*(torch.tensor(a) for a in [z]), None, *(torch.tensor(a) for a in w), "outgoing").numpy()
    assert np.abs(bad - ref).max() > 1e-3


@pytest.mark.parametrize("direction", TM.DIRECTIONS)
def test_fwd_pairs_matches_full_forward(direction):
    """The per-pair forward used for sampled full-size checks gives the full
    forward's values at the listed pairs."""
    B, N, Cz, Ch = 2, 6, 5, 4
    z, mask, *w = make(B, N, Cz, Ch, seed=12, masked=True)
    full = TM.fwd(z, mask, *w, direction)["out"]
    pairs = [(0, 1, 4), (1, 5, 0), (1, 2, 2), (0, 0, 5)]
    got = TM.fwd_pairs(z, mask, *w, direction, pairs)
    for r, (b, i, j) in enumerate(pairs):
        np.testing.assert_allclose(got[r], full[b, i, j], rtol=1e-12, atol=1e-13)
