"""GPU parity of the triangle multiplicative update, outgoing and incoming
("TurboPairFormer", Figure 12), through the C ABI, against the FP64 oracle
on the same seeded BF16 inputs.

Tolerances (relative RMSE against FP64): out <= 1e-2, every gradient
<= 2e-2.  The CUDA path rounds to BF16 at x, the gated operands a and b (the
projection p stays in FP32 accumulators), g, the contraction output X,
y = LayerNorm(X), u and out (forward), and at du, dX, dA, dB and dp
(backward); each rounding is a relative 2^-8 at most, the gates use the
hardware tanh (relative error about 2^-11), and the GEMMs accumulate in FP32.  Seven to eight such roundings in
sequence give a few 1e-3, the bars leave a factor two to four.
"""
import json

import numpy as np
import pytest
import torch

from parity_utils import LN_ROW_SUM_BOUND, cpu64, rel_rmse
from oracle import trimul as TMO
from protein_folding_triangle_gb300 import synthetic as S
from protein_folding_triangle_gb300 import triattn as T

pytestmark = pytest.mark.gpu

TOL_OUT = 1e-2
TOL_GRADS = 2e-2
NAMES = ("dz", "dln_in_w", "dln_in_b", "dw_p", "dln_out_w", "dln_out_b", "dw_o")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from protein_folding_triangle_gb300 import build
    build.build()
    T.load()


def run_gpu(x, direction):
    d = {k: (v.cuda().contiguous() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    out, ctx = T.triattn_trimul_fwd(d["z"], d["mask"], d["ln_in_w"], d["ln_in_b"], d["w_p"], d["ln_out_w"],
                                    d["ln_out_b"], d["w_o"], direction)
    grads = T.triattn_trimul_bwd(d["z"], d["mask"], d["ln_in_w"], d["w_p"], d["ln_out_w"], d["w_o"], ctx,
                                 d["d_out"], direction)
    torch.cuda.synchronize()
    return out, grads


def run_oracle(x, direction):
    args = (x["z"], x["mask"], x["ln_in_w"], x["ln_in_b"], x["w_p"], x["ln_out_w"], x["ln_out_b"], x["w_o"])
    return TMO.fwd(*args, direction)["out"], TMO.bwd(*args, x["d_out"], direction)


CASES = [
    # (B, N, C_z, C_h, pad_frac)
    (1, 40, 64, 32, 0.0),
    (2, 48, 32, 64, 0.2),
    (1, 136, 128, 128, 0.1),
    # input-LayerNorm runs of 3, 5 and 8 features per lane (scalar and 16-byte
    # accesses), and C_h = 96 (three channel-major loads per thread, two
    # threads per channel in the output-LayerNorm sums, the rest idle)
    (1, 48, 96, 96, 0.1),
    (1, 40, 160, 32, 0.0),
    (1, 40, 256, 64, 0.0),
]


@pytest.mark.parametrize("direction", ["outgoing", "incoming"])
@pytest.mark.parametrize("case", CASES, ids=[f"B{c[0]}N{c[1]}Cz{c[2]}Ch{c[3]}" for c in CASES])
def test_trimul_matches_oracle(case, direction):
    B, N, Cz, Ch, pad = case
    x = S.make_trimul_inputs(B, N, Cz, Ch, seed=N + Cz + Ch, pad_frac=pad)
    out, grads = run_gpu(x, direction)
    ref_out, ref = run_oracle(x, direction)
    errs = {"out": rel_rmse(cpu64(out), ref_out)}
    for name, g in zip(NAMES, grads):
        errs[name] = rel_rmse(cpu64(g), ref[name])
    print(json.dumps({"case": list(case), "direction": direction, **{k: round(v, 6) for k, v in errs.items()}}))
    assert errs["out"] <= TOL_OUT, errs
    for name in NAMES:
        assert errs[name] <= TOL_GRADS, (name, errs)


def test_trimul_padding_pairs_get_no_gradient_through_the_contraction():
    """Pairs whose mask is 0 contribute nothing to X: their dz comes only
    from their own output gate, so with d_out zero on them it is exactly 0."""
    B, N, Cz, Ch = 1, 40, 64, 32
    x = S.make_trimul_inputs(B, N, Cz, Ch, seed=1, pad_frac=0.2)
    keep = x["mask"].float()
    x["d_out"] = (x["d_out"].float() * keep[..., None]).to(torch.bfloat16)
    _, grads = run_gpu(x, "outgoing")
    dz = grads[0].float().cpu()
    assert torch.count_nonzero(dz[keep == 0]) == 0
    assert torch.count_nonzero(dz[keep == 1]) > 0


def test_trimul_bitwise_deterministic():
    x = S.make_trimul_inputs(1, 64, 64, 64, seed=4, pad_frac=0.1)
    for direction in ("outgoing", "incoming"):
        first = None
        for _ in range(3):
            out, grads = run_gpu(x, direction)
            cur = [out.view(torch.int16).cpu()] + [g.contiguous().view(torch.int32 if g.dtype == torch.float32
                                                                        else torch.int16).cpu() for g in grads]
            if first is None:
                first = cur
            else:
                for a, b in zip(first, cur):
                    assert torch.equal(a, b)


@pytest.mark.parametrize("direction", ["outgoing", "incoming"])
def test_trimul_full_size_every_element(direction):
    """Table 10's largest shape (B=1, N=768, C_z=C_h=128, 8% padding tokens):
    out and every gradient against the full FP64 oracle, element by element
    (relative RMSE over the whole tensor)."""
    B, N, C = 1, 768, 128
    x = S.make_trimul_inputs(B, N, C, C, seed=1, pad_frac=0.08)
    out, grads = run_gpu(x, direction)
    args = (x["z"], x["mask"], x["ln_in_w"], x["ln_in_b"], x["w_p"], x["ln_out_w"], x["ln_out_b"], x["w_o"])
    ref = TMO.bwd(*args, x["d_out"], direction)
    errs = {"out": rel_rmse(cpu64(out), ref["out"])}
    for name, g in zip(NAMES, grads):
        errs[name] = rel_rmse(cpu64(g), ref[name])
    print(json.dumps({"case": f"trimul N768 C128 {direction} every element",
                      **{k: round(v, 6) for k, v in errs.items()}}))
    assert errs["out"] <= TOL_OUT, errs
    for name in NAMES:
        assert errs[name] <= TOL_GRADS, (name, errs)


@pytest.mark.parametrize("direction", ["outgoing", "incoming"])
def test_trimul_full_size_sampled(direction):
    """Table 10's largest shape (B=1, N=768, C_z=C_h=128) with 8% padding
    tokens: 12 sampled output pairs against the per-pair oracle, the input
    LayerNorm's row sums of dz (sum_c dz[m, c] = 0 up to the BF16 rounding
    of dz and an FP32 residual, LN_ROW_SUM_BOUND), and
    bitwise repeatability of a second call."""
    B, N, C = 1, 768, 128
    x = S.make_trimul_inputs(B, N, C, C, seed=0, pad_frac=0.08)
    out, grads = run_gpu(x, direction)
    rng = np.random.default_rng(22)
    pairs = [(0, int(rng.integers(N)), int(rng.integers(N))) for _ in range(10)] + [(0, 0, N - 1), (0, N - 1, 5)]
    args = (x["z"], x["mask"], x["ln_in_w"], x["ln_in_b"], x["w_p"], x["ln_out_w"], x["ln_out_b"], x["w_o"])
    ref = TMO.fwd_pairs(*args, direction, pairs)
    got = np.stack([cpu64(out[b, i, j]) for (b, i, j) in pairs])
    err = rel_rmse(got, ref)
    d = grads[0].float().reshape(-1, C).double()
    s = d.sum(dim=1).abs()
    bound = LN_ROW_SUM_BOUND * d.abs().sum(dim=1) + 1e-30
    print(json.dumps({"case": f"trimul N768 C128 {direction} sampled", "out_sampled": round(err, 6),
                      "dz_row_sum_ratio_max": round(float((s / bound).max()), 4)}))
    assert err <= TOL_OUT
    assert bool((s <= bound).all())
    out2, grads2 = run_gpu(x, direction)
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(grads[3].view(torch.int32), grads2[3].view(torch.int32))


@pytest.mark.parametrize("direction", ["outgoing", "incoming"])
def test_trimul_autograd_matches_direct_calls(direction):
    """TriangleMultiplication (nn.Module + autograd) returns the direct calls'
    output and gradients (FP32 gradients cast to each parameter's dtype)."""
    from protein_folding_triangle_gb300 import layers
    B, N, Cz, Ch = 1, 40, 64, 32
    x = S.make_trimul_inputs(B, N, Cz, Ch, seed=32, pad_frac=0.1)
    dev = {k: (v.cuda().contiguous() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    m = layers.TriangleMultiplication(Cz, Ch, direction, device="cuda")
    names = ("ln_in_w", "ln_in_b", "w_p", "ln_out_w", "ln_out_b", "w_o")
    with torch.no_grad():
        for n in names:
            getattr(m, n).copy_(dev[n])
    z = dev["z"].clone().requires_grad_(True)
    out = m(z, dev["mask"])
    out.backward(dev["d_out"])
    ref_out, grads = run_gpu(x, direction)
    assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
    assert torch.equal(z.grad.view(torch.int16), grads[0].view(torch.int16))
    for n, g in zip(names, grads[1:]):
        p = getattr(m, n)
        assert torch.equal(p.grad, g.to(p.dtype))
