"""GPU parity of the triangle-attention module (LayerNorm, projections into
q, k, v and the bias, the core, output projection; "TurboPairFormer",
Figure 6) through the C ABI, against the FP64 module oracle on the same
seeded BF16 inputs.

Tolerances (relative RMSE against FP64): out <= 1e-2, every gradient
(dz, dgamma, dbeta, dW_in, dW_o) <= 2e-2.  The module adds four BF16
roundings to the core's own error (x, the projection P, the core output
once more through o_flat, and out; in the backward d_oflat and dP), each a
relative 2^-8 at most (BF16 round to nearest), on top of the core's 4e-3 / 1e-2 bars; the bars
here leave about a factor two over the core's.
"""
import json

import numpy as np
import pytest
import torch

from parity_utils import LN_ROW_SUM_BOUND, cpu64, rel_rmse
from oracle import module as MO
from protein_folding_triangle_gb300 import synthetic as S
from protein_folding_triangle_gb300 import triattn as T

pytestmark = pytest.mark.gpu

TOL_OUT = 1e-2
TOL_GRADS = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from protein_folding_triangle_gb300 import build
    build.build()
    T.load()


def run_gpu(x):
    dev = {k: (v.cuda().contiguous() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    H, D = x["H"], x["D"]
    out, ctx = T.tri_attn_module_fwd(dev["z"], dev["mask"], dev["ln_w"], dev["ln_b"], dev["w_in"], dev["w_o"], H, D)
    grads = T.tri_attn_module_bwd(dev["z"], dev["mask"], dev["ln_w"], dev["w_in"], dev["w_o"], ctx, dev["d_out"],
                                  H, D)
    torch.cuda.synchronize()
    assert T.device_status() == T.OK
    return out, grads


def run_oracle(x):
    args = (x["z"], x["mask"], x["ln_w"], x["ln_b"], x["w_in"], x["w_o"])
    f = MO.fwd(*args, x["H"], x["D"])
    g = MO.bwd(*args, x["d_out"], x["H"], x["D"])
    return f["out"], g


CASES = [
    # (B, N, C, H, D, mask_frac): one tile, a ragged tail, several tiles
    (1, 40, 64, 2, 16, 0.0),
    (2, 48, 32, 1, 32, 0.2),
    (1, 136, 128, 4, 32, 0.1),
    # LayerNorm runs of 3 and 6 features per lane (scalar and 4-byte accesses);
    # H = 3 gives a projection width of 291 (padded to 296)
    (1, 40, 96, 2, 16, 0.0),
    (1, 32, 192, 3, 32, 0.1),
    # N a multiple of 32: q, k, v, the bias planes and dO written by the GEMM
    # epilogues in the core's layout (the cases above with other N read the
    # pair rows in place); D = 16 with H = 3 puts a head and the bias columns
    # in one 32-column chunk
    (1, 64, 64, 3, 16, 0.1),
    (2, 32, 128, 4, 32, 0.2),
]


@pytest.mark.parametrize("case", CASES, ids=[f"B{c[0]}N{c[1]}C{c[2]}H{c[3]}D{c[4]}" for c in CASES])
def test_module_matches_oracle(case):
    B, N, C, H, D, mf = case
    x = S.make_module_inputs(B, N, C, H, D, seed=N + C, mask_frac=mf)
    out, (dz, dlw, dlb, dwi, dwo) = run_gpu(x)
    ref_out, ref = run_oracle(x)
    errs = {"out": rel_rmse(cpu64(out), ref_out), "dz": rel_rmse(cpu64(dz), ref["dz"]),
            "dgamma": rel_rmse(cpu64(dlw), ref["dgamma"]), "dbeta": rel_rmse(cpu64(dlb), ref["dbeta"]),
            "dw_in": rel_rmse(cpu64(dwi), ref["dw_in"]), "dw_o": rel_rmse(cpu64(dwo), ref["dw_o"])}
    print(json.dumps({"case": list(case), **{k: round(v, 6) for k, v in errs.items()}}))
    assert errs["out"] <= TOL_OUT, errs
    for k in ("dz", "dgamma", "dbeta", "dw_in", "dw_o"):
        assert errs[k] <= TOL_GRADS, (k, errs)


def test_module_bitwise_deterministic():
    x = S.make_module_inputs(1, 72, 64, 2, 32, seed=3, mask_frac=0.1)
    first = None
    for _ in range(3):
        out, grads = run_gpu(x)
        cur = [out.view(torch.int16).cpu()] + [g.contiguous().view(torch.int16).cpu() for g in grads]
        if first is None:
            first = cur
        else:
            for a, b in zip(first, cur):
                assert torch.equal(a, b)


def test_module_layernorm_statistics_in_ctx():
    """The saved x is LayerNorm(z) rounded to BF16: compared element by
    element with the oracle's x (first bytes of ctx)."""
    B, N, C, H, D = 1, 24, 96, 2, 16
    x = S.make_module_inputs(B, N, C, H, D, seed=5)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    _, ctx = T.tri_attn_module_fwd(dev["z"], None, dev["ln_w"], dev["ln_b"], dev["w_in"], dev["w_o"], H, D)
    torch.cuda.synchronize()
    xg = ctx[:B * N * N * C * 2].view(torch.bfloat16).reshape(B, N, N, C)
    ref, _, _ = MO.layernorm(cpu64(x["z"]), cpu64(x["ln_w"]), cpu64(x["ln_b"]))
    # one BF16 rounding of an FP32 value: relative 2^-8 at most per element
    err = np.abs(cpu64(xg) - ref)
    assert np.all(err <= 2.0 ** -8 * np.abs(ref) + 1e-6), float(err.max())


def test_module_rejects_bad_shapes_without_launching():
    z = torch.zeros((1, 40, 40, 48), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(48, dtype=torch.float32, device="cuda")
    with pytest.raises(T.TriAttnError):
        T.tri_attn_module_fwd(z, None, w, w, torch.zeros((48, 3 * 32 + 2), dtype=torch.bfloat16, device="cuda"),
                              torch.zeros((32, 48), dtype=torch.bfloat16, device="cuda"), 2, 16)


def layernorm_row_sums_ok(dz):
    """The LayerNorm makes the output invariant to a constant shift of one
    pair's features, so sum_c dz[m, c] = 0 for every pair m, up to the BF16
    rounding of dz and an FP32 residual (LN_ROW_SUM_BOUND)."""
    d = dz.float().reshape(-1, dz.shape[-1]).double()
    s = d.sum(dim=1).abs()
    bound = LN_ROW_SUM_BOUND * d.abs().sum(dim=1) + 1e-30
    return bool((s <= bound).all()), float((s / bound).max())


def test_module_full_size_sampled():
    """crop768 module (B=1, N=768, C=128, H=4, D=32, tail key mask) at the
    bench's size: 12 sampled output pairs against the per-pair oracle, the
    LayerNorm row sums of dz, and bitwise repeatability of a second call."""
    B, N, C, H, D = 1, 768, 128, 4, 32
    x = S.make_module_inputs(B, N, C, H, D, seed=0, mask_frac=0.08)
    out, grads = run_gpu(x)
    rng = np.random.default_rng(21)
    pairs = [(0, int(rng.integers(N)), int(rng.integers(N))) for _ in range(10)] + [(0, 0, N - 1), (0, N - 1, 3)]
    ref = MO.fwd_pairs(x["z"], x["mask"], x["ln_w"], x["ln_b"], x["w_in"], x["w_o"], H, D, pairs)
    got = np.stack([cpu64(out[b, i, j]) for (b, i, j) in pairs])
    err = rel_rmse(got, ref)
    ok, ratio = layernorm_row_sums_ok(grads[0])
    print(json.dumps({"case": "module crop768 C=128 sampled", "out_sampled": round(err, 6),
                      "dz_row_sum_ratio_max": round(ratio, 4)}))
    assert err <= TOL_OUT
    assert ok
    out2, grads2 = run_gpu(x)
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    for a, b in zip(grads, grads2):
        assert torch.equal(a.contiguous().view(torch.int16), b.contiguous().view(torch.int16))


def test_module_autograd_matches_direct_calls():
    """TriangleAttention (nn.Module + autograd) returns the direct calls'
    output and gradients (FP32 gradients cast to each parameter's dtype)."""
    from protein_folding_triangle_gb300 import layers
    B, N, C, H, D = 1, 40, 64, 2, 16
    x = S.make_module_inputs(B, N, C, H, D, seed=31, mask_frac=0.1)
    dev = {k: (v.cuda().contiguous() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    m = layers.TriangleAttention(C, H, D, device="cuda")
    with torch.no_grad():
        m.ln_w.copy_(dev["ln_w"])
        m.ln_b.copy_(dev["ln_b"])
        m.w_in.copy_(dev["w_in"])
        m.w_o.copy_(dev["w_o"])
    z = dev["z"].clone().requires_grad_(True)
    out = m(z, dev["mask"])
    out.backward(dev["d_out"])
    ref_out, grads = run_gpu(x)
    assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
    assert torch.equal(z.grad.view(torch.int16), grads[0].view(torch.int16))
    for p, g in ((m.ln_w, grads[1]), (m.ln_b, grads[2]), (m.w_in, grads[3]), (m.w_o, grads[4])):
        assert torch.equal(p.grad, g.to(p.dtype))
