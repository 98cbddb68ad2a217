"""The core on tensors in other row layouts (tri_attn_fwd_strided /
tri_attn_bwd_strided): q, k, v read from and dq, dk, dv written into the
pair rows of one projection-like matrix, o, its residual and dO in pair rows
of their own, as the triangle-attention module uses them.  The same kernels
run on the same values, only the addresses differ, so every output must equal
the contiguous call's byte for byte, and nothing outside the views may be
written."""
import pytest
import torch

from protein_folding_triangle_gb300 import synthetic as S
from protein_folding_triangle_gb300 import triattn as T

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from protein_folding_triangle_gb300 import build
    build.build()
    T.load()


def heads_view(buf, col, H, D):
    """[B, N_o, H, N, D] view of H heads side by side at column `col` of the
    pair rows of buf [B, N_o, N, ld]."""
    return buf[..., col:col + H * D].unflatten(-1, (H, D)).permute(0, 1, 3, 2, 4)


CASES = [
    # (B, N, H, D, mask, ld_qkv, ld_o[, N_o]): ragged N, D = 16 and 32, extra columns on
    # both sides, an outer-axis shard of 37 of 48 slices (groups of 4 past N_o)
    (1, 136, 2, 32, "tail", 3 * 2 * 32 + 2 + 6, 2 * 32 + 8),
    (2, 40, 3, 16, "random", 3 * 3 * 16 + 3 + 5 + 16, 3 * 16),
    (1, 200, 4, 32, None, 3 * 4 * 32 + 4 + 4, 4 * 32),
    (1, 17, 1, 32, "random", 3 * 32 + 8 + 8, 32),
    (2, 48, 2, 32, "tail", 3 * 2 * 32 + 2 + 14, 2 * 32, 37),
]


@pytest.mark.parametrize("case", CASES, ids=[f"B{c[0]}N{c[1]}H{c[2]}D{c[3]}No{c[7] if len(c) > 7 else c[1]}"
                                             for c in CASES])
def test_strided_matches_contiguous_bitwise(case):
    B, N, H, D, mask_kind, ldq, ldo = case[:7]
    No = case[7] if len(case) > 7 else N
    g = torch.Generator().manual_seed(N + H + D)
    x = S.make_inputs(S.custom(B, N, H, D, mask=mask_kind or "none", mask_frac=0.1 if mask_kind else 0.0), seed=N)
    if No < N:  # an outer-axis shard: the first No slices
        for n in ("q", "k", "v", "do", "mask"):
            if x[n] is not None:
                x[n] = x[n][:, :No].contiguous()
    dev = torch.device("cuda")
    q, k, v, bias, do = (x[n].to(dev) for n in ("q", "k", "v", "bias", "do"))
    mask = x["mask"].to(dev) if x["mask"] is not None else None
    o, lse, res = T.tri_attn_fwd(q, k, v, bias, mask)
    dq, dk, dv, db = T.tri_attn_bwd(q, k, v, bias, mask, o, res, lse, do)

    # pair-row buffers filled with random junk; the heads copied in at offsets
    off = 8 if ldq % 8 == 0 and ldq >= 3 * H * D + 8 else 0
    P = torch.randn(B, No, N, ldq, generator=g).to(torch.bfloat16).to(dev)
    qs, ks, vs = (heads_view(P, off + t * H * D, H, D) for t in range(3))
    qs.copy_(q); ks.copy_(k); vs.copy_(v)
    P0 = P.clone()
    Ob = torch.randn(B, No, N, ldo, generator=g).to(torch.bfloat16).to(dev)
    Eb = torch.randn(B, No, N, ldo, generator=g).to(torch.bfloat16).to(dev)
    Gb = torch.randn(B, No, N, ldo, generator=g).to(torch.bfloat16).to(dev)
    os_, es, dos = heads_view(Ob, 0, H, D), heads_view(Eb, 0, H, D), heads_view(Gb, 0, H, D)
    dos.copy_(do)
    Ob0, Eb0 = Ob.clone(), Eb.clone()
    lse_s = torch.empty_like(lse)
    T.tri_attn_fwd_strided(qs, ks, vs, bias, mask, os_, lse_s, es)
    torch.cuda.synchronize()
    assert torch.equal(os_.contiguous().view(torch.int16), o.view(torch.int16))
    assert torch.equal(es.contiguous().view(torch.int16), res.view(torch.int16))
    assert torch.equal(lse_s.view(torch.int32), lse.view(torch.int32))
    assert torch.equal(P.view(torch.int16), P0.view(torch.int16))  # inputs untouched
    # nothing written outside the o / residual views
    for buf, ref in ((Ob, Ob0), (Eb, Eb0)):
        assert torch.equal(buf[..., H * D:].view(torch.int16), ref[..., H * D:].view(torch.int16))

    dP = torch.randn(B, No, N, ldq, generator=g).to(torch.bfloat16).to(dev)
    dP0 = dP.clone()
    dqs, dks, dvs = (heads_view(dP, off + t * H * D, H, D) for t in range(3))
    dbs = torch.empty_like(db)
    T.tri_attn_bwd_strided(qs, ks, vs, bias, mask, os_, es, lse_s, dos, dqs, dks, dvs, dbs)
    torch.cuda.synchronize()
    for got, ref in ((dqs, dq), (dks, dk), (dvs, dv)):
        assert torch.equal(got.contiguous().view(torch.int16), ref.view(torch.int16))
    assert torch.equal(dbs.view(torch.int16), db.view(torch.int16))
    # mixed layouts: q, k, v and dO contiguous, o and its residual in pair rows,
    # dq, dk, dv into pair rows (the module's backward)
    dP.copy_(dP0)
    dbs.zero_()
    T.tri_attn_bwd_strided(q, k, v, bias, mask, os_, es, lse_s, do, dqs, dks, dvs, dbs)
    torch.cuda.synchronize()
    for got, ref in ((dqs, dq), (dks, dk), (dvs, dv)):
        assert torch.equal(got.contiguous().view(torch.int16), ref.view(torch.int16))
    assert torch.equal(dbs.view(torch.int16), db.view(torch.int16))
    keep = torch.ones(ldq, dtype=torch.bool)
    keep[off:off + 3 * H * D] = False
    assert torch.equal(dP[..., keep].view(torch.int16), dP0[..., keep].view(torch.int16))
