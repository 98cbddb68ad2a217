"""Non-deterministic ablation of the backward (FP32 atomics for dQ, dbias, or
both, or TMA bulk reductions for dQ, instead of the ordered single-writer
partials; "TurboPairFormer",
Table 12).  It must meet the same error bars against the FP64 oracle, and the
outputs that do not pass through atomics must be bitwise those of the ordered
backward."""
import pytest
import torch

from parity_utils import TOL_GRAD, TOL_O, compare_full, gpu_fwd_bwd, oracle_full, to_dev
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


@pytest.mark.parametrize("case", [(1, 136, 2, 32, "random"), (2, 200, 2, 16, "tail")],
                         ids=["N136D32", "B2N200D16"])
@pytest.mark.parametrize("atomic_mask", [T.ATOMIC_DQ, T.ATOMIC_DBIAS, T.ATOMIC_DBIAS_DQ, T.BULK_DQ,
                                         T.BULK_DQ_ATOMIC_DBIAS],
                         ids=["dq", "dbias", "dbias_dq", "bulk_dq", "bulk_dq_dbias"])
def test_atomic_ablation_parity(case, atomic_mask):
    B, N, H, D, mk = case
    w = S.custom(B, N, H, D, name="atom", mask=mk, mask_frac=0.1)
    x = S.make_inputs(w, seed=N + atomic_mask)
    xd = to_dev(x)
    ordered = gpu_fwd_bwd(xd)
    dq, dk, dv, db = T.tri_attn_bwd_atomic_ablation(xd["q"], xd["k"], xd["v"], xd["bias"], xd["mask"], ordered["o"],
                                                    ordered["resid"], ordered["lse"], xd["do"], atomic_mask)
    torch.cuda.synchronize()
    assert T.device_status() == T.OK
    assert torch.equal(dk, ordered["dk"]) and torch.equal(dv, ordered["dv"])
    if atomic_mask == T.ATOMIC_DBIAS:
        assert torch.equal(dq, ordered["dq"])
    if atomic_mask in (T.ATOMIC_DQ, T.BULK_DQ):
        assert torch.equal(db, ordered["dbias"])
    out = dict(ordered)
    out.update(dq=dq, dk=dk, dv=dv, dbias=db)
    errs = compare_full(out, oracle_full(x))
    assert errs["o"] <= TOL_O, errs
    for g in ("dq", "dk", "dv", "dbias"):
        assert errs[g] <= TOL_GRAD, (g, errs)
