"""The allocation-free backward entry point, tri_attn_bwd_noalloc.

Some callers cannot allocate device memory (a plugin whose host framework
owns all device memory, or a loop that cannot pay for cudaMalloc's implicit
synchronisation).  For them the library offers a backward that takes no
workspace and keeps its scratch in a fixed 64 MiB device array of its own.
This test calls it through the C ABI twice in a row and checks each result
against the regular workspace entry point.  Both run the same kernels on the
same inputs and the backward is deterministic, so the results must be equal
bit for bit; stale scratch contents left by the previous call would show.
It sits in a file of its own that pytest collects last, so a run that stops
at its first failure has run everything else.
"""
import ctypes

import pytest
import torch

from parity_utils import cpu64, rel_rmse, to_dev
from protein_folding_triangle_gb300 import synthetic as S
from protein_folding_triangle_gb300 import triattn as T

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from protein_folding_triangle_gb300 import build
    build.build()
    return T.load()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def call_noalloc(lib, x, o, resid, lse):
    dq, dk, dv = (torch.empty_like(x["q"]) for _ in range(3))
    db = torch.empty_like(x["bias"])
    s = T.shape_of(x["q"])
    code = lib.tri_attn_bwd_noalloc(ctypes.byref(s), _ptr(x["q"]), _ptr(x["k"]), _ptr(x["v"]), _ptr(x["bias"]),
                                    _ptr(x["mask"]), _ptr(o), _ptr(resid), _ptr(lse), _ptr(x["do"]), _ptr(dq),
                                    _ptr(dk), _ptr(dv), _ptr(db),
                                    ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return code, (dq, dk, dv, db)


@pytest.mark.parametrize("wname", ["tiny48", "masked136"])
def test_noalloc_matches_workspace_entry_point(lib, wname):
    w = S.WORKLOADS.get(wname) or S.custom(1, 136, 2, 32, name=wname, mask="random", mask_frac=0.1)
    assert T.bwd_workspace_bytes(T.Shape(w.B, w.No, w.N, w.H, w.D, 0)) <= T.NOALLOC_SCRATCH_BYTES
    x = to_dev(S.make_inputs(w, seed=7))
    o, lse, resid = T.tri_attn_fwd(x["q"], x["k"], x["v"], x["bias"], x["mask"])
    ref = T.tri_attn_bwd(x["q"], x["k"], x["v"], x["bias"], x["mask"], o, resid, lse, x["do"])
    torch.cuda.synchronize()
    for call in range(2):  # two calls in a row share the same scratch array
        code, got = call_noalloc(lib, x, o, resid, lse)
        assert code == T.OK, T.STATUS[code]
        torch.cuda.synchronize()
        assert T.device_status() == T.OK
        for name, g, r in zip(("dq", "dk", "dv", "dbias"), got, ref):
            assert torch.equal(g, r), (call, name, rel_rmse(cpu64(g), cpu64(r)))


def test_noalloc_rejects_shapes_beyond_its_scratch(lib):
    s = T.Shape(1, 384, 384, 4, 32, 0)  # needs about 438 MiB
    assert T.bwd_workspace_bytes(s) > T.NOALLOC_SCRATCH_BYTES
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the size check comes first
    code = lib.tri_attn_bwd_noalloc(ctypes.byref(s), fake, fake, fake, fake, None, fake, None, fake, fake, fake,
                                    fake, fake, fake, None)
    assert code == T.ERR_WORKSPACE
