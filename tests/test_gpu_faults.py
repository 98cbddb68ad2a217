"""Bounded device waits: a starved forward (its producer never loads the
first K tile) must end on its own with TRIATTN_ERR_TIMEOUT in the device
status word, and the context must stay usable afterwards.  Nothing here
faults, traps or hangs the GPU: every wait in the kernels is bounded by
%globaltimer and the limit is set to 20 ms for the starved call."""
import pytest
import torch

from parity_utils import TOL_O, compare_full, gpu_fwd_bwd, oracle_full, to_dev
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


def test_starved_forward_times_out_and_context_survives():
    w = S.custom(1, 64, 1, 32, name="starve")
    x = S.make_inputs(w, seed=1)
    xd = to_dev(x)
    assert T.device_status() == T.OK
    T.set_wait_limit_ns(20_000_000)
    T.test_set_starve(True)
    try:
        T.tri_attn_fwd(xd["q"], xd["k"], xd["v"], xd["bias"], xd["mask"])
        status = T.device_status()
    finally:
        T.test_set_starve(False)
        T.set_wait_limit_ns(0)
    assert status == T.ERR_TIMEOUT
    assert T.device_status() == T.OK          # the word was cleared
    out = gpu_fwd_bwd(xd)                      # the context still works
    errs = compare_full(out, oracle_full(x))
    assert errs["o"] <= TOL_O
