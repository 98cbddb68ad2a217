"""The library's tensor-core GEMM (tcgen05, TMA, TMEM accumulators) against
an FP64 matrix product of the same BF16 values, for every operand layout,
BF16 and FP32 outputs, ragged sizes, batches and the split-K path (whose
partials are added in fixed order: bitwise reproducible)."""
import pytest
import torch

from protein_folding_triangle_gb300 import triattn as T

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from protein_folding_triangle_gb300 import build
    build.build()
    T.load()


def operands(batch, M, N, K, ta, tb, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    a = torch.randn((batch, K, M) if ta else (batch, M, K), generator=g).to(torch.bfloat16)
    b = torch.randn((batch, N, K) if tb else (batch, K, N), generator=g).to(torch.bfloat16)
    return a.cuda(), b.cuda()


def reference(a, b, ta, tb):
    a64, b64 = a.double(), b.double()
    if ta:
        a64 = a64.transpose(-1, -2)
    if tb:
        b64 = b64.transpose(-1, -2)
    return a64 @ b64


def rel(x, r):
    return ((x.double() - r).pow(2).mean().sqrt() / r.pow(2).mean().sqrt()).item()


SHAPES = [
    (1, 128, 256, 64),    # one tile, one stage
    (1, 200, 296, 136),   # ragged M, N, K (row lengths multiples of 8)
    (3, 768, 768, 768),   # the contraction's shape, batched
    (2, 96, 128, 200),    # N = 128 tiles
    (1, 128, 640, 192),   # a projection: N = 640 (two 256 tiles and a ragged one)
]


@pytest.mark.parametrize("ta", [False, True], ids=["A_rows", "A_cols"])
@pytest.mark.parametrize("tb", [False, True], ids=["B_rows", "B_cols"])
@pytest.mark.parametrize("shape", SHAPES, ids=[f"b{s[0]}m{s[1]}n{s[2]}k{s[3]}" for s in SHAPES])
def test_gemm_layouts_and_shapes(shape, ta, tb):
    batch, M, N, K = shape
    a, b = operands(batch, M, N, K, ta, tb, seed=M + N + K + 2 * ta + tb)
    ref = reference(a, b, ta, tb)
    c32 = T.gemm(a, b, ta=ta, tb=tb, out_f32=True)
    c16 = T.gemm(a, b, ta=ta, tb=tb)
    torch.cuda.synchronize()
    assert T.device_status() == T.OK
    # FP32 output: only the FP32 accumulation order differs from FP64
    assert rel(c32, ref) < 1e-5, rel(c32, ref)
    # BF16 output: one rounding of each element (at most 2^-8 relative)
    assert rel(c16, ref) < 4e-3, rel(c16, ref)
    assert (c16.double() - ref).abs().le(ref.abs() * 2.0 ** -8 + 1e-4 * ref.abs().max()).all()


@pytest.mark.parametrize("ta,tb", [(True, False), (False, False)])
def test_gemm_split_k_is_deterministic(ta, tb):
    """A weight gradient's shape: a 128 x 640 output over K = 90000 pairs,
    too few output tiles to fill the GPU, so K is split into FP32 partials
    added in ascending order by a second kernel."""
    M, N, K = 128, 640, 90000
    assert T.load().triattn_gemm_workspace_bytes(M, N, K, 1) > 0
    a, b = operands(1, M, N, K, ta, tb, seed=5)
    ref = reference(a, b, ta, tb)
    c1 = T.gemm(a, b, ta=ta, tb=tb, out_f32=True)
    c2 = T.gemm(a, b, ta=ta, tb=tb, out_f32=True)
    torch.cuda.synchronize()
    assert torch.equal(c1, c2)
    assert rel(c1, ref) < 5e-5, rel(c1, ref)
