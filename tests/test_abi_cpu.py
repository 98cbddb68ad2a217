"""CPU-only checks of the C ABI boundary: the library loads, exports every
function include/triattn.h declares, and rejects bad arguments before it
touches a GPU.  Also the multi-rank timing combination of bench.py over two
gloo ranks."""
import ctypes
import os
import re

import pytest
import torch

from protein_folding_triangle_gb300 import build as B
from protein_folding_triangle_gb300 import triattn as T

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return T.load()


def header_functions():
    text = open(os.path.join(ROOT, "include", "triattn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b([a-z_][a-z0-9_]*)\s*\(", text)
    return sorted(set(n for n in names if n.startswith(("tri_attn", "triattn"))))


def test_exports_every_declared_function(lib):
    declared = header_functions()
    assert "tri_attn_fwd" in declared and "tri_attn_bwd" in declared
    for name in declared:
        assert hasattr(lib, name), name
    assert set(T.EXPORTED) >= set(declared)


def test_status_strings(lib):
    for code, name in T.STATUS.items():
        assert lib.triattn_status_string(code).decode() == name


FAKE = 1 << 20  # aligned, never dereferenced: validation fails first


def call_fwd(lib, shape, **ptrs):
    p = {n: ctypes.c_void_p(FAKE) for n in ("q", "k", "v", "bias", "o", "lse")}
    p.update({"mask": None, "o_resid": None})
    p.update(ptrs)
    return lib.tri_attn_fwd(ctypes.byref(shape), p["q"], p["k"], p["v"], p["bias"], p["mask"], p["o"], p["lse"],
                            p["o_resid"], None, ctypes.c_size_t(0), None)


def call_bwd(lib, shape, ws_bytes, ws=FAKE, **ptrs):
    names = ("q", "k", "v", "bias", "o", "lse", "dO", "dq", "dk", "dv", "dbias")
    p = {n: ctypes.c_void_p(FAKE) for n in names}
    p.update({"mask": None, "o_resid": None})
    p.update(ptrs)
    return lib.tri_attn_bwd(ctypes.byref(shape), p["q"], p["k"], p["v"], p["bias"], p["mask"], p["o"],
                            p["o_resid"], p["lse"], p["dO"], p["dq"], p["dk"], p["dv"], p["dbias"],
                            None if ws is None else ctypes.c_void_p(ws), ctypes.c_size_t(ws_bytes), None)


@pytest.mark.parametrize("shape,code", [
    ((1, 48, 48, 2, 24, 0), T.ERR_UNSUPPORTED),   # D not in {16, 32}
    ((1, 56, 48, 2, 16, 0), T.ERR_UNSUPPORTED),   # more outer slices than N
    ((1, 262145, 262145, 1, 16, 0), T.ERR_UNSUPPORTED),  # more than 65535 outer groups of 4
    ((1, 46341, 46341, 1, 16, 0), T.ERR_UNSUPPORTED),    # N * ceil(N / 128) * 128 beyond 2^31
    ((256, 48, 48, 256, 16, 0), T.ERR_UNSUPPORTED),      # B * H beyond the grid
    ((0, 48, 48, 2, 16, 0), T.ERR_INVALID_ARG),   # empty batch
    ((1, 0, 0, 2, 16, 0), T.ERR_INVALID_ARG),     # empty crop
    ((1, 48, 48, 0, 16, 0), T.ERR_INVALID_ARG),   # no heads
    ((1, 48, 48, 2, 16, 2), T.ERR_INVALID_ARG),   # unknown flag bit
])
def test_bad_shapes(lib, shape, code):
    s = T.Shape(*shape)
    assert call_fwd(lib, s) == code
    assert call_bwd(lib, s, 1 << 40) == code
    assert lib.triattn_bwd_workspace_bytes(ctypes.byref(s)) == 0
    assert lib.triattn_fwd_workspace_bytes(ctypes.byref(s)) == 0


@pytest.mark.parametrize("shape", [(1, 1, 1, 1, 16), (1, 17, 17, 2, 32), (2, 130, 130, 4, 16), (1, 1000, 1000, 1, 32),
                                   (1, 44, 48, 2, 16), (1, 5000, 5000, 1, 16), (3, 3, 64, 2, 32)])
def test_any_n_accepted_with_workspace_sizes(lib, shape):
    """Any N >= 1 and any shard 1 <= N_o <= N are accepted ("TurboPairFormer",
    Table 1 places no divisibility rule on N).  The forward's workspace holds
    one 144-byte key-mask record per (slice, 64-key tile) with four padding
    slices, then (N not a multiple of 8) the bias with rows padded to a
    multiple of 8 elements; the backward's transposed bias uses that row
    stride, and its dbias partials cover ceil(N_o / G) outer groups."""
    B, No, N, H, D = shape
    s = T.Shape(B, No, N, H, D, 0)
    r256 = lambda x: (x + 255) // 256 * 256
    jk64, jq, jk = -(-N // 64), -(-N // 128), -(-N // 128)
    Np = -(-N // 8) * 8
    rec = r256((B * No + 4) * jk64 * 144)
    pad = r256(B * H * N * Np * 2) if N % 8 else 0
    assert lib.triattn_fwd_workspace_bytes(ctypes.byref(s)) == rec + pad
    slices = B * No * H
    G = 4 if D == 32 else 8
    want = (r256(slices * jq * 128 * 16) + r256(B * H * N * Np * 2) + r256(jk * slices * jq * 128 * D * 4)
            + r256(-(-No // G) * B * H * jq * jk * 128 * 128 * 4))
    assert lib.triattn_bwd_workspace_bytes(ctypes.byref(s)) == want


def test_forward_workspace_checks(lib):
    """With a mask, or N not a multiple of 64, the forward needs its
    workspace: a missing or short one is TRIATTN_ERR_WORKSPACE before any
    launch; without a mask and N a multiple of 64 none is needed."""
    s = T.Shape(1, 40, 40, 2, 16, 0)
    need = lib.triattn_fwd_workspace_bytes(ctypes.byref(s))
    assert need > 0
    assert call_fwd(lib, s) == T.ERR_WORKSPACE
    p = {n: ctypes.c_void_p(FAKE) for n in ("q", "k", "v", "bias", "o", "lse")}
    short = lib.tri_attn_fwd(ctypes.byref(s), p["q"], p["k"], p["v"], p["bias"], None, p["o"], p["lse"], None,
                             ctypes.c_void_p(FAKE), ctypes.c_size_t(need - 256), None)
    assert short == T.ERR_WORKSPACE
    misaligned = lib.tri_attn_fwd(ctypes.byref(s), p["q"], p["k"], p["v"], p["bias"], None, p["o"], p["lse"], None,
                                  ctypes.c_void_p(FAKE + 16), ctypes.c_size_t(need), None)
    assert misaligned == T.ERR_WORKSPACE


def test_null_and_misaligned_pointers(lib):
    s = T.Shape(1, 48, 48, 2, 16, 0)
    assert call_fwd(lib, s, q=None) == T.ERR_INVALID_ARG
    assert call_fwd(lib, s, lse=None) == T.ERR_INVALID_ARG
    assert call_fwd(lib, s, k=ctypes.c_void_p(FAKE + 2)) == T.ERR_INVALID_ARG
    assert call_fwd(lib, s, mask=ctypes.c_void_p(FAKE + 1)) == T.ERR_INVALID_ARG
    assert call_fwd(lib, s, lse=ctypes.c_void_p(FAKE + 2)) == T.ERR_INVALID_ARG
    assert call_bwd(lib, s, 1 << 40, lse=ctypes.c_void_p(FAKE + 6)) == T.ERR_INVALID_ARG
    assert call_bwd(lib, s, 1 << 40, mask=ctypes.c_void_p(FAKE + 3)) == T.ERR_INVALID_ARG
    assert call_bwd(lib, s, 1 << 40, dbias=None) == T.ERR_INVALID_ARG
    assert call_bwd(lib, s, 1 << 40, o_resid=ctypes.c_void_p(FAKE + 4)) == T.ERR_INVALID_ARG


def test_workspace_checks(lib):
    s = T.Shape(1, 48, 48, 2, 16, 0)
    need = lib.triattn_bwd_workspace_bytes(ctypes.byref(s))
    # layout: query-row records [slices][J_Q * 128][8] BF16 + transposed bias [B*H][N][N]
    # BF16 + dQ partials [J_K][slices][J_Q][128 x D] FP32 + dbias partials
    # [N_o/G][B*H][J_Q][J_K][128 x 128] FP32 (G = 8 outer slices per CTA at D = 16),
    # each 256-aligned (padded to whole tiles)
    slices = 1 * 48 * 2
    r256 = lambda x: (x + 255) // 256 * 256
    assert need == (r256(slices * 1 * 128 * 16) + r256(1 * 2 * 48 * 48 * 2) + r256(1 * slices * 1 * 128 * 16 * 4)
                    + r256(6 * 1 * 2 * 1 * 1 * 128 * 128 * 4))
    assert call_bwd(lib, s, need - 1) == T.ERR_WORKSPACE
    assert call_bwd(lib, s, need, ws=None) == T.ERR_WORKSPACE
    assert call_bwd(lib, s, need, ws=FAKE + 16) == T.ERR_WORKSPACE


def test_trace_read_empty(lib):
    T.trace_enable(True)
    T.trace_enable(False)
    assert T.trace_read() == {}


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms, value = bench.combine_ranks(10.0 * (rank + 1), flop_per_step=10 ** 12, steps=4, world=world)
    out.put((rank, ms, value))
    dist.destroy_process_group()


def test_combine_ranks_two_gloo_ranks():
    import socket
    import torch.multiprocessing as mp
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, value in res:
        assert ms == 20.0                      # the slowest rank's time
        assert abs(value - 2 * 4 / 0.020) < 1e-9  # 2 ranks x 4 steps x 1 TFLOP over 20 ms, in TFLOP/s


def test_atomic_ablation_workspace_and_mask_checks(lib):
    """The non-deterministic ablation entry point: its workspace holds FP32
    accumulators instead of the partials of the operands it adds atomically,
    and any mask other than 1 (atomic dQ), 2 (atomic dbias), 3 (both), 4
    (bulk-reduced dQ) or 6 (bulk dQ, atomic dbias) is rejected before
    anything is launched."""
    s = T.Shape(1, 136, 136, 2, 32, 0)
    r256 = lambda x: (x + 255) // 256 * 256
    slices, jq, jk = 136 * 2, 2, 2
    base = r256(slices * jq * 128 * 16) + r256(2 * 136 * 136 * 2)
    dq_part = jk * slices * jq * 128 * 32 * 4
    dq_acc = slices * jq * 128 * 32 * 4
    db_part = (136 // 4) * 2 * jq * jk * 128 * 128 * 4
    db_acc = 2 * jk * 128 * jq * 128 * 4
    assert lib.triattn_bwd_atomic_workspace_bytes(ctypes.byref(s), 1) == base + r256(dq_acc) + r256(db_part)
    assert lib.triattn_bwd_atomic_workspace_bytes(ctypes.byref(s), 2) == base + r256(dq_part) + r256(db_acc)
    assert lib.triattn_bwd_atomic_workspace_bytes(ctypes.byref(s), 3) == base + r256(dq_acc) + r256(db_acc)
    assert lib.triattn_bwd_workspace_bytes(ctypes.byref(s)) == base + r256(dq_part) + r256(db_part)
    assert lib.triattn_bwd_atomic_workspace_bytes(ctypes.byref(s), 4) == base + r256(dq_acc) + r256(db_part)
    assert lib.triattn_bwd_atomic_workspace_bytes(ctypes.byref(s), 6) == base + r256(dq_acc) + r256(db_acc)
    for bad in (0, 5, 7, 8, -1):
        assert lib.triattn_bwd_atomic_workspace_bytes(ctypes.byref(s), bad) == 0
        fake = ctypes.c_void_p(1 << 40)
        args = [ctypes.byref(s)] + [fake] * 13 + [bad, fake, ctypes.c_size_t(1 << 40), None]
        assert lib.tri_attn_bwd_atomic_ablation(*args) == T.ERR_INVALID_ARG


def test_outer_shard_ranges():
    from protein_folding_triangle_gb300.sharding import outer_shard
    for n, world in ((768, 1), (768, 2), (768, 3), (768, 8), (200, 3), (48, 6), (8, 1), (771, 4), (17, 2),
                     (16, 3), (5, 5)):
        ranges = [outer_shard(n, r, world) for r in range(world)]
        assert ranges[0][0] == 0 and ranges[-1][1] == n
        for (lo, hi), (lo2, _) in zip(ranges, ranges[1:]):
            assert hi == lo2
        sizes = [hi - lo for lo, hi in ranges]
        assert all(sz >= 1 for sz in sizes)
        if n // 8 >= world:  # whole blocks of 8, the remainder on the last rank
            assert all(lo % 8 == 0 for lo, _ in ranges)
            assert max(sizes[:-1] + [sizes[-1] - n % 8]) - min(sizes[:-1] + [sizes[-1] - n % 8]) <= 8
        else:
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        outer_shard(2, 0, 3)


def test_shard_shapes_accepted(lib):
    """A shard of the outer axis (N_o < N, a multiple of 8) is a valid shape;
    its workspace counts only its own slices and groups."""
    full = T.Shape(1, 48, 48, 2, 32, 0)
    half = T.Shape(1, 24, 48, 2, 32, T.FLAG_DBIAS_FP32)
    wf = lib.triattn_bwd_workspace_bytes(ctypes.byref(full))
    wh = lib.triattn_bwd_workspace_bytes(ctypes.byref(half))
    assert 0 < wh < wf


def _combine_worker(rank, world, port, n_outer, q):
    """One rank of a 2-rank gloo group: the FP64 oracle's dbias of its shard,
    kept in FP32, gathered in rank order, then summed in rank order."""
    import numpy as np
    import torch.distributed as dist
    from oracle import oracle as O
    from protein_folding_triangle_gb300 import synthetic as S
    from protein_folding_triangle_gb300.sharding import gather_rank_ordered, outer_shard
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = S.custom(1, n_outer, 2, 16, name="shard", mask="random", mask_frac=0.1)
        x = S.make_inputs(w, seed=5)
        lo, hi = outer_shard(n_outer, rank, world)
        sh = {k: (None if v is None else (v if k == "bias" else v[:, lo:hi].contiguous())) for k, v in x.items()}
        _, _, _, db = O.bwd(sh["q"], sh["k"], sh["v"], sh["bias"], sh["mask"], sh["do"])
        parts = gather_rank_ordered(torch.from_numpy(db.astype(np.float32)))
        total = parts[0].clone()
        for r in range(1, world):
            total += parts[r]
        if rank == 0:
            _, _, _, ref = O.bwd(x["q"], x["k"], x["v"], x["bias"], x["mask"], x["do"])
            err = float(np.sqrt(np.mean((total.double().numpy() - ref) ** 2)) / np.sqrt(np.mean(ref ** 2)))
            q.put(("ok", err, [tuple(p.shape) for p in parts]))
    except Exception as e:  # noqa: BLE001
        q.put(("error", repr(e), None))
        raise
    finally:
        dist.destroy_process_group()


def test_sharded_dbias_gather_two_gloo_ranks():
    """The host side of the outer-axis split: two gloo ranks each own half of
    the slices; their FP32 dbias parts, gathered in rank order and added,
    give the full dbias (FP64 oracle on each shard vs on the whole axis)."""
    import multiprocessing as mp
    import socket
    ctx = mp.get_context("spawn")
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    q = ctx.Queue()
    procs = [ctx.Process(target=_combine_worker, args=(r, 2, port, 24, q)) for r in range(2)]
    for p in procs:
        p.start()
    status, err, shapes = q.get(timeout=240)
    for p in procs:
        p.join(timeout=60)
    assert status == "ok", err
    assert shapes == [(1, 2, 24, 24)] * 2
    assert err < 1e-6, err


def module_shape(B=1, N=40, C=64, H=2, D=16, flags=0):
    return T.ModuleShape(B, N, C, H, D, flags)


def call_module_fwd(lib, shape, ws_bytes, ws=FAKE, **ptrs):
    names = ("z", "ln_w", "ln_b", "w_in", "w_o", "out", "ctx")
    p = {n: ctypes.c_void_p(FAKE) for n in names}
    p["mask"] = None
    p.update(ptrs)
    return lib.tri_attn_module_fwd(ctypes.byref(shape), p["z"], p["mask"], p["ln_w"], p["ln_b"], p["w_in"],
                                   p["w_o"], p["out"], p["ctx"], ctypes.c_void_p(ws), ctypes.c_size_t(ws_bytes),
                                   None)


def call_module_bwd(lib, shape, ws_bytes, ws=FAKE, **ptrs):
    names = ("z", "ln_w", "w_in", "w_o", "ctx", "d_out", "dz", "d_ln_w", "d_ln_b", "d_w_in", "d_w_o")
    p = {n: ctypes.c_void_p(FAKE) for n in names}
    p["mask"] = None
    p.update(ptrs)
    return lib.tri_attn_module_bwd(ctypes.byref(shape), p["z"], p["mask"], p["ln_w"], p["w_in"], p["w_o"],
                                   p["ctx"], p["d_out"], p["dz"], p["d_ln_w"], p["d_ln_b"], p["d_w_in"],
                                   p["d_w_o"], ctypes.c_void_p(ws), ctypes.c_size_t(ws_bytes), None)


def test_module_sizes(lib):
    ctx, ws = T.module_sizes(1, 40, 64, 2, 16)
    B_, N, C, H, D = 1, 40, 64, 2, 16
    M, Fp = B_ * N * N, (3 * H * D + H + 7) // 8 * 8
    # ctx holds at least x, P (q, k, v are read where they lie in it), the
    # residual, o_flat (the core writes o there) and the bias planes
    assert ctx >= M * C * 2 + M * Fp * 2 + 2 * M * H * D * 2 + B_ * H * N * N * 2
    core = T.bwd_workspace_bytes(T.Shape(B_, N, N, H, D, 0))
    assert ws >= core + (32 << 20) + B_ * N * N * (3 * H * D + H) * 2
    for bad in [(1, 40, 48, 2, 16), (1, 40, 288, 2, 16), (1, 44, 64, 2, 16), (1, 40, 64, 2, 8), (0, 40, 64, 2, 16),
                (1, 40, 64, 65, 16), (128, 4096, 64, 2, 16)]:
        assert T.module_sizes(*bad) == (0, 0), bad


def test_module_rejects_bad_arguments(lib):
    s = module_shape()
    _, ws = T.module_sizes(1, 40, 64, 2, 16)
    assert call_module_fwd(lib, module_shape(C=48), ws) == T.ERR_UNSUPPORTED
    assert call_module_fwd(lib, module_shape(flags=1), ws) == T.ERR_INVALID_ARG
    assert call_module_fwd(lib, module_shape(B=0), ws) == T.ERR_INVALID_ARG
    assert call_module_fwd(lib, s, ws, z=None) == T.ERR_INVALID_ARG
    assert call_module_fwd(lib, s, ws, w_in=ctypes.c_void_p(FAKE + 8)) == T.ERR_INVALID_ARG
    assert call_module_fwd(lib, s, ws, ctx=ctypes.c_void_p(FAKE + 16)) == T.ERR_INVALID_ARG
    assert call_module_fwd(lib, s, ws - 1) == T.ERR_WORKSPACE
    assert call_module_fwd(lib, s, ws, ws=FAKE + 16) == T.ERR_WORKSPACE
    assert call_module_bwd(lib, module_shape(D=24), ws) == T.ERR_UNSUPPORTED
    assert call_module_bwd(lib, s, ws, d_w_o=None) == T.ERR_INVALID_ARG
    assert call_module_bwd(lib, s, ws, mask=ctypes.c_void_p(FAKE + 2)) == T.ERR_INVALID_ARG
    assert call_module_bwd(lib, s, 0) == T.ERR_WORKSPACE


def test_trimul_and_module_workspace_layouts(lib):
    """The scratch layouts, each part 256-byte aligned: the GEMMs' 32 MiB of
    split-K partials, then (TriMul) du, dp, dy, the channel-major dX, dA, dB,
    dx and the LayerNorm partial rows; (module) W_in padded to Fp columns, its
    FP32 gradient, dP, d_oflat, dbias, dx, the LayerNorm partial rows and the
    core's workspace.  The activation gradients dy and dx are BF16 (2 bytes
    per element); the LayerNorm backwards write one partial row per block of
    their fixed grids (456 pair-major, 304 channel-major)."""
    r256 = lambda x: (x + 255) // 256 * 256
    B, N, Cz, Ch = 1, 40, 64, 32
    M, NN = B * N * N, N * N
    Fp = (4 * Ch + Cz + 7) // 8 * 8
    want = (r256(32 << 20) + r256(M * Cz * 2) + r256(M * Fp * 2) + r256(M * Ch * 2) + 3 * r256(B * Ch * NN * 2)
            + r256(M * Cz * 2) + 2 * r256(456 * Cz * 4) + 2 * r256(304 * Ch * 4))
    assert T.trimul_sizes(B, N, Cz, Ch)[1] == want
    B, N, C, H, D = 1, 40, 64, 2, 16
    M, HD = B * N * N, H * D
    Fp = (3 * HD + H + 7) // 8 * 8
    core = max(T.bwd_workspace_bytes(T.Shape(B, N, N, H, D, 0)), lib.triattn_fwd_workspace_bytes(
        ctypes.byref(T.Shape(B, N, N, H, D, 0))))
    want = (r256(32 << 20) + r256(C * Fp * 2) + r256(C * Fp * 4) + r256(M * Fp * 2) + r256(M * HD * 2)
            + r256(B * H * N * N * 2) + r256(M * C * 2) + 2 * r256(456 * C * 4) + r256(core))
    assert T.module_sizes(B, N, C, H, D)[1] == want


def test_trimul_sizes_and_argument_checks(lib):
    ctx, ws = T.trimul_sizes(1, 40, 64, 32)
    M, Cz, Ch = 40 * 40, 64, 32
    # ctx holds at least x, g, a, b, X, y and u; the projection p is never stored
    assert ctx >= M * Cz * 2 + M * Cz * 2 + 3 * M * Ch * 2 + M * Ch * 2 + M * Cz * 2
    assert ctx < M * Cz * 2 + M * (4 * Ch + Cz) * 2 + 3 * M * Ch * 2 + M * Ch * 2 + M * Cz * 2
    assert ws >= (32 << 20) + M * (4 * Ch + Cz) * 2
    assert T.trimul_sizes(1, 40, 64, 32, "incoming") == (ctx, ws)
    for bad in [(1, 44, 64, 32), (1, 40, 48, 32), (1, 40, 64, 160), (1, 40, 64, 48), (0, 40, 64, 32)]:
        assert T.trimul_sizes(*bad) == (0, 0), bad
    with pytest.raises(ValueError):
        T.trimul_shape(1, 40, 64, 32, "sideways")
    f = ctypes.c_void_p(FAKE)

    def fwd(shape, nbytes, **kw):
        p = {n: f for n in ("z", "liw", "lib", "wp", "low", "lob", "wo", "out", "ctx")}
        p["mask"] = None
        p.update(kw)
        return lib.triattn_trimul_fwd(ctypes.byref(shape), p["z"], p["mask"], p["liw"], p["lib"], p["wp"], p["low"],
                                      p["lob"], p["wo"], p["out"], p["ctx"], f, ctypes.c_size_t(nbytes), None)

    def bwd(shape, nbytes, **kw):
        names = ("z", "liw", "wp", "low", "wo", "ctx", "dout", "dz", "dliw", "dlib", "dwp", "dlow", "dlob", "dwo")
        p = {n: f for n in names}
        p["mask"] = None
        p.update(kw)
        return lib.triattn_trimul_bwd(ctypes.byref(shape), p["z"], p["mask"], p["liw"], p["wp"], p["low"], p["wo"],
                                      p["ctx"], p["dout"], p["dz"], p["dliw"], p["dlib"], p["dwp"], p["dlow"],
                                      p["dlob"], p["dwo"], f, ctypes.c_size_t(nbytes), None)

    s = T.TriMulShape(1, 40, 64, 32, 0, 0)
    assert fwd(T.TriMulShape(1, 40, 64, 32, 2, 0), ws) == T.ERR_INVALID_ARG
    assert fwd(T.TriMulShape(1, 40, 64, 32, 0, 1), ws) == T.ERR_INVALID_ARG
    assert fwd(T.TriMulShape(1, 40, 64, 40, 0, 0), ws) == T.ERR_UNSUPPORTED
    assert fwd(s, ws, z=None) == T.ERR_INVALID_ARG
    assert fwd(s, ws, wp=ctypes.c_void_p(FAKE + 4)) == T.ERR_INVALID_ARG
    assert fwd(s, ws, ctx=ctypes.c_void_p(FAKE + 32)) == T.ERR_INVALID_ARG
    assert fwd(s, ws - 1) == T.ERR_WORKSPACE
    assert bwd(s, ws, dwo=None) == T.ERR_INVALID_ARG
    assert bwd(s, ws, mask=ctypes.c_void_p(FAKE + 6)) == T.ERR_INVALID_ARG
    assert bwd(T.TriMulShape(1, 40, 288, 32, 1, 0), ws) == T.ERR_UNSUPPORTED
    assert bwd(s, 100) == T.ERR_WORKSPACE


def test_chunk_slices_picks_the_largest_fitting_multiple():
    from protein_folding_triangle_gb300 import sharding as SH
    per = lambda c: 1000 + 10 * c  # noqa: E731  (grows with the chunk)
    assert SH.chunk_slices(64, per, 1000 + 10 * 24) == 24
    assert SH.chunk_slices(64, per, 1000 + 10 * 31) == 24
    assert SH.chunk_slices(64, per, 10 ** 9) == 64
    with pytest.raises(ValueError):
        SH.chunk_slices(64, per, 1000)          # not even 8 slices fit
    assert SH.chunk_slices(60, per, 10 ** 9) == 60   # the whole axis, not a multiple of 8
    assert SH.chunk_slices(60, per, 1000 + 10 * 59) == 56
    assert SH.chunk_slices(5, per, 10 ** 9) == 5


def test_chunked_backward_workspace_is_bounded(lib):
    """The per-chunk workspace of the chunked backward grows with the chunk,
    so capping it bounds the backward's memory; the one-call workspace of a
    4096-token crop (H = 4, D = 32) is far above any GPU's memory."""
    from protein_folding_triangle_gb300 import sharding as SH
    N, H, D = 4096, 4, 32
    one_call = T.bwd_workspace_bytes(T.Shape(1, N, N, H, D, 0))
    assert one_call > 400 * 2 ** 30
    per = lambda c: T.bwd_workspace_bytes(T.Shape(1, c, N, H, D, T.FLAG_DBIAS_FP32))  # noqa: E731
    c = SH.chunk_slices(N, per, 16 * 2 ** 30)
    assert 8 <= c < N and per(c) <= 16 * 2 ** 30 < per(c + 8)


def test_gemm_argument_checks(lib):
    """The tensor-core GEMM rejects bad sizes, strides and null pointers before
    touching the device; its split-K workspace is 0 for an invalid shape."""
    fake = ctypes.c_void_p(1 << 20)
    def call(ta=0, tb=0, M=128, N=128, K=64, lda=64, ldb=128, ldc=128, A=fake, B=fake, C=fake):
        return lib.triattn_gemm(ta, tb, M, N, K, A, lda, B, ldb, C, ldc, 0, 1, 0, 0, 0, None, 0, None)
    assert call(M=0) == T.ERR_INVALID_ARG
    assert call(K=-1) == T.ERR_INVALID_ARG
    assert call(lda=32) == T.ERR_INVALID_ARG          # lda < K
    assert call(ta=1, lda=64) == T.ERR_INVALID_ARG    # A is [K, M]: lda < M
    assert call(ldb=64) == T.ERR_INVALID_ARG          # ldb < N
    assert call(ldc=64) == T.ERR_INVALID_ARG          # ldc < N
    assert call(A=None) == T.ERR_INVALID_ARG
    assert lib.triattn_gemm_workspace_bytes(0, 1, 1, 1) == 0


def test_strided_layout_checks(lib):
    """tri_attn_fwd_strided / tri_attn_bwd_strided reject layouts the kernels
    cannot address (strides not multiples of 8 elements, overlapping rows,
    heads or slices) before any GPU work; the layouts of a contiguous tensor
    and of heads in pair rows pass validation (the call then fails on the
    missing workspace of this ragged shape)."""
    s = T.Shape(1, 40, 40, 2, 32, 0)
    f = ctypes.c_void_p(FAKE)

    def fwd(lq, lo, ws=None, nbytes=0):
        return lib.tri_attn_fwd_strided(ctypes.byref(s), f, f, f, lq, f, f, f, f, None, lo, ws,
                                        ctypes.c_size_t(nbytes), None)

    def bwd(lq, lo):
        return lib.tri_attn_bwd_strided(ctypes.byref(s), f, f, f, lq, f, None, f, None, lo, f, f, lo, f, f, f, lq, f,
                                        None, ctypes.c_size_t(0), None)

    good = T.Layout(2 * 40 * 32, 40 * 32, 32)       # [B, N_o, H, N, D]
    pair = T.Layout(40 * 200, 32, 200)              # heads side by side in pair rows of 200
    bad = [T.Layout(2 * 40 * 32, 40 * 32, 36),      # row not a multiple of 8
           T.Layout(2 * 40 * 32, 40 * 32, 24),      # rows overlap (row < D)
           T.Layout(2 * 40 * 32, 16, 200),          # heads overlap (head < D)
           T.Layout(40 * 200, 200, 200),            # head == row
           T.Layout(1000, 32, 200),                 # slices overlap (40 rows of 200 > 1000)
           T.Layout(40 * 200, 32, 56),              # the two heads of a row overlap (32 + 32 > 56)
           T.Layout(2 * 40 * 32, 40 * 32 - 8, 32),  # the rows of a head run into the next head
           T.Layout(0, 32, 200),
           T.Layout(1 << 36, 32, 200)]              # beyond the index range
    for lay in bad:
        assert fwd(ctypes.byref(lay), ctypes.byref(good)) == T.ERR_INVALID_ARG
        assert fwd(ctypes.byref(good), ctypes.byref(lay)) == T.ERR_INVALID_ARG
        assert bwd(ctypes.byref(lay), ctypes.byref(good)) == T.ERR_INVALID_ARG
        assert bwd(ctypes.byref(good), ctypes.byref(lay)) == T.ERR_INVALID_ARG
    # a null layout is an argument error on the strided entry points
    assert fwd(None, ctypes.byref(good)) == T.ERR_INVALID_ARG
    assert bwd(ctypes.byref(pair), None) == T.ERR_INVALID_ARG
    # one head: its head stride may equal the row stride
    s1 = T.Shape(1, 40, 40, 1, 32, 0)
    one = T.Layout(40 * 32, 32, 32)
    assert lib.tri_attn_fwd_strided(ctypes.byref(s1), f, f, f, ctypes.byref(one), f, f, f, f, None,
                                    ctypes.byref(one), None, ctypes.c_size_t(0), None) == T.ERR_WORKSPACE
    # valid layouts get as far as the workspace check (N = 40 needs the padded bias copy)
    assert fwd(ctypes.byref(pair), ctypes.byref(good)) == T.ERR_WORKSPACE
    assert bwd(ctypes.byref(pair), ctypes.byref(pair)) == T.ERR_WORKSPACE


def test_layout_of_views():
    """layout_of reads the row layout off a [B, N_o, H, N, D] view."""
    B, N, H, D, ld = 2, 24, 3, 16, 200
    P = torch.zeros(B, N, N, ld, dtype=torch.bfloat16)
    q = P[..., 8:8 + H * D].unflatten(-1, (H, D)).permute(0, 1, 3, 2, 4)
    lay = T.layout_of(q)
    assert (lay.slice, lay.head, lay.row) == (N * ld, D, ld)
    c = torch.zeros(B, N, H, N, D, dtype=torch.bfloat16)
    lay = T.layout_of(c)
    assert (lay.slice, lay.head, lay.row) == (H * N * D, N * D, D)
    with pytest.raises(ValueError):
        T.layout_of(c.transpose(3, 4))


def test_layers_parameters_and_no_cpu_path():
    """The torch modules hold the library's parameter layouts (W_in [C, 3HD + H]
    and W_o [HD, C] for triangle attention; W_p [C_z, 4C_h + C_z] and W_o [C_h,
    C_z] for the multiplicative update; BF16 weights, FP32 LayerNorm
    parameters), reject an unknown direction, and refuse CPU tensors instead of
    computing anything on the host."""
    from protein_folding_triangle_gb300 import layers
    att = layers.TriangleAttention(c_z=64, n_heads=2, head_dim=16)
    assert tuple(att.w_in.shape) == (64, 3 * 2 * 16 + 2) and att.w_in.dtype == torch.bfloat16
    assert tuple(att.w_o.shape) == (2 * 16, 64) and att.w_o.dtype == torch.bfloat16
    assert att.ln_w.dtype == torch.float32 and tuple(att.ln_b.shape) == (64,)
    mul = layers.TriangleMultiplication(c_z=64, c_hidden=32, direction="incoming")
    assert tuple(mul.w_p.shape) == (64, 4 * 32 + 64) and tuple(mul.w_o.shape) == (32, 64)
    assert tuple(mul.ln_out_w.shape) == (32,) and mul.ln_in_w.dtype == torch.float32
    with pytest.raises(ValueError):
        layers.TriangleMultiplication(c_z=64, c_hidden=32, direction="sideways")
    z = torch.zeros(1, 8, 8, 64, dtype=torch.bfloat16)
    for module in (att, mul):
        with pytest.raises((ValueError, RuntimeError)):
            module(z)
