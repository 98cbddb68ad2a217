// Kernel argument blocks and launch entry points shared by the C ABI layer.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>
#include <functional>

#include "ptx.cuh"

namespace triattn {

// Backward tile: 128 query rows x 128 keys (the forward steps over 64-key
// tiles of 128 query rows, see fwd.cu).
constexpr int kTileQ = 128;
constexpr int kTileK = 128;
// Outer slices per CTA: forward (shared bias tile) and backward (outer group
// of the key-tile-parallel backward).
constexpr int kGroupFwd = 4;
// Backward: dK and dV of all slices of the group stay in TMEM (2 * G * D of
// its 512 columns next to 256 for S^T and dP^T), so G = 8 at D = 16.
constexpr int kGroupBwdFor(int D) { return D == 16 ? 8 : 4; }

// Where the rows of a [B, N_o, H, N, D] tensor (D features contiguous) lie:
// row (b, o, h, n) starts slice * (b N_o + o) + head * h + row * n elements
// from the base.  The library's own layout is {H N D, N D, D}; the
// triangle-attention module's pair rows are {N ld, D, ld}.  Q, K, V (and dO)
// tiles are loaded through tensor maps: with the rows inside the heads
// (hn = 0; then slice = H head) a 3-D map (D, N, B N_o H) whose last
// coordinate is (b N_o + o) H + h, as for a contiguous tensor; with the heads
// inside the rows (hn = 1) a 4-D map (D, H, N, B N_o).
struct RowLayout {
  long long slice, head, row;
  int hn;
  __host__ __device__ long long offset(long long bo, int h, long long n) const {
    return bo * slice + h * head + n * row;
  }
};
inline RowLayout contiguous_layout(int N, int H, int D) {
  return RowLayout{static_cast<long long>(H) * N * D, static_cast<long long>(N) * D, D, 0};
}
// Rows [n0, n0 + box) of slice bo, head h through a map of the layout above.
__device__ __forceinline__ void tma_load_rows(void* dst, const CUtensorMap* map, uint64_t* bar, bool hn, int n0, int h,
                                              int bo, int H) {
  if (hn) tma_load_4d(dst, map, bar, 0, h, n0, bo);
  else tma_load_3d(dst, map, bar, 0, n0, bo * H + h);
}

// Forward key-mask record per (slice, 64-key tile): 64 BF16 mask values, then
// a 16-byte header whose first word is nonzero when any value is.
constexpr int kFwdMaskRec = 64 * 2 + 16;

struct FwdArgs {
  CUtensorMap tm_q, tm_k, tm_v, tm_bias;  // Q: 128-row boxes; K, V: 64-row boxes
  const void* mask;    // [B, N_o, N] or null
  const void* bias;    // [B*H, N, N]
  void* bias_padded;   // workspace [B*H, N, Np] (rows padded to a multiple of 8) or null when N % 8 == 0
  uint8_t* mrec;       // workspace [J_K][B*N_o + 4] records, or null (no mask, N % 64 == 0)
  void* o;
  float* lse;
  void* o_resid;
  RowLayout lq;      // q, k, v
  RowLayout lo;      // o, o_resid
  int B, N_o, N, H;
  int test_starve;   // test hook: skip the first K-tile load
  WaitCtl wc;
};

struct BwdArgs {
  CUtensorMap tm_q, tm_k, tm_v, tm_do, tm_biasT;
  const void* bias;  // [B*H][N][N]
  const void* mask;
  const void* o;
  const void* o_resid;
  const float* lse;
  const void* dO;
  void* dq;
  void* dk;
  void* dv;
  void* dbias;
  void* biasT;       // [B*H][N (k)][N (q)] transposed copy of the bias
  uint4* rec;        // [slices][J_Q * 128] query-row records (BF16 splits of -lse sqrt(D), -delta)
  float* dq_part;    // [J_K][slices][J_Q][128 x D]
  float* dbias_part; // [L][B*H*N*N]
  RowLayout lq;      // q, k, v
  RowLayout lo;      // o, o_resid
  RowLayout ldo;     // dO
  RowLayout lg;      // dq, dk, dv
  int B, N_o, N, H, D;
  int dbias_fp32;    // write dbias as FP32 (the sum over this call's slices)
  WaitCtl wc;
};

template <int D> cudaError_t setup_fwd();
// false once the context that setup_fwd configured is gone (a device reset)
bool fwd_attrs_current();
template <int D> cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t stream);
// The forward's preparation: key-mask records and the padded bias copy (each
// only when its workspace pointer is set).
cudaError_t launch_fwd_prep(const FwdArgs& a, cudaStream_t stream);
template <int D> int fwd_smem_bytes();

template <int D> cudaError_t setup_bwd();
template <int D> cudaError_t launch_bwd_preprocess(const BwdArgs& a, cudaStream_t stream);
cudaError_t launch_bwd_transpose_bias(const BwdArgs& a, cudaStream_t stream);
template <int D> cudaError_t launch_bwd_main(const BwdArgs& a, cudaStream_t stream);
template <int D> cudaError_t launch_bwd_reduce_dq(const BwdArgs& a, cudaStream_t stream);
cudaError_t launch_bwd_reduce_dbias(const BwdArgs& a, cudaStream_t stream);
template <int D> int bwd_smem_bytes();
// Non-deterministic ablation of the backward (FP32 atomics; never used by
// tri_attn_bwd): atomic_mask 1 = dQ, 2 = dbias, 3 = dbias and dQ by FP32
// atomics; 4 = dQ by TMA bulk reduction, 6 = that and dbias by atomics.
inline bool atomic_mask_ok(int m) { return m == 1 || m == 2 || m == 3 || m == 4 || m == 6; }
// the dQ tiles go into an FP32 accumulator (atomics or bulk reduction)
inline bool dq_accumulated(int m) { return (m & 5) != 0; }
template <int D> cudaError_t launch_bwd_main_atomic(const BwdArgs& a, int atomic_mask, cudaStream_t stream);
template <int D> cudaError_t launch_bwd_finish_dq(const BwdArgs& a, cudaStream_t stream);
cudaError_t launch_bwd_finish_dbias(const BwdArgs& a, cudaStream_t stream);
// dbias = bf16(sum over r of parts[r]) in ascending r (outer axis split across GPUs).
cudaError_t launch_dbias_combine(const float* parts, int R, size_t elems, void* dbias, cudaStream_t stream);

// Row-major C[M, N] = op(A) op(B) on the tensor cores (gemm.cu): A [M, K]
// (or [K, M] when ta), B [K, N] (or [N, K] when tb), BF16 operands, FP32
// accumulation, C BF16 or FP32 (c_f32); batched over matrices sA / sB / sC
// elements apart.  When the output tiles cannot fill the GPU, K is split into
// FP32 partials in `ws` (gemm_splitk_bytes) added in fixed order by a second
// kernel; without enough `ws` it runs unsplit.
cudaError_t launch_gemm(bool ta, bool tb, int M, int N, int K, const void* A, long long lda, const void* B,
                        long long ldb, void* C, long long ldc, bool c_f32, int batch, long long sA, long long sB,
                        long long sC, void* ws, size_t ws_bytes, const WaitCtl& wc, cudaStream_t s);
size_t gemm_splitk_bytes(int M, int N, int K, int batch);
// The triangle multiplicative update's input projection p = x W_p (x [B*NN]
// [C_z], W_p [C_z][4 C_h + C_z] with column blocks a_v, a_g, b_v, b_g, g) on
// the same tensor cores, p never stored: a = m sigmoid(a_g) a_v and
// b = m sigmoid(b_g) b_v channel-major [B][C_h][NN], g pair-major [B*NN][C_z]
// (mask m optional, [B*NN] BF16).  NN, C_z and C_h multiples of 32.
cudaError_t launch_gated_proj(int B, long long NN, int Cz, int Ch, const void* x, const void* w_p, const void* mask,
                              void* a, void* b, void* g, const WaitCtl& wc, cudaStream_t s);
// C = A op(B) (A [M, K] row-major; B [K, N], or [N, K] when tb) for the
// triangle-attention module, its rows the pairs (b, i, j) of [Bx, Ntok, Ntok]
// (Ntok a multiple of 32): columns [0, nblk H D) go to nblk tensors in the
// core's layout [nblk][Bx, Ntok, H, Ntok, D] at `heads`, the next nbias
// columns to the bias planes [Bx, nbias, Ntok, Ntok], the rest nowhere.
cudaError_t launch_gemm_heads(bool tb, int M, int N, int K, const void* A, long long lda, const void* B, long long ldb,
                              int nblk, int H, int D, int Ntok, int Bx, void* heads, void* bias_planes, int nbias,
                              const WaitCtl& wc, cudaStream_t s);
// Its backward through the gating: recomputes the four branch projections and
// writes dp's first 4 C_h columns (row stride ldp) from dA, dB (channel-major).
cudaError_t launch_gate_bwd_proj(int B, long long NN, int Cz, int Ch, const void* x, const void* w_p,
                                 const void* mask, const void* dA, const void* dB, void* dp, long long ldp,
                                 const WaitCtl& wc, cudaStream_t s);
// The bounded-wait control of the current device (status word, time limit).
WaitCtl current_wait_ctl();

// Kernel kinds of the trace (triattn_trace_enable / triattn_trace_read).
enum KernelKind {
  kKFwd = 0, kKPre, kKTrans, kKMain, kKRedDq, kKRedDb, kKMainAtomic, kKFinDq, kKFinDb, kKCombine, kKFwdPrep,
  kKModLnFwd, kKModLayout, kKModGemm, kKModLnBwd, kKModColSum,
  kKTmLnIn, kKTmProj, kKTmGate, kKTmContract, kKTmLnOut, kKTmOutGate, kKTmColSum, kKGemm, kKTmProjGate,
  kKinds
};
// Runs `launch` on stream `s`, bracketed by a pair of trace events while
// tracing is on.
cudaError_t trace_call(int kind, cudaStream_t s, const std::function<cudaError_t()>& launch);

}  // namespace triattn
