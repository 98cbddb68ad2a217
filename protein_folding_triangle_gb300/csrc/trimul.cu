// Triangle multiplicative update, outgoing and incoming, forward and backward
// ("TurboPairFormer", Figure 12; shapes from Table 10).  With M = B*N*N pairs:
//
//   x = LayerNorm(z)                               z, x  [M, C_z]
//   p = x W_p                                      W_p   [C_z, 4 C_h + C_z]
//   a = m sigmoid(p_ag) p_av,  b = m sigmoid(p_bg) p_bv   (m: optional pair mask)
//   outgoing: X[b,i,j,c] = sum_k a[b,i,k,c] b[b,j,k,c]
//   incoming: X[b,i,j,c] = sum_k a[b,k,i,c] b[b,k,j,c]
//   out = sigmoid(p_g) (LayerNorm(X) W_o)          W_o   [C_h, C_z]
//
// Data layout.  The pair tensors z, x, g, y = LayerNorm(X), u = y W_o are
// pair-major rows; p itself is never stored (below).  The branch operands a, b, the contraction output X and
// their gradients are channel-major: [B][C_h][N][N], so that channel c of
// example b is one row-major N x N matrix A_c (A_c[r][s] = a[b,r,s,c]).  Both
// directions and all three products of the contraction are then one
// strided-batched GEMM over the B*C_h matrices with the right operand flags:
//   outgoing  X_c = A_c B_c^T    dA_c = dX_c B_c     dB_c = dX_c^T A_c
//   incoming  X_c = A_c^T B_c    dA_c = B_c dX_c^T   dB_c = A_c dX_c
// The input projection p = x W_p runs on the library's tensor-core GEMM
// (gemm.cu) with the gating and masking in its epilogue, which writes a and b
// channel-major and g pair-major from the FP32 accumulators, so the 4 C_h +
// C_z wide p never goes to memory; the backward recomputes the four branch
// projections the same way (bitwise the same values) and forms dp's branch
// columns from dA and dB in the epilogue.  The kernels here do the output
// LayerNorm while transposing X back (64 pairs per block through shared
// memory), the output gate, and their backward passes; the other projections,
// the weight gradients and the contraction are plain GEMMs on the same
// tensor cores (BF16 operands, FP32 accumulation; the contraction one batched
// GEMM over the channel matrices, the weight gradients split along the pair
// axis into FP32 partials added in fixed order).  No floating-point atomics:
// every reduction has a fixed order.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <type_traits>

#include "kernels.cuh"
#include "pairops.cuh"
#include "triattn.h"

namespace triattn {
namespace {

using namespace pairops;

constexpr int kPairs = 64;         // pairs per block of the channel-major kernels
constexpr int kCmBwdBlocks = 152 * 2;  // fixed: the output-LayerNorm partial rows depend on it

__device__ __forceinline__ float sigm(float x) { return 1.f / (1.f + __expf(-x)); }

__device__ __forceinline__ void unpack8(const uint4 w, float (&f)[8]) {
  f[0] = bf16lo_to_f32(w.x); f[1] = bf16hi_to_f32(w.x);
  f[2] = bf16lo_to_f32(w.y); f[3] = bf16hi_to_f32(w.y);
  f[4] = bf16lo_to_f32(w.z); f[5] = bf16hi_to_f32(w.z);
  f[6] = bf16lo_to_f32(w.w); f[7] = bf16hi_to_f32(w.w);
}
__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                    pack_bf16x2(f[6], f[7]));
}
__device__ __forceinline__ uint4 ld16(const uint16_t* p) { return *reinterpret_cast<const uint4*>(p); }
__device__ __forceinline__ void st16(uint16_t* p, uint4 v) { *reinterpret_cast<uint4*>(p) = v; }

// A [Ch][64] channel-major tile of pairs [pos0, pos0 + 64) of example b in
// shared memory, as BF16 (the output LayerNorm forward): row c holds the 64
// pairs as 32 words (even pair in the low half) plus one padding word, so
// that both the row-wise fills and the column-wise reads of one pair are free
// of bank conflicts.
constexpr int kRowW = kPairs / 2 + 1;
// The same fill in two steps, so that all of a thread's loads are in flight
// before the first shared-memory store (every kernel here runs 256 threads).
template <int Ch>
__device__ __forceinline__ void fetch_cm_tile(const uint16_t* __restrict__ src, size_t b, size_t pos0, size_t NN,
                                              uint4 (&r)[Ch * 8 / 256]) {
#pragma unroll
  for (int k = 0; k < Ch * 8 / 256; ++k) {
    const int it = threadIdx.x + 256 * k;
    r[k] = ld16(src + (b * Ch + (it >> 3)) * NN + pos0 + 8 * (it & 7));
  }
}
template <int Ch>
__device__ __forceinline__ void put_cm_tile(const uint4 (&r)[Ch * 8 / 256], uint32_t* s) {
#pragma unroll
  for (int k = 0; k < Ch * 8 / 256; ++k) {
    const int it = threadIdx.x + 256 * k;
    uint32_t* d = s + (it >> 3) * kRowW + 4 * (it & 7);
    d[0] = r[k].x;
    d[1] = r[k].y;
    d[2] = r[k].z;
    d[3] = r[k].w;
  }
}
__device__ __forceinline__ float tile_h(const uint32_t* s, int c, int pr) {
  const uint32_t w = s[c * kRowW + (pr >> 1)];
  return (pr & 1) ? bf16hi_to_f32(w) : bf16lo_to_f32(w);
}

// y = LayerNorm(X) for 64 pairs: X channel-major in, y pair-major out (BF16),
// mean and rstd saved.  Thread (pair pr, quarter qq) owns the 8-channel
// chunks qq, qq + 4, ...; the four threads of a pair are adjacent lanes.
template <int Ch>
__global__ void __launch_bounds__(256) ln_cm_fwd_kernel(const uint16_t* __restrict__ X,
                                                        const float* __restrict__ gamma,
                                                        const float* __restrict__ beta, uint16_t* __restrict__ y,
                                                        float* __restrict__ mean_out, float* __restrict__ rstd_out,
                                                        size_t NN) {
  extern __shared__ uint32_t sXh[];  // [Ch][kRowW] BF16 pairs
  constexpr int kCh = Ch / 32;
  const size_t m0 = static_cast<size_t>(blockIdx.x) * kPairs;
  const size_t b = m0 / NN, pos0 = m0 % NN;
  {
    uint4 r[Ch * 8 / 256];
    fetch_cm_tile<Ch>(X, b, pos0, NN, r);
    put_cm_tile<Ch>(r, sXh);
  }
  __syncthreads();
  const int pr = threadIdx.x >> 2, qq = threadIdx.x & 3;
  float v[kCh][8];
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < kCh; ++i)
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      v[i][e] = tile_h(sXh, 8 * (qq + 4 * i) + e, pr);
      s += v[i][e];
    }
  s += __shfl_xor_sync(0xffffffffu, s, 1);
  s += __shfl_xor_sync(0xffffffffu, s, 2);
  const float mean = s * (1.f / Ch);
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < kCh; ++i)
#pragma unroll
    for (int e = 0; e < 8; ++e) ss += (v[i][e] - mean) * (v[i][e] - mean);
  ss += __shfl_xor_sync(0xffffffffu, ss, 1);
  ss += __shfl_xor_sync(0xffffffffu, ss, 2);
  const float rstd = rsqrtf(ss * (1.f / Ch) + 1e-5f);
  const size_t m = m0 + pr;
#pragma unroll
  for (int i = 0; i < kCh; ++i) {
    const int c0 = 8 * (qq + 4 * i);
    float o[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) o[e] = (v[i][e] - mean) * rstd * gamma[c0 + e] + beta[c0 + e];
    st16(y + m * Ch + c0, pack8(o));
  }
  if (qq == 0) {
    mean_out[m] = mean;
    rstd_out[m] = rstd;
  }
}

// 16-byte global -> shared copies that bypass the registers (cp.async, L2
// only), in commit groups; wait<n> returns once at most n groups are pending.
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int n>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(n) : "memory"); }

// Backward of the output LayerNorm: dX (channel-major BF16) from dy (pair-major
// BF16) and X.  A block walks its tiles of 64 pairs.  Thread (pair slot pl,
// part p) takes the C_h / 8 channels [p C_h / 8, (p + 1) C_h / 8) of pairs
// pl and pl + 32; a pair's sums are a butterfly over its 8 part threads.
// The X tile comes into shared memory by cp.async, double buffered (the next
// tile's copy, and its dy and statistics in registers, are in flight while
// this one is worked on), as channel rows of 128 bytes whose 16-byte chunks
// are rotated by XOR with the row's part, so that the 8 parts reading one
// pair hit distinct banks; dX overwrites it in place and is stored
// channel-major from there.  dgamma / dbeta: each thread adds its channels
// over its pairs in register accumulators (tile order); at the end a fixed
// butterfly adds the 4 pair slots of a warp and the block adds its 8 warps in
// order: one partial row per block.
template <int Ch>
struct CmBwd {
  static constexpr int kCT = Ch / 8;            // channels per thread
  static constexpr int kTileBytes = Ch * 128;   // one X tile: Ch rows of 64 BF16 pairs
  static constexpr int kGam = 2 * kTileBytes;   // gamma [Ch] fp32
  static constexpr int kRed = kGam + Ch * 4;    // [8 warps][2][Ch] fp32
  static constexpr int kBytes = kRed + 8 * 2 * Ch * 4;
};
template <int Ch>
__global__ void __launch_bounds__(256, 2) ln_cm_bwd_kernel(const uint16_t* __restrict__ X,
                                                           const uint16_t* __restrict__ dy,
                                                           const float* __restrict__ gamma,
                                                           const float* __restrict__ mean_in,
                                                           const float* __restrict__ rstd_in,
                                                           uint16_t* __restrict__ dX, float* __restrict__ part_g,
                                                           float* __restrict__ part_b, size_t NN, size_t tiles) {
  using L = CmBwd<Ch>;
  constexpr int kCT = L::kCT;
  extern __shared__ __align__(128) uint8_t smc[];
  float* sGam = reinterpret_cast<float*>(smc + L::kGam);
  float* sRed = reinterpret_cast<float*>(smc + L::kRed);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int p = tid & 7, pl = tid >> 3;
  const int c0 = p * kCT;
  for (int c = tid; c < Ch; c += 256) sGam[c] = gamma[c];
  float accg[kCT], accb[kCT];
#pragma unroll
  for (int j = 0; j < kCT; ++j) accg[j] = accb[j] = 0.f;
  // X tile -> buffer bb (one commit group)
  auto fill = [&](size_t tile, int bb) {
    const size_t m0 = tile * kPairs;
    const size_t b = m0 / NN, pos0 = m0 % NN;
    uint8_t* buf = smc + bb * L::kTileBytes;
#pragma unroll
    for (int k = 0; k < Ch * 8 / 256; ++k) {
      const int it = tid + 256 * k;
      const int c = it >> 3, q = it & 7;
      cp_async16(buf + c * 128 + ((q ^ (c / kCT)) << 4), X + (b * Ch + c) * NN + pos0 + 8 * q);
    }
    cp_async_commit();
  };
  struct Dy {
    Packed<kCT> d[2];
    float mean[2], rstd[2];
  };
  auto fetch = [&](size_t tile, Dy& r) {
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      const size_t m = tile * kPairs + 32 * s + pl;
      ld_packed<kCT>(dy + m * Ch + c0, r.d[s]);
      r.mean[s] = mean_in[m];
      r.rstd[s] = rstd_in[m];
    }
  };
  Dy cur, nxt;
  if (blockIdx.x < tiles) {
    fill(blockIdx.x, 0);
    fetch(blockIdx.x, cur);
  }
  int k = 0;
  for (size_t tile = blockIdx.x; tile < tiles; tile += gridDim.x, ++k) {
    const int bb = k & 1;
    if (tile + gridDim.x < tiles) {
      fill(tile + gridDim.x, bb ^ 1);  // that buffer was drained before the last barrier
      fetch(tile + gridDim.x, nxt);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();  // this tile's X (and gamma) visible to every thread
    uint8_t* buf = smc + bb * L::kTileBytes;
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      const int pr = 32 * s + pl, w = pr >> 1;
      // byte offset of this pair's element in a channel row of this part
      const int off = (((w >> 2) ^ p) << 4) + (w & 3) * 4 + (pr & 1) * 2;
      uint16_t* xp = reinterpret_cast<uint16_t*>(buf + c0 * 128 + off);
      const float mean = cur.mean[s], rstd = cur.rstd[s];
      float d[kCT], xh[kCT];
      unpack<kCT>(cur.d[s], d);
      float sg = 0.f, sgx = 0.f;
#pragma unroll
      for (int j = 0; j < kCT; ++j) {
        xh[j] = (bf16lo_to_f32(xp[j * 64]) - mean) * rstd;  // rows are 64 halfwords apart
        const float g = d[j] * sGam[c0 + j];
        sg += g;
        sgx += g * xh[j];
        accg[j] += d[j] * xh[j];
        accb[j] += d[j];
      }
#pragma unroll
      for (int off2 = 1; off2 < 8; off2 <<= 1) {
        sg += __shfl_xor_sync(0xffffffffu, sg, off2);
        sgx += __shfl_xor_sync(0xffffffffu, sgx, off2);
      }
      const float a = sg * (1.f / Ch), bb2 = sgx * (1.f / Ch);
#pragma unroll
      for (int j = 0; j < kCT; ++j)
        xp[j * 64] = static_cast<uint16_t>(pack_bf16x2(rstd * (d[j] * sGam[c0 + j] - a - xh[j] * bb2), 0.f) & 0xFFFFu);
    }
    __syncthreads();  // dX of the tile complete in the buffer
    {
      const size_t m0 = tile * kPairs;
      const size_t b = m0 / NN, pos0 = m0 % NN;
#pragma unroll
      for (int kk = 0; kk < Ch * 8 / 256; ++kk) {
        const int it = tid + 256 * kk;
        const int c = it >> 3, q = it & 7;
        st16(dX + (b * Ch + c) * NN + pos0 + 8 * q,
             *reinterpret_cast<const uint4*>(buf + c * 128 + ((q ^ (c / kCT)) << 4)));
      }
    }
    cur = nxt;
    __syncthreads();  // the buffer is drained before the next iteration refills it
  }
  // the 4 pair slots of a warp (lanes 8 apart), then the 8 warps in order
#pragma unroll
  for (int j = 0; j < kCT; ++j)
#pragma unroll
    for (int off2 = 8; off2 < 32; off2 <<= 1) {
      accg[j] += __shfl_xor_sync(0xffffffffu, accg[j], off2);
      accb[j] += __shfl_xor_sync(0xffffffffu, accb[j], off2);
    }
  if (lane < 8) {
#pragma unroll
    for (int j = 0; j < kCT; ++j) {
      sRed[(warp * 2) * Ch + c0 + j] = accg[j];
      sRed[(warp * 2 + 1) * Ch + c0 + j] = accb[j];
    }
  }
  __syncthreads();
  for (int c = tid; c < Ch; c += 256) {
    float g = 0.f, bsum = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      g += sRed[(w * 2) * Ch + c];
      bsum += sRed[(w * 2 + 1) * Ch + c];
    }
    part_g[static_cast<size_t>(blockIdx.x) * Ch + c] = g;
    part_b[static_cast<size_t>(blockIdx.x) * Ch + c] = bsum;
  }
}

// out = sigmoid(g) u, 8 features per thread (g, u, out [M, C_z]).
__global__ void __launch_bounds__(256) gate_out_kernel(const uint16_t* __restrict__ g_in,
                                                       const uint16_t* __restrict__ u, uint16_t* __restrict__ out,
                                                       int Cz, size_t M) {
  const size_t t = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int chunks = Cz / 8;
  if (t >= M * chunks) return;
  const size_t m = t / chunks;
  const int c0 = 8 * static_cast<int>(t % chunks);
  float g[8], uv[8], o[8];
  unpack8(ld16(g_in + m * Cz + c0), g);
  unpack8(ld16(u + m * Cz + c0), uv);
#pragma unroll
  for (int e = 0; e < 8; ++e) o[e] = sigm(g[e]) * uv[e];
  st16(out + m * Cz + c0, pack8(o));
}

// Backward of the output gate: du = d_out sigmoid(g) (BF16 [M, C_z]) and
// dp[:, goff + c] = d_out u sigmoid(g) (1 - sigmoid(g)) (dp row stride ld).
__global__ void __launch_bounds__(256) gate_out_bwd_kernel(const uint16_t* __restrict__ g_in, int ld, int goff,
                                                           const uint16_t* __restrict__ u,
                                                           const uint16_t* __restrict__ d_out,
                                                           uint16_t* __restrict__ du, uint16_t* __restrict__ dp,
                                                           int Cz, size_t M) {
  const size_t t = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int chunks = Cz / 8;
  if (t >= M * chunks) return;
  const size_t m = t / chunks;
  const int c0 = 8 * static_cast<int>(t % chunks);
  float g[8], uv[8], d[8], o1[8], o2[8];
  unpack8(ld16(g_in + m * Cz + c0), g);
  unpack8(ld16(u + m * Cz + c0), uv);
  unpack8(ld16(d_out + m * Cz + c0), d);
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const float sg = sigm(g[e]);
    o1[e] = d[e] * sg;
    o2[e] = d[e] * uv[e] * sg * (1.f - sg);
  }
  st16(du + m * Cz + c0, pack8(o1));
  st16(dp + m * ld + goff + c0, pack8(o2));
}

// ---------------------------------------------------------------- host side
size_t rup(size_t x) { return (x + 255) / 256 * 256; }

struct TmDims {
  size_t B, N, NN, M, Cz, Ch, F, Fp;
  bool incoming;
};
TmDims tm_dims(const triattn_trimul_shape* s) {
  TmDims d;
  d.B = s->B;
  d.N = s->N;
  d.NN = d.N * d.N;
  d.M = d.B * d.NN;
  d.Cz = s->C_z;
  d.Ch = s->C_h;
  d.F = 4 * d.Ch + d.Cz;
  d.Fp = (d.F + 7) / 8 * 8;
  d.incoming = s->direction == TRIATTN_TRIMUL_INCOMING;
  return d;
}

struct TmCtx {
  size_t x, mean_in, rstd_in, g, a, b, X, mean_out, rstd_out, y, u, total;
};
TmCtx tm_ctx(const TmDims& d) {
  TmCtx c;
  size_t o = 0;
  const size_t cm = d.B * d.Ch * d.NN * 2;
  c.x = o;        o += rup(d.M * d.Cz * 2);
  c.mean_in = o;  o += rup(d.M * 4);
  c.rstd_in = o;  o += rup(d.M * 4);
  c.g = o;        o += rup(d.M * d.Cz * 2);
  c.a = o;        o += rup(cm);
  c.b = o;        o += rup(cm);
  c.X = o;        o += rup(cm);
  c.mean_out = o; o += rup(d.M * 4);
  c.rstd_out = o; o += rup(d.M * 4);
  c.y = o;        o += rup(d.M * d.Ch * 2);
  c.u = o;        o += rup(d.M * d.Cz * 2);
  c.total = o;
  return c;
}

struct TmWs {
  size_t gemm, du, dp, dy, dX, dA, dB, dx, pg_in, pb_in, pg_out, pb_out, total;
};
TmWs tm_ws(const TmDims& d) {
  TmWs w;
  size_t o = 0;
  const size_t cm = d.B * d.Ch * d.NN * 2;
  w.gemm = o;   o += rup(kGemmWorkspace);
  w.du = o;     o += rup(d.M * d.Cz * 2);
  w.dp = o;     o += rup(d.M * d.Fp * 2);
  w.dy = o;     o += rup(d.M * d.Ch * 2);
  w.dX = o;     o += rup(cm);
  w.dA = o;     o += rup(cm);
  w.dB = o;     o += rup(cm);
  w.dx = o;     o += rup(d.M * d.Cz * 2);
  w.pg_in = o;  o += rup(static_cast<size_t>(kLnBlocks) * d.Cz * 4);
  w.pb_in = o;  o += rup(static_cast<size_t>(kLnBlocks) * d.Cz * 4);
  w.pg_out = o; o += rup(static_cast<size_t>(kCmBwdBlocks) * d.Ch * 4);
  w.pb_out = o; o += rup(static_cast<size_t>(kCmBwdBlocks) * d.Ch * 4);
  w.total = o;
  return w;
}

triattn_status check_trimul(const triattn_trimul_shape* s) {
  if (s == nullptr || s->flags != 0 || s->B < 1 || s->N < 1 || s->C_z < 1 || s->C_h < 1 ||
      (s->direction != TRIATTN_TRIMUL_OUTGOING && s->direction != TRIATTN_TRIMUL_INCOMING))
    return TRIATTN_ERR_INVALID_ARG;
  if (s->N % 8 != 0 || s->N > 4096 || !ln_width_ok(s->C_z) || s->C_h % 32 != 0 || s->C_h > 128)
    return TRIATTN_ERR_UNSUPPORTED;
  if (static_cast<size_t>(s->B) * s->N * s->N > 0x7fffffffull) return TRIATTN_ERR_UNSUPPORTED;
  return TRIATTN_OK;
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
unsigned blocks_for(size_t n) { return static_cast<unsigned>((n + 255) / 256); }

// Dynamic shared memory of the channel-major kernels.
template <int Ch> constexpr int ln_cm_fwd_smem() { return Ch * kRowW * 4; }
template <int Ch> constexpr int ln_cm_bwd_smem() { return CmBwd<Ch>::kBytes; }

template <int Ch>
cudaError_t set_attrs() {
  cudaError_t e = cudaFuncSetAttribute(ln_cm_fwd_kernel<Ch>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       ln_cm_fwd_smem<Ch>());
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(ln_cm_bwd_kernel<Ch>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             ln_cm_bwd_smem<Ch>());
  return e;
}

// The channel-major kernels, dispatched on C_h.
struct CmLaunch {
  const TmDims& d;
  cudaStream_t s;

  template <int Ch>
  cudaError_t ln_fwd(const uint16_t* X, const float* g, const float* b, uint16_t* y, float* mean, float* rstd) const {
    cudaError_t e = set_attrs<Ch>();
    if (e != cudaSuccess) return e;
    ln_cm_fwd_kernel<Ch><<<static_cast<unsigned>(d.M / kPairs), 256, ln_cm_fwd_smem<Ch>(), s>>>(X, g, b, y, mean, rstd,
                                                                                          d.NN);
    return cudaGetLastError();
  }
  template <int Ch>
  cudaError_t ln_bwd(const uint16_t* X, const uint16_t* dy, const float* g, const float* mean, const float* rstd,
                     uint16_t* dX, float* pg, float* pb) const {
    cudaError_t e = set_attrs<Ch>();
    if (e != cudaSuccess) return e;
    const size_t tiles = d.M / kPairs;
    ln_cm_bwd_kernel<Ch><<<kCmBwdBlocks, 256, ln_cm_bwd_smem<Ch>(), s>>>(X, dy, g, mean, rstd, dX, pg, pb, d.NN, tiles);
    return cudaGetLastError();
  }
};

// f(std::integral_constant<int, Ch>) for the supported C_h.
template <typename F>
cudaError_t by_ch(size_t Ch, F&& f) {
  switch (Ch) {
    case 32: return f(std::integral_constant<int, 32>{});
    case 64: return f(std::integral_constant<int, 64>{});
    case 96: return f(std::integral_constant<int, 96>{});
    case 128: return f(std::integral_constant<int, 128>{});
  }
  return cudaErrorInvalidValue;
}

// The contraction as one strided-batched GEMM over the B * C_h channel
// matrices: C_c = op(P_c) op(Q_c), every matrix N x N, row-major.
triattn_status contract(void* gws, cudaStream_t s, const TmDims& d, bool tp, bool tq, const void* P,
                        const void* Q, void* C) {
  const int n = static_cast<int>(d.N);
  const long long st = static_cast<long long>(d.NN);
  return gemm_traced(kKTmContract, gws, s, tp, tq, n, n, n, P, n, Q, n, C, n, false, static_cast<int>(d.B * d.Ch),
                     st, st, st);
}

}  // namespace
}  // namespace triattn

using namespace triattn;

extern "C" {

size_t triattn_trimul_ctx_bytes(const triattn_trimul_shape* shape) {
  if (check_trimul(shape) != TRIATTN_OK) return 0;
  return tm_ctx(tm_dims(shape)).total;
}

size_t triattn_trimul_workspace_bytes(const triattn_trimul_shape* shape) {
  if (check_trimul(shape) != TRIATTN_OK) return 0;
  return tm_ws(tm_dims(shape)).total;
}

triattn_status triattn_trimul_fwd(const triattn_trimul_shape* shape, const void* z, const void* mask,
                                  const float* ln_in_w, const float* ln_in_b, const void* w_p,
                                  const float* ln_out_w, const float* ln_out_b, const void* w_o, void* out,
                                  void* ctx, void* workspace, size_t workspace_bytes, void* stream) {
  triattn_status st = check_trimul(shape);
  if (st != TRIATTN_OK) return st;
  const void* req[] = {z, ln_in_w, ln_in_b, w_p, ln_out_w, ln_out_b, w_o, out, ctx};
  for (const void* q : req)
    if (q == nullptr || !al16(q)) return TRIATTN_ERR_INVALID_ARG;
  if ((mask != nullptr && !al16(mask)) || (reinterpret_cast<uintptr_t>(ctx) & 255u) != 0)
    return TRIATTN_ERR_INVALID_ARG;
  const TmDims d = tm_dims(shape);
  const TmCtx c = tm_ctx(d);
  const TmWs w = tm_ws(d);
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || workspace_bytes < w.total)
    return TRIATTN_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* cx = static_cast<uint8_t*>(ctx);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void* const gws = ws + w.gemm;
  const int M = static_cast<int>(d.M), Cz = static_cast<int>(d.Cz), Ch = static_cast<int>(d.Ch);
  const uint16_t* mk = static_cast<const uint16_t*>(mask);
  uint16_t* G = reinterpret_cast<uint16_t*>(cx + c.g);
  uint16_t* A = reinterpret_cast<uint16_t*>(cx + c.a);
  uint16_t* Bo = reinterpret_cast<uint16_t*>(cx + c.b);
  uint16_t* X = reinterpret_cast<uint16_t*>(cx + c.X);
  uint16_t* y = reinterpret_cast<uint16_t*>(cx + c.y);
  uint16_t* u = reinterpret_cast<uint16_t*>(cx + c.u);
  const CmLaunch L{d, s};
  // x = LayerNorm(z);  p = x W_p
  if (trace_call(kKTmLnIn, s, [&] {
        return ln_rows_fwd(d.M, Cz, z, ln_in_w, ln_in_b, cx + c.x, reinterpret_cast<float*>(cx + c.mean_in),
                           reinterpret_cast<float*>(cx + c.rstd_in), s);
      }) != cudaSuccess)
    return TRIATTN_ERR_CUDA;
  // p = x W_p on the tensor cores with the gating in the epilogue: a, b
  // gated, masked, channel-major; g pair-major; p itself is not stored
  if (trace_call(kKTmProjGate, s, [&] {
        return launch_gated_proj(static_cast<int>(d.B), static_cast<long long>(d.NN), Cz, Ch, cx + c.x, w_p, mk, A,
                                 Bo, G, current_wait_ctl(), s);
      }) != cudaSuccess)
    return TRIATTN_ERR_CUDA;
  // X_c = A_c B_c^T (outgoing) or A_c^T B_c (incoming)
  if (contract(gws, s, d, d.incoming, !d.incoming, A, Bo, X) != TRIATTN_OK) return TRIATTN_ERR_CUDA;
  // y = LayerNorm(X) (pair-major);  u = y W_o;  out = sigmoid(g) u
  if (trace_call(kKTmLnOut, s, [&] {
        return by_ch(d.Ch, [&](auto ic) {
          return L.template ln_fwd<decltype(ic)::value>(X, ln_out_w, ln_out_b, y,
                                                        reinterpret_cast<float*>(cx + c.mean_out),
                                                        reinterpret_cast<float*>(cx + c.rstd_out));
        });
      }) != cudaSuccess)
    return TRIATTN_ERR_CUDA;
  if (gemm_traced(kKTmProj, gws, s, false, false, M, Cz, Ch, y, Ch, w_o, Cz, u, Cz, false) != TRIATTN_OK)
    return TRIATTN_ERR_CUDA;
  const cudaError_t e = trace_call(kKTmOutGate, s, [&] {
    gate_out_kernel<<<blocks_for(d.M * d.Cz / 8), 256, 0, s>>>(G, u, static_cast<uint16_t*>(out), Cz, d.M);
    return cudaGetLastError();
  });
  return e == cudaSuccess ? TRIATTN_OK : TRIATTN_ERR_CUDA;
}

triattn_status triattn_trimul_bwd(const triattn_trimul_shape* shape, const void* z, const void* mask,
                                  const float* ln_in_w, const void* w_p, const float* ln_out_w, const void* w_o,
                                  const void* ctx, const void* d_out, void* dz, float* d_ln_in_w, float* d_ln_in_b,
                                  float* d_w_p, float* d_ln_out_w, float* d_ln_out_b, float* d_w_o,
                                  void* workspace, size_t workspace_bytes, void* stream) {
  triattn_status st = check_trimul(shape);
  if (st != TRIATTN_OK) return st;
  const void* req[] = {z, ln_in_w, w_p, ln_out_w, w_o, ctx, d_out, dz, d_ln_in_w, d_ln_in_b, d_w_p,
                       d_ln_out_w, d_ln_out_b, d_w_o};
  for (const void* q : req)
    if (q == nullptr || !al16(q)) return TRIATTN_ERR_INVALID_ARG;
  if ((mask != nullptr && !al16(mask)) || (reinterpret_cast<uintptr_t>(ctx) & 255u) != 0)
    return TRIATTN_ERR_INVALID_ARG;
  const TmDims d = tm_dims(shape);
  const TmCtx c = tm_ctx(d);
  const TmWs w = tm_ws(d);
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || workspace_bytes < w.total)
    return TRIATTN_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const uint8_t* cx = static_cast<const uint8_t*>(ctx);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void* const gws = ws + w.gemm;
  const int M = static_cast<int>(d.M), Cz = static_cast<int>(d.Cz), Ch = static_cast<int>(d.Ch),
            F = static_cast<int>(d.F), Fp = static_cast<int>(d.Fp);
  const uint16_t* mk = static_cast<const uint16_t*>(mask);
  const uint16_t* G = reinterpret_cast<const uint16_t*>(cx + c.g);
  const uint16_t* A = reinterpret_cast<const uint16_t*>(cx + c.a);
  const uint16_t* Bo = reinterpret_cast<const uint16_t*>(cx + c.b);
  const uint16_t* X = reinterpret_cast<const uint16_t*>(cx + c.X);
  uint16_t* du = reinterpret_cast<uint16_t*>(ws + w.du);
  uint16_t* dp = reinterpret_cast<uint16_t*>(ws + w.dp);
  uint16_t* dy = reinterpret_cast<uint16_t*>(ws + w.dy);
  uint16_t* dX = reinterpret_cast<uint16_t*>(ws + w.dX);
  uint16_t* dA = reinterpret_cast<uint16_t*>(ws + w.dA);
  uint16_t* dB = reinterpret_cast<uint16_t*>(ws + w.dB);
  uint16_t* dx = reinterpret_cast<uint16_t*>(ws + w.dx);
  const CmLaunch L{d, s};
  // out = sigmoid(g) u:  du, and dp's output-gate columns
  if (trace_call(kKTmOutGate, s, [&] {
        gate_out_bwd_kernel<<<blocks_for(d.M * d.Cz / 8), 256, 0, s>>>(
            G, Fp, 4 * Ch, reinterpret_cast<const uint16_t*>(cx + c.u), static_cast<const uint16_t*>(d_out), du, dp,
            Cz, d.M);
        return cudaGetLastError();
      }) != cudaSuccess)
    return TRIATTN_ERR_CUDA;
  // u = y W_o:  dW_o = y^T du,  dy = du W_o^T (BF16, as every activation gradient here)
  if (gemm_traced(kKTmProj, gws, s, true, false, Ch, Cz, M, cx + c.y, Ch, du, Cz, d_w_o, Cz, true) !=
          TRIATTN_OK ||
      gemm_traced(kKTmProj, gws, s, false, true, M, Ch, Cz, du, Cz, w_o, Cz, dy, Ch, false) != TRIATTN_OK)
    return TRIATTN_ERR_CUDA;
  // y = LayerNorm(X):  dX (channel-major), output-LayerNorm partial sums
  float* pg_out = reinterpret_cast<float*>(ws + w.pg_out);
  float* pb_out = reinterpret_cast<float*>(ws + w.pb_out);
  if (trace_call(kKTmLnOut, s, [&] {
        return by_ch(d.Ch, [&](auto ic) {
          return L.template ln_bwd<decltype(ic)::value>(X, dy, ln_out_w,
                                                        reinterpret_cast<const float*>(cx + c.mean_out),
                                                        reinterpret_cast<const float*>(cx + c.rstd_out), dX, pg_out,
                                                        pb_out);
        });
      }) != cudaSuccess)
    return TRIATTN_ERR_CUDA;
  // the contraction
  triattn_status cs;
  if (!d.incoming) {
    cs = contract(gws, s, d, false, false, dX, Bo, dA);                      // dA_c = dX_c B_c
    if (cs == TRIATTN_OK) cs = contract(gws, s, d, true, false, dX, A, dB);  // dB_c = dX_c^T A_c
  } else {
    cs = contract(gws, s, d, false, true, Bo, dX, dA);                       // dA_c = B_c dX_c^T
    if (cs == TRIATTN_OK) cs = contract(gws, s, d, false, false, A, dX, dB); // dB_c = A_c dX_c
  }
  if (cs != TRIATTN_OK) return cs;
  // the gating:  dp's first 4 C_h columns, the branch projections recomputed
  // from x on the tensor cores
  if (trace_call(kKTmProjGate, s, [&] {
        return launch_gate_bwd_proj(static_cast<int>(d.B), static_cast<long long>(d.NN), Cz, Ch, cx + c.x, w_p, mk,
                                    dA, dB, dp, Fp, current_wait_ctl(), s);
      }) != cudaSuccess)
    return TRIATTN_ERR_CUDA;
  // p = x W_p:  dW_p = x^T dp,  dx = dp W_p^T (BF16)
  if (gemm_traced(kKTmProj, gws, s, true, false, Cz, F, M, cx + c.x, Cz, dp, Fp, d_w_p, F, true) != TRIATTN_OK ||
      gemm_traced(kKTmProj, gws, s, false, true, M, Cz, F, dp, Fp, w_p, F, dx, Cz, false) != TRIATTN_OK)
    return TRIATTN_ERR_CUDA;
  // x = LayerNorm(z)
  float* pg_in = reinterpret_cast<float*>(ws + w.pg_in);
  float* pb_in = reinterpret_cast<float*>(ws + w.pb_in);
  if (trace_call(kKTmLnIn, s, [&] {
        return ln_rows_bwd(d.M, Cz, z, dx, ln_in_w, reinterpret_cast<const float*>(cx + c.mean_in),
                           reinterpret_cast<const float*>(cx + c.rstd_in), dz, pg_in, pb_in, s);
      }) != cudaSuccess)
    return TRIATTN_ERR_CUDA;
  const cudaError_t e = trace_call(kKTmColSum, s, [&] {
    cudaError_t r = column_sums(pg_in, pb_in, kLnBlocks, Cz, d_ln_in_w, d_ln_in_b, s);
    if (r == cudaSuccess) r = column_sums(pg_out, pb_out, kCmBwdBlocks, Ch, d_ln_out_w, d_ln_out_b, s);
    return r;
  });
  return e == cudaSuccess ? TRIATTN_OK : TRIATTN_ERR_CUDA;
}

}  // extern "C"
