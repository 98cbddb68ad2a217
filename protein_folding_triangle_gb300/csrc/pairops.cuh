// Kernels and helpers shared by the pair-tensor layers (the triangle-attention
// module and the triangle multiplicative update): LayerNorm over the feature
// axis of a row-major [M, C] pair tensor, forward and backward, the
// fixed-order sums of the LayerNorm parameter gradients, and the traced call
// of the library's tensor-core GEMM in row-major terms.
#pragma once
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "kernels.cuh"
#include "triattn.h"

// Everything here has internal linkage: each translation unit that includes
// this header gets its own copy of the kernels and of the handle table.
namespace triattn {
namespace {
namespace pairops {

constexpr int kMaxC = 256;          // LayerNorm: up to 8 features per lane
constexpr int kLnBwdPerSm = 3;                   // backward blocks resident per SM (register bound)
constexpr int kLnBlocks = 152 * kLnBwdPerSm;     // backward grid, one wave; the dgamma / dbeta partial rows depend on it
constexpr int kLnFwdPerSm = 4;                   // forward blocks resident per SM
constexpr int kLnFwdBlocks = 152 * kLnFwdPerSm;  // forward grid (no partials), one wave
constexpr size_t kGemmWorkspace = 32u << 20;  // split-K partials of the weight-gradient GEMMs

inline bool ln_width_ok(int C) { return C >= 32 && C <= kMaxC && C % 32 == 0; }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// K consecutive features of one row, in the widest aligned vector accesses
// the count allows (rows are C = 32 K elements, so lane l's run starts at
// l K, which is 2 K-byte aligned for BF16 and 4 K-byte aligned for FP32).
template <int K>
__device__ __forceinline__ void ld_bf16(const uint16_t* p, float (&f)[K]) {
  if constexpr (K % 8 == 0) {
#pragma unroll
    for (int j = 0; j < K / 8; ++j) {
      const uint4 w = reinterpret_cast<const uint4*>(p)[j];
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        f[8 * j + 2 * h] = bf16lo_to_f32(ws[h]);
        f[8 * j + 2 * h + 1] = bf16hi_to_f32(ws[h]);
      }
    }
  } else if constexpr (K % 4 == 0) {
#pragma unroll
    for (int j = 0; j < K / 4; ++j) {
      const uint2 w = reinterpret_cast<const uint2*>(p)[j];
      f[4 * j] = bf16lo_to_f32(w.x);
      f[4 * j + 1] = bf16hi_to_f32(w.x);
      f[4 * j + 2] = bf16lo_to_f32(w.y);
      f[4 * j + 3] = bf16hi_to_f32(w.y);
    }
  } else if constexpr (K % 2 == 0) {
#pragma unroll
    for (int j = 0; j < K / 2; ++j) {
      const uint32_t w = reinterpret_cast<const uint32_t*>(p)[j];
      f[2 * j] = bf16lo_to_f32(w);
      f[2 * j + 1] = bf16hi_to_f32(w);
    }
  } else {
#pragma unroll
    for (int e = 0; e < K; ++e) f[e] = bf16lo_to_f32(p[e]);
  }
}
template <int K>
__device__ __forceinline__ void st_bf16(uint16_t* p, const float (&f)[K]) {
  if constexpr (K % 8 == 0) {
#pragma unroll
    for (int j = 0; j < K / 8; ++j)
      reinterpret_cast<uint4*>(p)[j] =
          make_uint4(pack_bf16x2(f[8 * j], f[8 * j + 1]), pack_bf16x2(f[8 * j + 2], f[8 * j + 3]),
                     pack_bf16x2(f[8 * j + 4], f[8 * j + 5]), pack_bf16x2(f[8 * j + 6], f[8 * j + 7]));
  } else if constexpr (K % 4 == 0) {
#pragma unroll
    for (int j = 0; j < K / 4; ++j)
      reinterpret_cast<uint2*>(p)[j] =
          make_uint2(pack_bf16x2(f[4 * j], f[4 * j + 1]), pack_bf16x2(f[4 * j + 2], f[4 * j + 3]));
  } else if constexpr (K % 2 == 0) {
#pragma unroll
    for (int j = 0; j < K / 2; ++j) reinterpret_cast<uint32_t*>(p)[j] = pack_bf16x2(f[2 * j], f[2 * j + 1]);
  } else {
#pragma unroll
    for (int e = 0; e < K; ++e) p[e] = static_cast<uint16_t>(pack_bf16x2(f[e], 0.f) & 0xFFFFu);
  }
}
template <int K>
__device__ __forceinline__ void ld_f32(const float* p, float (&f)[K]) {
  if constexpr (K % 4 == 0) {
#pragma unroll
    for (int j = 0; j < K / 4; ++j) {
      const float4 v = reinterpret_cast<const float4*>(p)[j];
      f[4 * j] = v.x;
      f[4 * j + 1] = v.y;
      f[4 * j + 2] = v.z;
      f[4 * j + 3] = v.w;
    }
  } else if constexpr (K % 2 == 0) {
#pragma unroll
    for (int j = 0; j < K / 2; ++j) {
      const float2 v = reinterpret_cast<const float2*>(p)[j];
      f[2 * j] = v.x;
      f[2 * j + 1] = v.y;
    }
  } else {
#pragma unroll
    for (int e = 0; e < K; ++e) f[e] = p[e];
  }
}

// K consecutive BF16 features of one row kept packed (two per word; for odd
// K the last word holds one), loaded with the widest aligned accesses, and
// their unpacking: a warp can keep several rows in flight for the registers
// of one unpacked row.
template <int K>
struct Packed {
  uint32_t w[(K + 1) / 2];
};
template <int K>
__device__ __forceinline__ void ld_packed(const uint16_t* p, Packed<K>& r) {
  if constexpr (K % 8 == 0) {
#pragma unroll
    for (int j = 0; j < K / 8; ++j) {
      const uint4 v = reinterpret_cast<const uint4*>(p)[j];
      r.w[4 * j] = v.x;
      r.w[4 * j + 1] = v.y;
      r.w[4 * j + 2] = v.z;
      r.w[4 * j + 3] = v.w;
    }
  } else if constexpr (K % 4 == 0) {
#pragma unroll
    for (int j = 0; j < K / 4; ++j) {
      const uint2 v = reinterpret_cast<const uint2*>(p)[j];
      r.w[2 * j] = v.x;
      r.w[2 * j + 1] = v.y;
    }
  } else if constexpr (K % 2 == 0) {
#pragma unroll
    for (int j = 0; j < K / 2; ++j) r.w[j] = reinterpret_cast<const uint32_t*>(p)[j];
  } else {
#pragma unroll
    for (int j = 0; j < (K + 1) / 2; ++j)
      r.w[j] = static_cast<uint32_t>(p[2 * j]) | (2 * j + 1 < K ? static_cast<uint32_t>(p[2 * j + 1]) << 16 : 0u);
  }
}
template <int K>
__device__ __forceinline__ void unpack(const Packed<K>& r, float (&f)[K]) {
#pragma unroll
  for (int e = 0; e < K; ++e) f[e] = (e & 1) ? bf16hi_to_f32(r.w[e >> 1]) : bf16lo_to_f32(r.w[e >> 1]);
}

// One warp per pair: x = (z - mean) * rstd * gamma + beta (BF16), mean and
// rstd saved in FP32.  Lane l holds the C / 32 consecutive features from
// l C / 32; the loads of several pairs are in flight together.
template <int C>
__global__ void __launch_bounds__(256, kLnFwdPerSm) ln_fwd_kernel(const uint16_t* __restrict__ z,
                                                                  const float* __restrict__ gamma,
                                                                  const float* __restrict__ beta,
                                                                  uint16_t* __restrict__ x,
                                                                  float* __restrict__ mean_out,
                                                                  float* __restrict__ rstd_out, size_t M) {
  constexpr int kPer = C / 32;
  constexpr int kRows = C <= 128 ? 8 : 4;  // rows a warp has in flight
  const int lane = threadIdx.x & 31;
  const int c0 = lane * kPer;
  float gm[kPer], bt[kPer];
  ld_f32<kPer>(gamma + c0, gm);
  ld_f32<kPer>(beta + c0, bt);
  const size_t warps = static_cast<size_t>(gridDim.x) * (blockDim.x / 32);
  for (size_t m0 = static_cast<size_t>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32; m0 < M;
       m0 += kRows * warps) {
    // the loads of all kRows rows in flight before the first reduction
    Packed<kPer> zr[kRows];
#pragma unroll
    for (int r = 0; r < kRows; ++r)
      if (m0 + r * warps < M) ld_packed<kPer>(z + (m0 + r * warps) * C + c0, zr[r]);
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      const size_t m = m0 + r * warps;
      if (m >= M) break;  // the same m in every lane
      float v[kPer];
      unpack<kPer>(zr[r], v);
      float s = 0.f;
#pragma unroll
      for (int e = 0; e < kPer; ++e) s += v[e];
      const float mean = warp_sum(s) * (1.f / C);
      float ss = 0.f;
#pragma unroll
      for (int e = 0; e < kPer; ++e) ss += (v[e] - mean) * (v[e] - mean);
      const float rstd = rsqrtf(warp_sum(ss) * (1.f / C) + 1e-5f);
      float o[kPer];
#pragma unroll
      for (int e = 0; e < kPer; ++e) o[e] = (v[e] - mean) * rstd * gm[e] + bt[e];
      st_bf16<kPer>(x + m * C + c0, o);
      if (lane == 0) {
        mean_out[m] = mean;
        rstd_out[m] = rstd;
      }
    }
  }
}

// One warp per pair: dz = rstd (g - mean(g) - xhat mean(g xhat)), g = dx gamma,
// dx BF16.  The warp also accumulates dgamma = sum dx xhat and dbeta = sum dx
// over its pairs (fixed grid-stride assignment, ascending); the block adds
// its 8 warps' sums in warp order and writes one partial row per block.  Lane
// l holds the C / 32 consecutive features from l C / 32; the loads of
// several pairs are in flight together.
template <int C>
__global__ void __launch_bounds__(256, kLnBwdPerSm) ln_bwd_kernel(const uint16_t* __restrict__ z,
                                                                  const uint16_t* __restrict__ dx,
                                                                  const float* __restrict__ gamma,
                                                                  const float* __restrict__ mean_in,
                                                                  const float* __restrict__ rstd_in,
                                                                  uint16_t* __restrict__ dz,
                                                                  float* __restrict__ part_gamma,
                                                                  float* __restrict__ part_beta, size_t M) {
  constexpr int kPer = C / 32;
  constexpr int kRows = C <= 128 ? 4 : (C <= 192 ? 2 : 1);  // rows a warp has in flight
  __shared__ float red_g[8][C], red_b[8][C];
  const int lane = threadIdx.x & 31, warp = threadIdx.x / 32;
  const int c0 = lane * kPer;
  float gm[kPer];
  ld_f32<kPer>(gamma + c0, gm);
  const size_t warps = static_cast<size_t>(gridDim.x) * (blockDim.x / 32);
  float accg[kPer], accb[kPer];
#pragma unroll
  for (int e = 0; e < kPer; ++e) accg[e] = accb[e] = 0.f;
  for (size_t m0 = static_cast<size_t>(blockIdx.x) * 8 + warp; m0 < M; m0 += kRows * warps) {
    Packed<kPer> zr[kRows], dr[kRows];
    float mu[kRows], rs[kRows];
#pragma unroll
    for (int r = 0; r < kRows; ++r)
      if (m0 + r * warps < M) {
        const size_t m = m0 + r * warps;
        ld_packed<kPer>(z + m * C + c0, zr[r]);
        ld_packed<kPer>(dx + m * C + c0, dr[r]);
        mu[r] = mean_in[m];
        rs[r] = rstd_in[m];
      }
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      const size_t m = m0 + r * warps;
      if (m >= M) break;  // the same m in every lane
      const float mean = mu[r], rstd = rs[r];
      float xh[kPer], d[kPer], g[kPer];
      unpack<kPer>(zr[r], xh);
      unpack<kPer>(dr[r], d);
      float sg = 0.f, sgx = 0.f;
#pragma unroll
      for (int e = 0; e < kPer; ++e) {
        xh[e] = (xh[e] - mean) * rstd;
        accg[e] += d[e] * xh[e];
        accb[e] += d[e];
        g[e] = d[e] * gm[e];
        sg += g[e];
        sgx += g[e] * xh[e];
      }
      const float a = warp_sum(sg) * (1.f / C), bb = warp_sum(sgx) * (1.f / C);
      float o[kPer];
#pragma unroll
      for (int e = 0; e < kPer; ++e) o[e] = rstd * (g[e] - a - xh[e] * bb);
      st_bf16<kPer>(dz + m * C + c0, o);
    }
  }
#pragma unroll
  for (int e = 0; e < kPer; ++e) {
    red_g[warp][c0 + e] = accg[e];
    red_b[warp][c0 + e] = accb[e];
  }
  __syncthreads();
  for (int c = threadIdx.x; c < C; c += blockDim.x) {
    float sg = 0.f, sb = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      sg += red_g[w][c];
      sb += red_b[w][c];
    }
    part_gamma[static_cast<size_t>(blockIdx.x) * C + c] = sg;
    part_beta[static_cast<size_t>(blockIdx.x) * C + c] = sb;
  }
}

// One warp per output column (columns 0 .. C-1: dgamma from pg, C .. 2C-1:
// dbeta from pb): lane l adds rows l, l + 32, ... in ascending order, then a
// fixed butterfly adds the 32 lane sums.
__global__ void __launch_bounds__(256) column_sum_kernel(const float* __restrict__ pg, const float* __restrict__ pb,
                                                         int rows, int C, float* __restrict__ dgamma,
                                                         float* __restrict__ dbeta) {
  const int col = blockIdx.x * 8 + threadIdx.x / 32, lane = threadIdx.x & 31;
  if (col >= 2 * C) return;
  const float* part = col < C ? pg : pb;
  const int c = col < C ? col : col - C;
  float s = 0.f;
  for (int r = lane; r < rows; r += 32) s += part[static_cast<size_t>(r) * C + c];
  s = warp_sum(s);
  if (lane == 0) (col < C ? dgamma : dbeta)[c] = s;
}

template <int C>
cudaError_t ln_fwd_launch(size_t M, const void* z, const float* g, const float* b, void* x, float* mean,
                          float* rstd, cudaStream_t s) {
  ln_fwd_kernel<C><<<kLnFwdBlocks, 256, 0, s>>>(static_cast<const uint16_t*>(z), g, b, static_cast<uint16_t*>(x),
                                             mean, rstd, M);
  return cudaGetLastError();
}
template <int C>
cudaError_t ln_bwd_launch(size_t M, const void* z, const void* dx, const float* g, const float* mean,
                          const float* rstd, void* dz, float* pg, float* pb, cudaStream_t s) {
  ln_bwd_kernel<C><<<kLnBlocks, 256, 0, s>>>(static_cast<const uint16_t*>(z), static_cast<const uint16_t*>(dx), g,
                                             mean, rstd,
                                             static_cast<uint16_t*>(dz), pg, pb, M);
  return cudaGetLastError();
}

// x = LayerNorm(z) over rows of C features (BF16 in and out), mean and rstd saved.
inline cudaError_t ln_rows_fwd(size_t M, int C, const void* z, const float* g, const float* b, void* x, float* mean,
                               float* rstd, cudaStream_t s) {
  switch (C) {
    case 32: return ln_fwd_launch<32>(M, z, g, b, x, mean, rstd, s);
    case 64: return ln_fwd_launch<64>(M, z, g, b, x, mean, rstd, s);
    case 96: return ln_fwd_launch<96>(M, z, g, b, x, mean, rstd, s);
    case 128: return ln_fwd_launch<128>(M, z, g, b, x, mean, rstd, s);
    case 160: return ln_fwd_launch<160>(M, z, g, b, x, mean, rstd, s);
    case 192: return ln_fwd_launch<192>(M, z, g, b, x, mean, rstd, s);
    case 224: return ln_fwd_launch<224>(M, z, g, b, x, mean, rstd, s);
    case 256: return ln_fwd_launch<256>(M, z, g, b, x, mean, rstd, s);
  }
  return cudaErrorInvalidValue;
}
// dz (BF16) from dx (BF16); kLnBlocks partial rows of dgamma and dbeta.
inline cudaError_t ln_rows_bwd(size_t M, int C, const void* z, const void* dx, const float* g, const float* mean,
                               const float* rstd, void* dz, float* pg, float* pb, cudaStream_t s) {
  switch (C) {
    case 32: return ln_bwd_launch<32>(M, z, dx, g, mean, rstd, dz, pg, pb, s);
    case 64: return ln_bwd_launch<64>(M, z, dx, g, mean, rstd, dz, pg, pb, s);
    case 96: return ln_bwd_launch<96>(M, z, dx, g, mean, rstd, dz, pg, pb, s);
    case 128: return ln_bwd_launch<128>(M, z, dx, g, mean, rstd, dz, pg, pb, s);
    case 160: return ln_bwd_launch<160>(M, z, dx, g, mean, rstd, dz, pg, pb, s);
    case 192: return ln_bwd_launch<192>(M, z, dx, g, mean, rstd, dz, pg, pb, s);
    case 224: return ln_bwd_launch<224>(M, z, dx, g, mean, rstd, dz, pg, pb, s);
    case 256: return ln_bwd_launch<256>(M, z, dx, g, mean, rstd, dz, pg, pb, s);
  }
  return cudaErrorInvalidValue;
}

// dgamma / dbeta [C] from `rows` partial rows each, fixed order.
inline cudaError_t column_sums(const float* pg, const float* pb, int rows, int C, float* dgamma, float* dbeta,
                               cudaStream_t s) {
  column_sum_kernel<<<static_cast<unsigned>((2 * C + 7) / 8), 256, 0, s>>>(pg, pb, rows, C, dgamma, dbeta);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- GEMMs
// The library's tensor-core GEMM (gemm.cu) as one traced launch of kind
// `kind`: row-major C[M, N] = op(A) op(B), BF16 operands, FP32 accumulation,
// C BF16 or FP32; `gemm_ws` (kGemmWorkspace bytes of the caller's workspace)
// holds the split-K partials of the weight gradients.
inline triattn_status gemm_traced(int kind, void* gemm_ws, cudaStream_t s, bool ta, bool tb, int M, int N, int K,
                                  const void* A, int lda, const void* B, int ldb, void* C, int ldc, bool c_f32,
                                  int batch = 1, long long strideA = 0, long long strideB = 0,
                                  long long strideC = 0) {
  const WaitCtl wc = current_wait_ctl();
  const cudaError_t e = trace_call(kind, s, [&] {
    return launch_gemm(ta, tb, M, N, K, A, lda, B, ldb, C, ldc, c_f32, batch, strideA, strideB, strideC, gemm_ws,
                       kGemmWorkspace, wc, s);
  });
  return e == cudaSuccess ? TRIATTN_OK : TRIATTN_ERR_CUDA;
}

}  // namespace pairops
}  // namespace
}  // namespace triattn
