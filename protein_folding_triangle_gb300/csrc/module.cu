// Triangle-attention module around the attention core ("TurboPairFormer",
// Figure 6): LayerNorm of the pair tensor, the projections into q, k, v and
// the pair bias, the core, and the output projection, forward and backward.
//
//   x = LayerNorm(Z; gamma, beta)            Z, x   [M = B*N*N, C]
//   P = x W_in                               W_in   [C, F], F = 3HD + H
//   q, k, v  = heads of P[:, 0:HD], P[:, HD:2HD], P[:, 2HD:3HD]  -> [B, N, H, N, D]
//   bias[b, h, q, k] = P[(b, q, k), 3HD + h]                       -> [B, H, N, N]
//   o = core(q, k, v, bias, mask)            o      [B, N, H, N, D]
//   out = o_flat W_o                         o_flat [M, HD], W_o [HD, C]
//
// The projections are the library's tensor-core GEMM (gemm.cu: BF16 in, FP32
// accumulate; the weight gradients split along the pair axis into FP32
// partials added in fixed order); the LayerNorm, the head scatter / gather
// between the pair layout and the core's layout, and the column sums of the
// LayerNorm parameter gradients are the kernels below.  Every reduction has
// a fixed order, so results are bitwise reproducible.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "kernels.cuh"
#include "pairops.cuh"
#include "triattn.h"

namespace triattn {
namespace {

using namespace pairops;

// bias[b, h, q, k] = pairs[(b, q, k), off + h]   (to_pairs = false)
// pairs[(b, q, k), off + h] = bias[b, h, q, k]   (to_pairs = true)
// One thread per pair: its H values share one sector of the pair row, and
// consecutive threads touch consecutive elements of every bias plane.
__global__ void __launch_bounds__(256) bias_plane_kernel(uint16_t* __restrict__ pairs, int ld, int off,
                                                         uint16_t* __restrict__ bias, int NN, int H, size_t M,
                                                         bool to_pairs) {
  const size_t m = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (m >= M) return;
  const size_t b = m / NN, qk = m % NN;
  uint16_t* row = pairs + m * ld;
  for (int h = 0; h < H; ++h) {
    uint16_t* pb = bias + (b * H + h) * NN + qk;
    if (to_pairs) row[off + h] = *pb;
    else *pb = row[off + h];
  }
  // the row's padding columns [off + H, ld) enter the backward GEMMs (times
  // zero weights): they must hold zeros, not whatever the workspace held
  if (to_pairs)
    for (int c = off + H; c < ld; ++c) row[c] = 0;
}

// dst [rows, ldd] = src [rows, cols] with zero columns [cols, ldd) (the
// projection matrix padded to a row length that is a multiple of 8).
__global__ void __launch_bounds__(256) pad_columns_kernel(const uint16_t* __restrict__ src, int cols,
                                                          uint16_t* __restrict__ dst, int ldd, int rows) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= rows * ldd) return;
  const int r = t / ldd, c = t % ldd;
  dst[t] = c < cols ? src[static_cast<size_t>(r) * cols + c] : static_cast<uint16_t>(0);
}

// ---------------------------------------------------------------- layouts
size_t rup(size_t x) { return (x + 255) / 256 * 256; }

struct ModDims {
  size_t M, F, Fp, HD, C, H, D, B, N;
};
ModDims dims_of(const triattn_module_shape* s) {
  ModDims d;
  d.B = s->B;
  d.N = s->N;
  d.C = s->C;
  d.H = s->H;
  d.D = s->D;
  d.HD = d.H * d.D;
  d.M = d.B * d.N * d.N;
  d.F = 3 * d.HD + d.H;
  d.Fp = (d.F + 7) / 8 * 8;  // row stride of P / dP: 16-byte aligned rows
  return d;
}

// Saved between forward and backward (the caller's "context" buffer).
// Two data flows.  With N a multiple of 32 ("heads" flow) the projection
// GEMM's epilogue writes q, k, v straight into the core's layout and the bias
// planes, and the dO GEMM writes dO in the core's layout, so the core reads
// contiguous tiles; otherwise q, k, v stay in P's pair rows and dO in
// d_oflat's, read there through the strided entry points.  Either way the
// core writes o and its residual into pair rows of H*D features and dq, dk,
// dv into dP's pair rows.
bool heads_flow(const ModDims& d) { return d.N % 32 == 0; }

struct CtxLayout {
  size_t x, mean, rstd, p, bias, lse, resid, oflat, total;  // p: P, or q | k | v in the core's layout
};
CtxLayout ctx_layout(const ModDims& d) {
  CtxLayout c;
  size_t o = 0;
  const size_t act = d.B * d.N * d.H * d.N * d.D * 2;  // one [B, N, H, N, D] bf16 tensor
  c.x = o;     o += rup(d.M * d.C * 2);
  c.mean = o;  o += rup(d.M * 4);
  c.rstd = o;  o += rup(d.M * 4);
  c.p = o;     o += rup(heads_flow(d) ? 3 * act : d.M * d.Fp * 2);
  c.bias = o;  o += rup(d.B * d.H * d.N * d.N * 2);
  c.lse = o;   o += rup(d.B * d.N * d.H * d.N * 4);
  c.resid = o; o += rup(d.M * d.HD * 2);
  c.oflat = o; o += rup(d.M * d.HD * 2);
  c.total = o;
  return c;
}
// q, k, v (and dq, dk, dv) in pair rows of ld = Fp; o, its residual and dO in
// pair rows of ld = H*D
triattn_layout pair_layout(const ModDims& d, size_t ld) {
  return triattn_layout{static_cast<long long>(d.N * ld), static_cast<long long>(d.D), static_cast<long long>(ld)};
}
triattn_layout core_layout(const ModDims& d) {
  return triattn_layout{static_cast<long long>(d.H * d.N * d.D), static_cast<long long>(d.N * d.D),
                        static_cast<long long>(d.D)};
}

// Scratch of one forward or backward call.
struct WsLayout2 {
  size_t gemm, w_in_pad, dw_in_pad, p, doflat, dbias, dx, pg, pb, core, total;
};
WsLayout2 ws_layout2(const ModDims& d, const triattn_shape& core) {
  WsLayout2 w;
  size_t o = 0;
  w.gemm = o;   o += rup(kGemmWorkspace);
  w.w_in_pad = o;  o += rup(d.C * d.Fp * 2);   // W_in with zero columns up to Fp
  w.dw_in_pad = o; o += rup(d.C * d.Fp * 4);   // dW_in, Fp wide
  w.p = o;      o += rup(d.M * d.Fp * 2);  // dP (backward)
  w.doflat = o; o += rup(d.M * d.HD * 2);  // d_oflat, or dO in the core's layout (same size)
  w.dbias = o;  o += rup(d.B * d.H * d.N * d.N * 2);
  w.dx = o;     o += rup(d.M * d.C * 2);
  w.pg = o;     o += rup(static_cast<size_t>(kLnBlocks) * d.C * 4);
  w.pb = o;     o += rup(static_cast<size_t>(kLnBlocks) * d.C * 4);
  // the core's forward and backward workspaces (one at a time)
  w.core = o;   o += rup(std::max(triattn_bwd_workspace_bytes(&core), triattn_fwd_workspace_bytes(&core)));
  w.total = o;
  return w;
}

triattn_status check_module(const triattn_module_shape* s, triattn_shape* core) {
  if (s == nullptr || s->flags != 0 || s->B < 1 || s->N < 1 || s->C < 1 || s->H < 1 || s->D < 1)
    return TRIATTN_ERR_INVALID_ARG;
  if (!ln_width_ok(s->C) || s->H > 64) return TRIATTN_ERR_UNSUPPORTED;
  // the layout kernels move 16-byte groups of pair rows: N a multiple of 8,
  // up to 4096 tokens
  if (s->N % 8 != 0 || s->N > 4096) return TRIATTN_ERR_UNSUPPORTED;
  // the projection GEMMs take the pair count as a 32-bit row count
  if (static_cast<size_t>(s->B) * s->N * s->N > 0x7fffffffull) return TRIATTN_ERR_UNSUPPORTED;
  *core = triattn_shape{s->B, s->N, s->N, s->H, s->D, 0u};
  if (triattn_bwd_workspace_bytes(core) == 0) return TRIATTN_ERR_UNSUPPORTED;  // the core's own shape rules
  return TRIATTN_OK;
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

unsigned blocks_for(size_t n) { return static_cast<unsigned>((n + 255) / 256); }

cudaError_t bias_planes(const ModDims& d, uint16_t* pairs, int ld, int off, uint16_t* bias, bool to_pairs,
                        cudaStream_t s) {
  return trace_call(kKModLayout, s, [&] {
    bias_plane_kernel<<<blocks_for(d.M), 256, 0, s>>>(pairs, ld, off, bias, static_cast<int>(d.N * d.N),
                                                             static_cast<int>(d.H), d.M, to_pairs);
    return cudaGetLastError();
  });
}

cudaError_t pad_w_in(const ModDims& d, const void* w_in, uint16_t* w_in_pad, cudaStream_t s) {
  return trace_call(kKModLayout, s, [&] {
    pad_columns_kernel<<<blocks_for(d.C * d.Fp), 256, 0, s>>>(static_cast<const uint16_t*>(w_in),
                                                              static_cast<int>(d.F), w_in_pad, static_cast<int>(d.Fp),
                                                              static_cast<int>(d.C));
    return cudaGetLastError();
  });
}

}  // namespace
}  // namespace triattn

using namespace triattn;

extern "C" {

size_t triattn_module_ctx_bytes(const triattn_module_shape* shape) {
  triattn_shape core;
  if (check_module(shape, &core) != TRIATTN_OK) return 0;
  return ctx_layout(dims_of(shape)).total;
}

size_t triattn_module_workspace_bytes(const triattn_module_shape* shape) {
  triattn_shape core;
  if (check_module(shape, &core) != TRIATTN_OK) return 0;
  return ws_layout2(dims_of(shape), core).total;
}

triattn_status tri_attn_module_fwd(const triattn_module_shape* shape, const void* z, const void* mask,
                                   const float* ln_w, const float* ln_b, const void* w_in, const void* w_o, void* out,
                                   void* ctx, void* workspace, size_t workspace_bytes, void* stream) {
  triattn_shape core;
  triattn_status st = check_module(shape, &core);
  if (st != TRIATTN_OK) return st;
  const void* req[] = {z, ln_w, ln_b, w_in, w_o, out, ctx};
  for (const void* p : req)
    if (p == nullptr || !al16(p)) return TRIATTN_ERR_INVALID_ARG;
  if (mask != nullptr && !al16(mask)) return TRIATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ctx) & 255u) != 0) return TRIATTN_ERR_INVALID_ARG;
  const ModDims d = dims_of(shape);
  const CtxLayout c = ctx_layout(d);
  const WsLayout2 w = ws_layout2(d, core);
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || workspace_bytes < w.total)
    return TRIATTN_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* cx = static_cast<uint8_t*>(ctx);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void* const gws = ws + w.gemm;
  const int M = static_cast<int>(d.M), C = static_cast<int>(d.C), HD = static_cast<int>(d.HD),
            Fp = static_cast<int>(d.Fp);
  float* mean = reinterpret_cast<float*>(cx + c.mean);
  float* rstd = reinterpret_cast<float*>(cx + c.rstd);
  uint16_t* P = reinterpret_cast<uint16_t*>(cx + c.p);
  // x = LayerNorm(z)
  if (trace_call(kKModLnFwd, s, [&] { return ln_rows_fwd(d.M, C, z, ln_w, ln_b, cx + c.x, mean, rstd, s); }) != cudaSuccess)
    return TRIATTN_ERR_CUDA;
  // P = x W_in
  // (through W_in padded to Fp columns: the GEMM's TMA tiles need rows whose
  // length is a multiple of 8 elements)
  uint16_t* w_in_pad = reinterpret_cast<uint16_t*>(ws + w.w_in_pad);
  if (pad_w_in(d, w_in, w_in_pad, s) != cudaSuccess) return TRIATTN_ERR_CUDA;
  const triattn_layout lo = pair_layout(d, d.HD);
  if (heads_flow(d)) {
    // q, k, v into the core's layout and the bias planes, from the GEMM's epilogue
    const int Ni = static_cast<int>(d.N), Hi = static_cast<int>(d.H), Di = static_cast<int>(d.D);
    if (trace_call(kKModGemm, s, [&] {
          return launch_gemm_heads(false, M, Fp, C, cx + c.x, C, w_in_pad, Fp, 3, Hi, Di, Ni, static_cast<int>(d.B),
                                   P, cx + c.bias, Hi, current_wait_ctl(), s);
        }) != cudaSuccess)
      return TRIATTN_ERR_CUDA;
    const size_t act = d.B * d.N * d.H * d.N * d.D;
    const triattn_layout lq = core_layout(d);
    st = tri_attn_fwd_strided(&core, P, P + act, P + 2 * act, &lq, cx + c.bias, mask, cx + c.oflat,
                              reinterpret_cast<float*>(cx + c.lse), cx + c.resid, &lo, ws + w.core, w.total - w.core,
                              stream);
  } else {
    if (gemm_traced(kKModGemm, gws, s, false, false, M, Fp, C, cx + c.x, C, w_in_pad, Fp, P, Fp, false) !=
        TRIATTN_OK)
      return TRIATTN_ERR_CUDA;
    if (bias_planes(d, P, Fp, 3 * HD, reinterpret_cast<uint16_t*>(cx + c.bias), false, s) != cudaSuccess)
      return TRIATTN_ERR_CUDA;
    // the core reads q, k, v from P's pair rows
    const triattn_layout lq = pair_layout(d, d.Fp);
    st = tri_attn_fwd_strided(&core, P, P + HD, P + 2 * HD, &lq, cx + c.bias, mask, cx + c.oflat,
                              reinterpret_cast<float*>(cx + c.lse), cx + c.resid, &lo, ws + w.core, w.total - w.core,
                              stream);
  }
  if (st != TRIATTN_OK) return st;
  // out = o_flat W_o (the core wrote o into o_flat's pair rows)
  return gemm_traced(kKModGemm, gws, s, false, false, M, C, HD, cx + c.oflat, HD, w_o, C, out, C, false);
}

triattn_status tri_attn_module_bwd(const triattn_module_shape* shape, const void* z, const void* mask,
                                   const float* ln_w, const void* w_in, const void* w_o, const void* ctx,
                                   const void* d_out, void* dz, float* d_ln_w, float* d_ln_b, float* d_w_in,
                                   float* d_w_o, void* workspace, size_t workspace_bytes, void* stream) {
  triattn_shape core;
  triattn_status st = check_module(shape, &core);
  if (st != TRIATTN_OK) return st;
  const void* req[] = {z, ln_w, w_in, w_o, ctx, d_out, dz, d_ln_w, d_ln_b, d_w_in, d_w_o};
  for (const void* p : req)
    if (p == nullptr || !al16(p)) return TRIATTN_ERR_INVALID_ARG;
  if (mask != nullptr && !al16(mask)) return TRIATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ctx) & 255u) != 0) return TRIATTN_ERR_INVALID_ARG;
  const ModDims d = dims_of(shape);
  const CtxLayout c = ctx_layout(d);
  const WsLayout2 w = ws_layout2(d, core);
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || workspace_bytes < w.total)
    return TRIATTN_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const uint8_t* cx = static_cast<const uint8_t*>(ctx);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void* const gws = ws + w.gemm;
  const int M = static_cast<int>(d.M), C = static_cast<int>(d.C), HD = static_cast<int>(d.HD),
            Fp = static_cast<int>(d.Fp);
  // out = o_flat W_o:  dW_o = o_flat^T d_out,  d_oflat = d_out W_o^T (in the
  // heads flow straight into dO in the core's layout)
  if (gemm_traced(kKModGemm, gws, s, true, false, HD, C, M, cx + c.oflat, HD, d_out, C, d_w_o, C, true) != TRIATTN_OK)
    return TRIATTN_ERR_CUDA;
  const bool hf = heads_flow(d);
  if (hf) {
    const int Ni = static_cast<int>(d.N), Hi = static_cast<int>(d.H), Di = static_cast<int>(d.D);
    if (trace_call(kKModGemm, s, [&] {
          return launch_gemm_heads(true, M, HD, C, d_out, C, w_o, C, 1, Hi, Di, Ni, static_cast<int>(d.B),
                                   ws + w.doflat, nullptr, 0, current_wait_ctl(), s);
        }) != cudaSuccess)
      return TRIATTN_ERR_CUDA;
  } else if (gemm_traced(kKModGemm, gws, s, false, true, M, HD, C, d_out, C, w_o, C, ws + w.doflat, HD, false) !=
             TRIATTN_OK) {
    return TRIATTN_ERR_CUDA;
  }
  // the attention core, dq, dk, dv written into dP = [dq | dk | dv | dbias]
  // where they lie in the pair layout
  const uint16_t* P = reinterpret_cast<const uint16_t*>(cx + c.p);
  uint16_t* dP = reinterpret_cast<uint16_t*>(ws + w.p);
  const size_t act = d.B * d.N * d.H * d.N * d.D;
  const triattn_layout lq = hf ? core_layout(d) : pair_layout(d, d.Fp), lo = pair_layout(d, d.HD),
                       ldo = hf ? core_layout(d) : pair_layout(d, d.HD), lg = pair_layout(d, d.Fp);
  const size_t step = hf ? act : static_cast<size_t>(HD);
  st = tri_attn_bwd_strided(&core, P, P + step, P + 2 * step, &lq, cx + c.bias, mask, cx + c.oflat, cx + c.resid,
                            &lo, reinterpret_cast<const float*>(cx + c.lse), ws + w.doflat, &ldo, dP, dP + HD,
                            dP + 2 * HD, &lg, ws + w.dbias, ws + w.core, w.total - w.core, stream);
  if (st != TRIATTN_OK) return st;
  if (bias_planes(d, dP, Fp, 3 * HD, reinterpret_cast<uint16_t*>(ws + w.dbias), true, s) != cudaSuccess)
    return TRIATTN_ERR_CUDA;
  // P = x W_in:  dW_in = x^T dP,  dx = dP W_in^T (BF16), both Fp wide (dP's
  // padding columns are zero, so are W_in's); dW_in's first F columns copied out
  uint16_t* w_in_pad = reinterpret_cast<uint16_t*>(ws + w.w_in_pad);
  float* dw_in_pad = reinterpret_cast<float*>(ws + w.dw_in_pad);
  if (pad_w_in(d, w_in, w_in_pad, s) != cudaSuccess) return TRIATTN_ERR_CUDA;
  if (gemm_traced(kKModGemm, gws, s, true, false, C, Fp, M, cx + c.x, C, dP, Fp, dw_in_pad, Fp, true) !=
          TRIATTN_OK ||
      gemm_traced(kKModGemm, gws, s, false, true, M, C, Fp, dP, Fp, w_in_pad, Fp, ws + w.dx, C, false) !=
          TRIATTN_OK)
    return TRIATTN_ERR_CUDA;
  if (trace_call(kKModLayout, s, [&] {
        return cudaMemcpy2DAsync(d_w_in, d.F * 4, dw_in_pad, d.Fp * 4, d.F * 4, d.C, cudaMemcpyDeviceToDevice, s);
      }) != cudaSuccess)
    return TRIATTN_ERR_CUDA;
  // x = LayerNorm(z)
  float* pg = reinterpret_cast<float*>(ws + w.pg);
  float* pb = reinterpret_cast<float*>(ws + w.pb);
  if (trace_call(kKModLnBwd, s, [&] {
        return ln_rows_bwd(d.M, C, z, ws + w.dx, ln_w,
                          reinterpret_cast<const float*>(cx + c.mean), reinterpret_cast<const float*>(cx + c.rstd),
                          dz, pg, pb, s);
      }) != cudaSuccess)
    return TRIATTN_ERR_CUDA;
  const cudaError_t e = trace_call(kKModColSum, s, [&] {
    return column_sums(pg, pb, kLnBlocks, C, d_ln_w, d_ln_b, s);
  });
  return e == cudaSuccess ? TRIATTN_OK : TRIATTN_ERR_CUDA;
}

}  // extern "C"
