// Backward kernels of triangular attention on sm_103a.
//
// "TurboPairFormer: Fast and Stable Protein Folding Model Training with an
// Optimized Triangle Attention Kernel":
//   Figure 7(b)  preprocess: compensated row correction delta in FP32;
//   Figure 2, Figure 7(c)-(d), Table 11 row "Key tile (ours)": one thread
//                block owns a key tile in each slice of an outer group,
//                visits every query tile, recomputes S, P, dP and dS once,
//                keeps dK and dV on chip, writes one dQ partial per key tile
//                and one dbias partial per outer group, each single-writer;
//   Figure 11(a) ("materialized partials"): separate kernels add the
//                partials in ascending index order in FP32.
#include "kernels.cuh"

namespace triattn {

namespace {

constexpr int BM = kTileQ;   // query rows per tile
constexpr int BN = kTileK;   // keys per CTA (TMEM lanes of dK / dV)
constexpr int G = kGroupBwd; // outer slices per CTA
constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------- preprocess
// delta[row] = sum_d dO[row,d] * (O[row,d] + E[row,d])  (E omitted when null).
template <int D>
__global__ void __launch_bounds__(256) preprocess_kernel(const uint16_t* __restrict__ dO,
                                                         const uint16_t* __restrict__ o,
                                                         const uint16_t* __restrict__ e,
                                                         float* __restrict__ delta, size_t rows) {
  const size_t row = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (row >= rows) return;
  const uint4* gp = reinterpret_cast<const uint4*>(dO + row * D);
  const uint4* op = reinterpret_cast<const uint4*>(o + row * D);
  const uint4* ep = e ? reinterpret_cast<const uint4*>(e + row * D) : nullptr;
  float acc = 0.f;
#pragma unroll
  for (int v = 0; v < D / 8; ++v) {
    const uint4 gw = __ldg(gp + v), ow = __ldg(op + v);
    uint4 ew = make_uint4(0, 0, 0, 0);
    if (ep) ew = __ldg(ep + v);
    const uint32_t g4[4] = {gw.x, gw.y, gw.z, gw.w}, o4[4] = {ow.x, ow.y, ow.z, ow.w},
                   e4[4] = {ew.x, ew.y, ew.z, ew.w};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      acc = fmaf(bf16lo_to_f32(g4[u]), bf16lo_to_f32(o4[u]) + bf16lo_to_f32(e4[u]), acc);
      acc = fmaf(bf16hi_to_f32(g4[u]), bf16hi_to_f32(o4[u]) + bf16hi_to_f32(e4[u]), acc);
    }
  }
  delta[row] = acc;
}

// ---------------------------------------------------------------- main kernel
//
// Thread roles (18 warps):
//   warp 0       TMA producer: K, V of the G slices once; per query tile one
//                bias tile; per (query tile, slice) the Q and dO tiles.
//   warp 1       TMEM owner and tcgen05 MMA issuer (converged warp, one
//                elected lane issues; descriptors are precomputed).
//   warps 2-17   four elementwise warpgroups.  Each covers all 128 TMEM lanes
//                (thread = query row for S / dP / dQ, key row for dK / dV);
//                warpgroup w handles key columns [32w, 32w + 32).
//
// Per step s = (query tile i, slice g), two elementwise phases:
//   P-phase   P = 2^(S log2e/sqrt(D) + (bias + mask) log2e - lse log2e)
//             -> BF16 P into 128-byte-swizzled shared memory (FP32 P stays
//             in registers); the S columns of TMEM are then free.
//   dS-phase  dS = P (dP - delta); dbias accumulator += dS (FP32 registers);
//             BF16 dS into shared memory.
// MMA order: S(s+1) and dV_g += P^T dO are issued when the P-phase of s ends
// (they overlap the dS-phase); dK_g += dS^T Q and dP(s+1) when the dS-phase
// ends; the dQ tile dS K goes into the S columns as soon as the warps have
// loaded S(s+1) into registers, so it runs under the P-phase of s+1, which
// then reads it (and only then writes P(s+1) to shared memory).  dK is scaled
// by 1/sqrt(D) when it leaves TMEM, the dQ tile when it is read.  After slice
// G-1 of a query tile the FP32 dbias partial of the outer group is written
// once.
template <int D>
struct BwdSmem {
  static constexpr int kTile = BM * D * 2;              // 128 rows x D bf16
  static constexpr int kP = 0;                          // P  [128 q][128 k] bf16, SW128, 2 blocks
  static constexpr int kDS = kP + BM * BN * 2;          // dS [128 q][128 k] bf16, SW128, 2 blocks
  static constexpr int kBias = kDS + BM * BN * 2;       // 2 stages x [128 q][128 k] bf16
  static constexpr int kK = kBias + 2 * BM * BN * 2;    // G K tiles (stationary)
  static constexpr int kV = kK + G * kTile;             // G V tiles (stationary)
  static constexpr int kQ = kV + G * kTile;             // 2 stages of Q tiles
  static constexpr int kDO = kQ + 2 * kTile;            // 2 stages of dO tiles
  static constexpr int kMask = kDO + 2 * kTile;         // G x 128 fp32 (base-2 scaled key mask)
  static constexpr int kFlag = kMask + G * BN * 4;      // G x 16 bytes: 8-key chunk has a nonzero mask
  static constexpr int kBar = kFlag + G * 16;
  static constexpr int kBytes = kBar + 256;
  static_assert(kBytes <= 232448, "shared memory budget");
};

constexpr int kNWG = 4;                // elementwise warpgroups
constexpr int kCols = BN / kNWG;       // key columns per warpgroup
constexpr int kEW = 128 * kNWG;        // elementwise threads
constexpr int kMainThreads = 64 + kEW;

struct BwdBars {
  uint64_t kv_full;
  uint64_t qdo_full[2], qdo_empty[2];
  uint64_t b_full[2], b_empty[2];
  uint64_t s_full, dp_full, s_cons, p_ready, ds_ready, dq_full;
  uint32_t tmem_slot;
  int abort;
};

template <int D>
__global__ void __launch_bounds__(kMainThreads, 1)
    bwd_main_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_bias, const uint16_t* __restrict__ mask,
                    const float* __restrict__ lse, const float* __restrict__ delta, uint16_t* __restrict__ dk,
                    uint16_t* __restrict__ dv, float* __restrict__ dq_part, float* __restrict__ dbias_part, int N_o,
                    int N, int H, WaitCtl wc) {
  using L = BwdSmem<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw;
  BwdBars* bars = reinterpret_cast<BwdBars*>(sm + L::kBar);
  volatile int* abort = &bars->abort;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int ktile = blockIdx.x;
  const int grp = blockIdx.y;
  const int o0 = grp * G;
  const int bh = blockIdx.z;
  const int b = bh / H;
  const int h = bh - b * H;
  const int JQ = (N + BM - 1) / BM;
  const int nsteps = JQ * G;

  // The swizzled tiles below need a 1024-byte aligned base.
  if ((smem_u32(sm) & 1023u) != 0) {
    if (tid == 0) atomicOr(wc.status, 2u);
    return;
  }

  // TMEM columns: dV_g at g*D, dK_g at 4D + g*D, S (128), dP (128); the dQ
  // tile (D columns) reuses the first S columns once S has been loaded.
  constexpr uint32_t kTS = 8 * D;
  constexpr uint32_t kTDP = kTS + 128;
  constexpr uint32_t kTDQ = kTS;
  static_assert(kTDP + 128 <= 512, "TMEM budget");

  if (tid == 0) {
    mbar_init(&bars->kv_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->qdo_full[i], 1);
      mbar_init(&bars->qdo_empty[i], 1);
      mbar_init(&bars->b_full[i], 1);
      mbar_init(&bars->b_empty[i], kEW);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->s_cons, kEW);
    mbar_init(&bars->p_ready, kEW);
    mbar_init(&bars->ds_ready, kEW);
    mbar_init(&bars->dq_full, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(&bars->tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      prefetch_tmap(&tm_do);
      prefetch_tmap(&tm_bias);
      mbar_expect_tx(&bars->kv_full, 2 * G * L::kTile);
      for (int g = 0; g < G; ++g) {
        const int boh = (b * N_o + o0 + g) * H + h;
        tma_load_3d(sm + L::kK + g * L::kTile, &tm_k, &bars->kv_full, 0, ktile * BN, boh);
        tma_load_3d(sm + L::kV + g * L::kTile, &tm_v, &bars->kv_full, 0, ktile * BN, boh);
      }
      for (int s = 0; s < nsteps && !*abort; ++s) {
        const int i = s / G, g = s % G;
        if (g == 0) {
          const int st = i & 1;
          if (!mbar_wait(&bars->b_empty[st], ((i >> 1) & 1) ^ 1, wc, abort)) break;
          mbar_expect_tx(&bars->b_full[st], BM * BN * 2);
          uint8_t* bdst = sm + L::kBias + st * (BM * BN * 2);
          tma_load_3d(bdst, &tm_bias, &bars->b_full[st], ktile * BN, i * BM, bh);
          tma_load_3d(bdst + BM * 128, &tm_bias, &bars->b_full[st], ktile * BN + 64, i * BM, bh);
        }
        const int st = s & 1;
        if (!mbar_wait(&bars->qdo_empty[st], ((s >> 1) & 1) ^ 1, wc, abort)) break;
        const int boh = (b * N_o + o0 + g) * H + h;
        mbar_expect_tx(&bars->qdo_full[st], 2 * L::kTile);
        tma_load_3d(sm + L::kQ + st * L::kTile, &tm_q, &bars->qdo_full[st], 0, i * BM, boh);
        tma_load_3d(sm + L::kDO + st * L::kTile, &tm_do, &bars->qdo_full[st], 0, i * BM, boh);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t kSwz = (D == 32) ? 4u : 6u;  // 64B / 32B swizzle for D-wide rows
    constexpr uint32_t kSbo = 8u * D * 2u;
    constexpr uint32_t idSS = idesc_bf16_f32(BM, BN, 0, 0);     // S, dP
    constexpr uint32_t idKV = idesc_bf16_f32(BN, D, 1, 1);      // dV, dK: A MN-major, B MN-major
    constexpr uint32_t idQ = idesc_bf16_f32(BM, D, 0, 1);       // dQ: A K-major, B MN-major
    constexpr uint32_t kTile16 = L::kTile >> 4;                 // tile size in descriptor units
    constexpr uint32_t kRowStep = (16 * D * 2) >> 4;            // 16 rows of a D-wide tile
    // base descriptors; per-MMA offsets are added to the start-address field
    const uint64_t dQb = smem_desc(smem_u32(sm + L::kQ), 16, kSbo, kSwz);
    const uint64_t dDOb = smem_desc(smem_u32(sm + L::kDO), 16, kSbo, kSwz);
    const uint64_t dKb = smem_desc(smem_u32(sm + L::kK), 16, kSbo, kSwz);
    const uint64_t dVb = smem_desc(smem_u32(sm + L::kV), 16, kSbo, kSwz);
    const uint64_t dPmn = smem_desc(smem_u32(sm + L::kP), 16384, 1024, 2);   // P as MN-major A
    const uint64_t dDSmn = smem_desc(smem_u32(sm + L::kDS), 16384, 1024, 2); // dS as MN-major A
    const uint64_t dDSk = smem_desc(smem_u32(sm + L::kDS), 16, 1024, 2);     // dS as K-major A
    auto issue_s = [&](int s) {  // S = Q K^T
      const uint64_t qd = dQb + (s & 1) * kTile16, kd = dKb + (s % G) * kTile16;
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) mma_ss(tmem + kTS, qd + 2 * kk, kd + 2 * kk, idSS, kk > 0 ? 1u : 0u);
        mma_commit(&bars->s_full);
      }
      __syncwarp();
    };
    auto issue_dp = [&](int s) {  // dP = dO V^T
      const uint64_t dod = dDOb + (s & 1) * kTile16, vd = dVb + (s % G) * kTile16;
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) mma_ss(tmem + kTDP, dod + 2 * kk, vd + 2 * kk, idSS, kk > 0 ? 1u : 0u);
        mma_commit(&bars->dp_full);
      }
      __syncwarp();
    };
    bool ok = __all_sync(0xffffffffu, mbar_wait(&bars->kv_full, 0, wc, abort)) &&
              __all_sync(0xffffffffu, mbar_wait(&bars->qdo_full[0], 0, wc, abort));
    if (ok) {
      tc_fence_after();
      issue_s(0);
      issue_dp(0);
    }
    for (int s = 0; s < nsteps && ok; ++s) {
      const int i = s / G, g = s % G, st = s & 1;
      const uint64_t qd = dQb + st * kTile16, dod = dDOb + st * kTile16, kd = dKb + g * kTile16;
      // P-phase of s done: S columns free (dQ of s-1 read), P in shared memory
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->p_ready, s & 1, wc, abort))) { ok = false; break; }
      tc_fence_after();
      if (s + 1 < nsteps) {
        if (!__all_sync(0xffffffffu, mbar_wait(&bars->qdo_full[(s + 1) & 1], ((s + 1) >> 1) & 1, wc, abort))) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_s(s + 1);
      }
      if (elect_one()) {
        const uint32_t tdv = tmem + g * D;
#pragma unroll
        for (int kk = 0; kk < BM / 16; ++kk)  // dV_g += P^T dO (A = P^T: keys contiguous, MN-major)
          mma_ss(tdv, dPmn + kk * 128, dod + kk * kRowStep, idKV, (i > 0 || kk > 0) ? 1u : 0u);
      }
      __syncwarp();
      // dS-phase of s done: dP columns free, dS in shared memory
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->ds_ready, s & 1, wc, abort))) { ok = false; break; }
      tc_fence_after();
      if (elect_one()) {
        const uint32_t tdk = tmem + 4 * D + g * D;
#pragma unroll
        for (int kk = 0; kk < BM / 16; ++kk)  // dK_g += dS^T Q
          mma_ss(tdk, dDSmn + kk * 128, qd + kk * kRowStep, idKV, (i > 0 || kk > 0) ? 1u : 0u);
      }
      __syncwarp();
      if (s + 1 < nsteps) {
        issue_dp(s + 1);
        // the dQ tile goes into the S columns once S(s+1) has been loaded
        if (!__all_sync(0xffffffffu, mbar_wait(&bars->s_cons, (s + 1) & 1, wc, abort))) { ok = false; break; }
        tc_fence_after();
      }
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)  // dQ tile = dS K (A = dS K-major, B = K MN-major)
          mma_ss(tmem + kTDQ, dDSk + (kk >> 2) * 1024 + (kk & 3) * 2, kd + kk * kRowStep, idQ, kk > 0 ? 1u : 0u);
        mma_commit(&bars->dq_full);        // covers every MMA issued so far
        mma_commit(&bars->qdo_empty[st]);
      }
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------ elementwise warpgroups
    const int ew = tid - 64;                  // 0..511
    const int quarter = warp & 3;             // TMEM lane quarter of this warp
    const int wg = (warp - 2) >> 2;           // key-column quarter handled by this warpgroup
    const int r = quarter * 32 + lane;        // TMEM lane: query row (S, dP, dQ) / key row (dK, dV)
    const int col0 = wg * kCols;
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const float scale_log2 = kLog2e * rsqrtf(static_cast<float>(D));
    const float inv_sqrt_d = rsqrtf(static_cast<float>(D));
    float* mask2 = reinterpret_cast<float*>(sm + L::kMask);
    uint8_t* mflag = sm + L::kFlag;
    uint8_t* sP = sm + L::kP;
    uint8_t* sDS = sm + L::kDS;

    // Base-2 key mask of the G slices (-inf past N) and, per 8-key chunk, a
    // flag telling whether any of its mask values is nonzero.  Staged before
    // any bounded wait so the two barriers below are always fully entered.
    for (int idx = ew; idx < G * BN; idx += kEW) {
      const int g = idx / BN, key = ktile * BN + (idx % BN);
      float mv = -INFINITY;
      if (key < N) {
        mv = 0.f;
        if (mask != nullptr)
          mv = __uint_as_float(static_cast<uint32_t>(__ldg(mask + (static_cast<size_t>(b) * N_o + o0 + g) * N + key))
                               << 16) *
               kLog2e;
      }
      mask2[idx] = mv;
    }
    named_bar_sync(1, kEW);
    if (ew < G * 16) {
      bool any = false;
#pragma unroll
      for (int e = 0; e < 8; ++e) any |= (mask2[ew * 8 + e] != 0.f);
      mflag[ew] = any ? 1 : 0;
    }
    named_bar_sync(1, kEW);

    // lse and delta of this thread's query row, loaded one step ahead; the
    // raw values are converted only when used.  Rows past N get P = 0.
    auto row_stats = [&](int s, float& l, float& dl) {
      const int i = s / G, g = s % G;
      const int q = min(i * BM + r, N - 1);
      const size_t row = (static_cast<size_t>((b * N_o + o0 + g) * H + h)) * N + q;
      l = ldg_f32_pinned(lse + row);
      dl = ldg_f32_pinned(delta + row);
    };
    // this key tile's dQ tile of step t (in the S columns of TMEM): D/4
    // columns per warpgroup, scaled by 1/sqrt(D), stored chunk-major per
    // 128-row tile: [J_K][slices][J_Q][D/4 float4 chunks][128 rows]
    auto store_dq_tile = [&](int t) {
      const int ti = t / G, tg = t % G;
      const size_t slice = static_cast<size_t>((b * N_o + o0 + tg) * H + h);
      const size_t nslices = static_cast<size_t>(gridDim.z) * N_o;
      float4* out = reinterpret_cast<float4*>(dq_part) +
                    ((static_cast<size_t>(ktile) * nslices + slice) * JQ + ti) * (BM * D / 4) + wg * (D / 16) * BM + r;
      if constexpr (D == 32) {
        uint32_t qr[8];
        tmem_ld8(tmem + lane_addr + kTDQ + 8 * wg, qr);
        tc_wait_ld();
#pragma unroll
        for (int v = 0; v < 2; ++v)
          out[v * BM] = make_float4(__uint_as_float(qr[4 * v]) * inv_sqrt_d, __uint_as_float(qr[4 * v + 1]) * inv_sqrt_d,
                                    __uint_as_float(qr[4 * v + 2]) * inv_sqrt_d,
                                    __uint_as_float(qr[4 * v + 3]) * inv_sqrt_d);
      } else {
        uint32_t qr[4];
        tmem_ld4(tmem + lane_addr + kTDQ + 4 * wg, qr);
        tc_wait_ld();
        out[0] = make_float4(__uint_as_float(qr[0]) * inv_sqrt_d, __uint_as_float(qr[1]) * inv_sqrt_d,
                             __uint_as_float(qr[2]) * inv_sqrt_d, __uint_as_float(qr[3]) * inv_sqrt_d);
      }
    };
    float lse_n, dl_n;
    row_stats(0, lse_n, dl_n);
    float2 dbacc[kCols / 2];  // dbias accumulators for this thread's key columns
#pragma unroll
    for (int k = 0; k < kCols / 2; ++k) dbacc[k] = make_float2(0.f, 0.f);
    const float2 c2 = make_float2(scale_log2, scale_log2);
    const float2 l2e2 = make_float2(kLog2e, kLog2e);
    bool ok = true;

    for (int s = 0; s < nsteps && ok; ++s) {
      const int i = s / G, g = s % G;
      const float lse_raw = lse_n, dl_raw = dl_n;
      if (s + 1 < nsteps) row_stats(s + 1, lse_n, dl_n);
      const bool row_ok = i * BM + r < N;
      const int bst = i & 1;
      if (g == 0 && !__all_sync(0xffffffffu, mbar_wait(&bars->b_full[bst], (i >> 1) & 1, wc, abort))) {
        ok = false;
        break;
      }
      const uint8_t* bias_s = sm + L::kBias + bst * (BM * BN * 2);
      const float* mk = mask2 + g * BN;

      // ---------------- P-phase
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->s_full, s & 1, wc, abort))) { ok = false; break; }
      tc_fence_after();
      float2 p[kCols / 2];
      {
        uint32_t sv[kCols];
        tmem_ld32(tmem + lane_addr + kTS + col0, sv);
        // fully masked rows (lse = -inf) and rows past N: P = 0
        const float lse2 = (row_ok && lse_raw != -INFINITY) ? lse_raw * kLog2e : INFINITY;
        tc_wait_ld_regs(sv);
        // S is in registers: the MMA warp may put the previous dQ tile there
        tc_fence_before();
        mbar_arrive(&bars->s_cons);
        const float2 nl2 = make_float2(-lse2, -lse2);
#pragma unroll
        for (int v = 0; v < kCols / 8; ++v) {  // 8 keys per 16-byte chunk
          const int cc = (col0 >> 3) + v;
          const uint32_t off = (cc >> 3) * (BM * 128) + sw128(r, cc & 7);
          const uint4 bw = *reinterpret_cast<const uint4*>(bias_s + off);
          const uint32_t bws[4] = {bw.x, bw.y, bw.z, bw.w};
          const bool masked = mflag[g * 16 + cc] != 0;
          float4 m0 = make_float4(0.f, 0.f, 0.f, 0.f), m1 = m0;
          if (masked) {
            m0 = *reinterpret_cast<const float4*>(mk + cc * 8);
            m1 = *reinterpret_cast<const float4*>(mk + cc * 8 + 4);
          }
          const float2 mm[4] = {make_float2(m0.x, m0.y), make_float2(m0.z, m0.w), make_float2(m1.x, m1.y),
                                make_float2(m1.z, m1.w)};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 s2 = make_float2(__uint_as_float(sv[v * 8 + 2 * e]), __uint_as_float(sv[v * 8 + 2 * e + 1]));
            const float2 b2 = make_float2(bf16lo_to_f32(bws[e]), bf16hi_to_f32(bws[e]));
            float2 t = ffma2(b2, l2e2, ffma2(s2, c2, nl2));
            if (masked) t = fadd2(t, mm[e]);
            p[v * 4 + e] = make_float2(ex2_approx(t.x), ex2_approx(t.y));
          }
        }
      }
      if (g == G - 1) mbar_arrive(&bars->b_empty[bst]);  // last read of this bias tile
      if (s > 0) {
        // the previous step's MMAs are complete: dQ tile in the S columns,
        // P and dS in shared memory no longer read
        if (!__all_sync(0xffffffffu, mbar_wait(&bars->dq_full, (s - 1) & 1, wc, abort))) { ok = false; break; }
        tc_fence_after();
        store_dq_tile(s - 1);
      }
#pragma unroll
      for (int v = 0; v < kCols / 8; ++v) {
        const int cc = (col0 >> 3) + v;
        const uint32_t off = (cc >> 3) * (BM * 128) + sw128(r, cc & 7);
        *reinterpret_cast<uint4*>(sP + off) =
            make_uint4(pack_bf16x2(p[4 * v].x, p[4 * v].y), pack_bf16x2(p[4 * v + 1].x, p[4 * v + 1].y),
                       pack_bf16x2(p[4 * v + 2].x, p[4 * v + 2].y), pack_bf16x2(p[4 * v + 3].x, p[4 * v + 3].y));
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bars->p_ready);

      // ---------------- dS-phase
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->dp_full, s & 1, wc, abort))) { ok = false; break; }
      tc_fence_after();
      {
        const float dl = row_ok ? dl_raw : 0.f;
        const float2 ndl2 = make_float2(-dl, -dl);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {  // 16 keys at a time
          uint32_t a[8], bq[8];
          tmem_ld8(tmem + lane_addr + kTDP + col0 + hh * 16, a);
          tmem_ld8(tmem + lane_addr + kTDP + col0 + hh * 16 + 8, bq);
          tc_wait_ld_regs(a, bq);
          uint32_t dw[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const uint32_t x0 = e < 4 ? a[2 * e] : bq[2 * e - 8];
            const uint32_t x1 = e < 4 ? a[2 * e + 1] : bq[2 * e - 7];
            const float2 dp2 = make_float2(__uint_as_float(x0), __uint_as_float(x1));
            const float2 ds = fmul2(p[hh * 8 + e], fadd2(dp2, ndl2));
            dbacc[hh * 8 + e] = fadd2(dbacc[hh * 8 + e], ds);
            dw[e] = pack_bf16x2(ds.x, ds.y);
          }
#pragma unroll
          for (int v = 0; v < 2; ++v) {
            const int cc = (col0 >> 3) + hh * 2 + v;
            const uint32_t off = (cc >> 3) * (BM * 128) + sw128(r, cc & 7);
            *reinterpret_cast<uint4*>(sDS + off) = make_uint4(dw[4 * v], dw[4 * v + 1], dw[4 * v + 2], dw[4 * v + 3]);
          }
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bars->ds_ready);
      if (g == G - 1) {
        // single-writer dbias partial of this outer group for tile (i, ktile),
        // stored chunk-major ([32 float4 chunks][128 rows]) so that each warp
        // store covers 512 contiguous bytes
        float4* dst = reinterpret_cast<float4*>(dbias_part) +
                      ((((static_cast<size_t>(grp) * gridDim.z + bh) * JQ + i) * gridDim.x + ktile) * (BM * BN / 4)) +
                      (col0 / 4) * BM + r;
#pragma unroll
        for (int k4 = 0; k4 < kCols / 4; ++k4)
          dst[k4 * BM] = make_float4(dbacc[2 * k4].x, dbacc[2 * k4].y, dbacc[2 * k4 + 1].x, dbacc[2 * k4 + 1].y);
#pragma unroll
        for (int k = 0; k < kCols / 2; ++k) dbacc[k] = make_float2(0.f, 0.f);
      }
    }
    // the last step's dQ tile
    if (ok && __all_sync(0xffffffffu, mbar_wait(&bars->dq_full, (nsteps - 1) & 1, wc, abort))) {
      tc_fence_after();
      store_dq_tile(nsteps - 1);
    } else {
      ok = false;
    }

    // ------------------------------------------------------------ epilogue: dV_g and dK_g of slice g = wg
    if (ok) {
      // the last dq_full wait above covers every MMA of this CTA
      const int krow = ktile * BN + r;  // key of this thread's TMEM lane
      const int g = wg;
      const size_t row = (static_cast<size_t>((b * N_o + o0 + g) * H + h)) * N + krow;
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const uint32_t t = tmem + lane_addr + which * 4 * D + g * D;
        const float sc = which == 0 ? 1.f : inv_sqrt_d;
        uint32_t w[D / 2];
        if constexpr (D == 32) {
          uint32_t raw[32];
          tmem_ld32(t, raw);
          tc_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e)
            w[e] = pack_bf16x2(__uint_as_float(raw[2 * e]) * sc, __uint_as_float(raw[2 * e + 1]) * sc);
        } else {
          uint32_t raw[16];
          tmem_ld16(t, raw);
          tc_wait_ld();
#pragma unroll
          for (int e = 0; e < 8; ++e)
            w[e] = pack_bf16x2(__uint_as_float(raw[2 * e]) * sc, __uint_as_float(raw[2 * e + 1]) * sc);
        }
        if (krow < N) {
          uint4* dst = reinterpret_cast<uint4*>((which == 0 ? dv : dk) + row * D);
#pragma unroll
          for (int v = 0; v < D / 8; ++v) dst[v] = make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------- reductions
// dQ[row, :] = sum_{t = 0 .. J_K-1} dq_part[t][row, :]   (ascending t, FP32).
// One block per 128-row tile of one slice: coalesced float4 reads of the
// chunk-major partials, FP32 sums in fixed order, transpose through shared
// memory, coalesced BF16 row writes.
template <int D>
__global__ void __launch_bounds__(256) reduce_dq_kernel(const float4* __restrict__ part, uint16_t* __restrict__ dq,
                                                        int N, int JQ, int JK, size_t tiles) {
  constexpr int kChunks = BM * D / 4;      // float4 per tile
  constexpr int kStride = D + 4;           // padded row stride (floats) of the transpose buffer
  __shared__ float tile[BM * kStride];
  const size_t t = blockIdx.x;             // tile = slice * JQ + i
  const int i = static_cast<int>(t % JQ);
  const size_t slice = t / JQ;
  for (int e = threadIdx.x; e < kChunks; e += blockDim.x) {
    const float4* p = part + t * kChunks + e;
    float4 acc = __ldcs(p);
    for (int kt = 1; kt < JK; ++kt) {
      const float4 v = __ldcs(p + static_cast<size_t>(kt) * tiles * kChunks);
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    const int c = e / BM, r = e % BM;
    *reinterpret_cast<float4*>(&tile[r * kStride + 4 * c]) = acc;
  }
  __syncthreads();
  constexpr int kItems = BM * D / 8;       // 16-byte output items (8 bf16)
  for (int e = threadIdx.x; e < kItems; e += blockDim.x) {
    const int r = e / (D / 8), c8 = e % (D / 8);
    const int q = i * BM + r;
    if (q >= N) continue;
    const float* src = &tile[r * kStride + 8 * c8];
    const uint4 w = make_uint4(pack_bf16x2(src[0], src[1]), pack_bf16x2(src[2], src[3]), pack_bf16x2(src[4], src[5]),
                               pack_bf16x2(src[6], src[7]));
    *reinterpret_cast<uint4*>(dq + (slice * N + q) * D + 8 * c8) = w;
  }
}

// dbias[b,h,q,k] = sum_{l = 0 .. L-1} dbias_part[l][b,h,q,k]   (ascending l, FP32).
// One block per 16-row slab of a 128 x 128 tile (b*h, query tile i, key tile
// t); the loads of four consecutive partials are issued together, the adds
// stay in ascending order.
constexpr int kSlab = 16;
__global__ void __launch_bounds__(256) reduce_dbias_kernel(const float4* __restrict__ part,
                                                           uint16_t* __restrict__ dbias, int N, int JQ, int JK,
                                                           int ngroups, size_t tiles) {
  constexpr int kChunks = BM * BN / 4;     // float4 per tile
  constexpr int kSlabChunks = kSlab * BN / 4;
  constexpr int kStride = BN + 8;          // padded row stride (bf16) of the transpose buffer
  __shared__ uint16_t tile[kSlab * kStride];
  const size_t t = blockIdx.x / (BM / kSlab);
  const int slab = blockIdx.x % (BM / kSlab);
  const int kt = static_cast<int>(t % JK);
  const int i = static_cast<int>((t / JK) % JQ);
  const size_t bh = t / (static_cast<size_t>(JK) * JQ);
  const size_t lstride = tiles * kChunks;
  for (int e = threadIdx.x; e < kSlabChunks; e += blockDim.x) {
    const int c = e / kSlab, rr = e % kSlab;
    const float4* p = part + t * kChunks + c * BM + slab * kSlab + rr;
    float4 acc = __ldcs(p);
    int l = 1;
    for (; l + 4 <= ngroups; l += 4) {
      const float4 v0 = __ldcs(p + static_cast<size_t>(l) * lstride);
      const float4 v1 = __ldcs(p + static_cast<size_t>(l + 1) * lstride);
      const float4 v2 = __ldcs(p + static_cast<size_t>(l + 2) * lstride);
      const float4 v3 = __ldcs(p + static_cast<size_t>(l + 3) * lstride);
      acc.x = (((acc.x + v0.x) + v1.x) + v2.x) + v3.x;
      acc.y = (((acc.y + v0.y) + v1.y) + v2.y) + v3.y;
      acc.z = (((acc.z + v0.z) + v1.z) + v2.z) + v3.z;
      acc.w = (((acc.w + v0.w) + v1.w) + v2.w) + v3.w;
    }
    for (; l < ngroups; ++l) {
      const float4 v = __ldcs(p + static_cast<size_t>(l) * lstride);
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    *reinterpret_cast<uint2*>(&tile[rr * kStride + 4 * c]) = make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
  }
  __syncthreads();
  constexpr int kItems = kSlab * BN / 8;   // 16-byte items
  for (int e = threadIdx.x; e < kItems; e += blockDim.x) {
    const int rr = e / (BN / 8), c8 = e % (BN / 8);
    const int q = i * BM + slab * kSlab + rr, k = kt * BN + 8 * c8;
    if (q >= N || k >= N) continue;        // N is a multiple of 8: an item is all in or all out
    *reinterpret_cast<uint4*>(dbias + (bh * N + q) * N + k) = *reinterpret_cast<const uint4*>(&tile[rr * kStride + 8 * c8]);
  }
}

}  // namespace

template <int D>
int bwd_smem_bytes() { return BwdSmem<D>::kBytes; }

template <int D>
cudaError_t setup_bwd() {
  return cudaFuncSetAttribute(bwd_main_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, BwdSmem<D>::kBytes);
}

template <int D>
cudaError_t launch_bwd_preprocess(const BwdArgs& a, cudaStream_t stream) {
  const size_t rows = static_cast<size_t>(a.B) * a.N_o * a.H * a.N;
  const unsigned grid = static_cast<unsigned>((rows + 255) / 256);
  preprocess_kernel<D><<<grid, 256, 0, stream>>>(static_cast<const uint16_t*>(a.dO),
                                                 static_cast<const uint16_t*>(a.o),
                                                 static_cast<const uint16_t*>(a.o_resid), a.delta, rows);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_bwd_main(const BwdArgs& a, cudaStream_t stream) {
  const int JK = (a.N + BN - 1) / BN;
  dim3 grid(JK, a.N_o / G, a.B * a.H);
  bwd_main_kernel<D><<<grid, kMainThreads, BwdSmem<D>::kBytes, stream>>>(
      a.tm_q, a.tm_k, a.tm_v, a.tm_do, a.tm_bias, static_cast<const uint16_t*>(a.mask), a.lse, a.delta,
      static_cast<uint16_t*>(a.dk), static_cast<uint16_t*>(a.dv), a.dq_part, a.dbias_part, a.N_o, a.N, a.H, a.wc);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_bwd_reduce_dq(const BwdArgs& a, cudaStream_t stream) {
  const int JK = (a.N + BN - 1) / BN, JQ = (a.N + BM - 1) / BM;
  const size_t tiles = static_cast<size_t>(a.B) * a.N_o * a.H * JQ;
  reduce_dq_kernel<D><<<static_cast<unsigned>(tiles), 256, 0, stream>>>(
      reinterpret_cast<const float4*>(a.dq_part), static_cast<uint16_t*>(a.dq), a.N, JQ, JK, tiles);
  return cudaGetLastError();
}

cudaError_t launch_bwd_reduce_dbias(const BwdArgs& a, cudaStream_t stream) {
  const int JK = (a.N + BN - 1) / BN, JQ = (a.N + BM - 1) / BM;
  const size_t tiles = static_cast<size_t>(a.B) * a.H * JQ * JK;
  reduce_dbias_kernel<<<static_cast<unsigned>(tiles * (BM / kSlab)), 256, 0, stream>>>(
      reinterpret_cast<const float4*>(a.dbias_part), static_cast<uint16_t*>(a.dbias), a.N, JQ, JK, a.N_o / G, tiles);
  return cudaGetLastError();
}

template cudaError_t setup_bwd<16>();
template cudaError_t setup_bwd<32>();
template cudaError_t launch_bwd_preprocess<16>(const BwdArgs&, cudaStream_t);
template cudaError_t launch_bwd_preprocess<32>(const BwdArgs&, cudaStream_t);
template cudaError_t launch_bwd_main<16>(const BwdArgs&, cudaStream_t);
template cudaError_t launch_bwd_main<32>(const BwdArgs&, cudaStream_t);
template cudaError_t launch_bwd_reduce_dq<16>(const BwdArgs&, cudaStream_t);
template cudaError_t launch_bwd_reduce_dq<32>(const BwdArgs&, cudaStream_t);
template int bwd_smem_bytes<16>();
template int bwd_smem_bytes<32>();

}  // namespace triattn
