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
constexpr int kThreads = 192;
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
  static constexpr int kBar = kMask + G * BN * 4;
  static constexpr int kBytes = kBar + 256;
  static_assert(kBytes <= 232448, "shared memory budget");
};

struct BwdBars {
  uint64_t kv_full;
  uint64_t qdo_full[2], qdo_empty[2];
  uint64_t b_full[2], b_empty[2];
  uint64_t sdp_full, ds_ready, mma_done, tmem_free;
  uint32_t tmem_slot;
  int abort;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
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
  const size_t rows_total_bh = static_cast<size_t>(N);  // rows per (b,o,h)

  // The swizzled tiles below need a 1024-byte aligned base.
  if ((smem_u32(sm) & 1023u) != 0) {
    if (tid == 0) atomicOr(wc.status, 2u);
    return;
  }

  constexpr uint32_t kTS = 8 * D;                       // S (128 cols)
  constexpr uint32_t kTDP = kTS + 128;                  // dP (128 cols)
  constexpr uint32_t kTDQ = (D == 32) ? kTS : kTDP + 128;  // dQ tile (D cols)

  if (tid == 0) {
    mbar_init(&bars->kv_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->qdo_full[i], 1);
      mbar_init(&bars->qdo_empty[i], 1);
      mbar_init(&bars->b_full[i], 1);
      mbar_init(&bars->b_empty[i], BM);
    }
    mbar_init(&bars->sdp_full, 1);
    mbar_init(&bars->ds_ready, BM);
    mbar_init(&bars->mma_done, 1);
    mbar_init(&bars->tmem_free, BM);
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
    if (lane == 0) {
      constexpr uint32_t kSwz = (D == 32) ? 4u : 6u;  // 64B / 32B swizzle for D-wide rows
      constexpr uint32_t kSbo = 8u * D * 2u;
      constexpr uint32_t idSS = idesc_bf16_f32(BM, BN, 0, 0);     // S, dP
      constexpr uint32_t idKV = idesc_bf16_f32(BN, D, 1, 1);      // dV, dK: A MN-major, B MN-major
      constexpr uint32_t idQ = idesc_bf16_f32(BM, D, 0, 1);       // dQ: A K-major, B MN-major
      const uint32_t sP = smem_u32(sm + L::kP), sDS = smem_u32(sm + L::kDS);
      const uint32_t sK = smem_u32(sm + L::kK), sV = smem_u32(sm + L::kV);
      const uint32_t sQ = smem_u32(sm + L::kQ), sDO = smem_u32(sm + L::kDO);
      bool ok = mbar_wait(&bars->kv_full, 0, wc, abort);
      for (int s = 0; s < nsteps && ok; ++s) {
        const int i = s / G, g = s % G, st = s & 1;
        if (!mbar_wait(&bars->qdo_full[st], (s >> 1) & 1, wc, abort)) { ok = false; break; }
        if (s > 0 && !mbar_wait(&bars->tmem_free, (s - 1) & 1, wc, abort)) { ok = false; break; }
        tc_fence_after();
        const uint32_t qb = sQ + st * L::kTile, dob = sDO + st * L::kTile;
        const uint32_t kb = sK + g * L::kTile, vb = sV + g * L::kTile;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          mma_ss(tmem + kTS, smem_desc(qb + kk * 32, 16, kSbo, kSwz), smem_desc(kb + kk * 32, 16, kSbo, kSwz), idSS,
                 kk > 0 ? 1u : 0u);
          mma_ss(tmem + kTDP, smem_desc(dob + kk * 32, 16, kSbo, kSwz), smem_desc(vb + kk * 32, 16, kSbo, kSwz),
                 idSS, kk > 0 ? 1u : 0u);
        }
        mma_commit(&bars->sdp_full);
        if (!mbar_wait(&bars->ds_ready, s & 1, wc, abort)) { ok = false; break; }
        tc_fence_after();
        const uint32_t tdv = tmem + g * D, tdk = tmem + 4 * D + g * D;
#pragma unroll
        for (int kk = 0; kk < BM / 16; ++kk) {
          // dV_g += P^T dO ; dK_g += dS^T Q   (A = P^T / dS^T: keys contiguous, MN-major)
          const uint64_t bdo = smem_desc(dob + kk * 16 * D * 2, 16, kSbo, kSwz);
          const uint64_t bq = smem_desc(qb + kk * 16 * D * 2, 16, kSbo, kSwz);
          mma_ss(tdv, smem_desc(sP + kk * 2048, 16384, 1024, 2), bdo, idKV, (i > 0 || kk > 0) ? 1u : 0u);
          mma_ss(tdk, smem_desc(sDS + kk * 2048, 16384, 1024, 2), bq, idKV, (i > 0 || kk > 0) ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          // dQ tile = dS K  (A = dS: keys contiguous = K-major; B = K: D contiguous = MN-major)
          const uint64_t a = smem_desc(sDS + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024, 2);
          const uint64_t bk = smem_desc(kb + kk * 16 * D * 2, 16, kSbo, kSwz);
          mma_ss(tmem + kTDQ, a, bk, idQ, kk > 0 ? 1u : 0u);
        }
        mma_commit(&bars->mma_done);
        mma_commit(&bars->qdo_empty[st]);
      }
    }
  } else {
    // ------------------------------------------------------------ elementwise warpgroup
    const int ew = tid - 64;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;   // query row in tile (S / dP / dQ lane) and key row (dK / dV lane)
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const float scale_log2 = kLog2e * rsqrtf(static_cast<float>(D));
    const float inv_sqrt_d = rsqrtf(static_cast<float>(D));
    float* mask2 = reinterpret_cast<float*>(sm + L::kMask);
    uint8_t* sP = sm + L::kP;
    uint8_t* sDS = sm + L::kDS;
    const int key = ktile * BN + ew;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float mv = -INFINITY;
      if (key < N) {
        mv = 0.f;
        if (mask != nullptr)
          mv = __uint_as_float(static_cast<uint32_t>(__ldg(mask + (static_cast<size_t>(b) * N_o + o0 + g) * N + key))
                               << 16) *
               kLog2e;
      }
      mask2[g * BN + ew] = mv;
    }
    named_bar_sync(1, BM);

    auto row_stats = [&](int s, float& lse2, float& dl) {
      const int i = s / G, g = s % G;
      const int q = i * BM + r;
      lse2 = INFINITY;
      dl = 0.f;
      if (q < N) {
        const size_t row = (static_cast<size_t>((b * N_o + o0 + g) * H + h)) * rows_total_bh + q;
        const float l = __ldg(lse + row);
        if (l != -INFINITY) lse2 = l * kLog2e;
        dl = __ldg(delta + row);
      }
    };
    float lse2_n, dl_n;
    row_stats(0, lse2_n, dl_n);
    float dbacc[BN];
#pragma unroll
    for (int k = 0; k < BN; ++k) dbacc[k] = 0.f;
    bool ok = true;

    for (int s = 0; s < nsteps && ok; ++s) {
      const int i = s / G, g = s % G;
      const float lse2 = lse2_n, dl = dl_n;
      if (s + 1 < nsteps) row_stats(s + 1, lse2_n, dl_n);
      const int bst = i & 1;
      if (g == 0 && !__all_sync(0xffffffffu, mbar_wait(&bars->b_full[bst], (i >> 1) & 1, wc, abort))) {
        ok = false;
        break;
      }
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->sdp_full, s & 1, wc, abort))) { ok = false; break; }
      tc_fence_after();
      const uint8_t* bias_s = sm + L::kBias + bst * (BM * BN * 2);
      const float* mk = mask2 + g * BN;
#pragma unroll
      for (int c = 0; c < 4; ++c) {  // 32 keys per chunk
        uint32_t sraw[32], praw[32];
        tmem_ld32(tmem + lane_addr + kTS + c * 32, sraw);
        tmem_ld32(tmem + lane_addr + kTDP + c * 32, praw);
        tc_wait_ld();
        uint32_t pw[16], dw[16];
#pragma unroll
        for (int v = 0; v < 4; ++v) {  // 8 keys per 16-byte chunk
          const int cc = c * 4 + v;      // 16-byte chunk index along the key axis (0..15)
          const uint4 bw = *reinterpret_cast<const uint4*>(bias_s + (cc >> 3) * (BM * 128) + sw128(r, cc & 7));
          const float4 m0 = *reinterpret_cast<const float4*>(mk + cc * 8);
          const float4 m1 = *reinterpret_cast<const float4*>(mk + cc * 8 + 4);
          const float bb[8] = {bf16lo_to_f32(bw.x), bf16hi_to_f32(bw.x), bf16lo_to_f32(bw.y), bf16hi_to_f32(bw.y),
                               bf16lo_to_f32(bw.z), bf16hi_to_f32(bw.z), bf16lo_to_f32(bw.w), bf16hi_to_f32(bw.w)};
          const float mm[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
          float pv[8], dsv[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int kk = v * 8 + e;
            const float t = fmaf(__uint_as_float(sraw[kk]), scale_log2, fmaf(bb[e], kLog2e, mm[e] - lse2));
            const float p = ex2_approx(t);
            const float ds = p * (__uint_as_float(praw[kk]) - dl);
            dbacc[c * 32 + kk] += ds;
            pv[e] = p;
            dsv[e] = ds * inv_sqrt_d;
          }
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            pw[v * 4 + e] = pack_bf16x2(pv[2 * e], pv[2 * e + 1]);
            dw[v * 4 + e] = pack_bf16x2(dsv[2 * e], dsv[2 * e + 1]);
          }
        }
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const int cc = c * 4 + v;
          const uint32_t off = (cc >> 3) * (BM * 128) + sw128(r, cc & 7);
          *reinterpret_cast<uint4*>(sP + off) = make_uint4(pw[4 * v], pw[4 * v + 1], pw[4 * v + 2], pw[4 * v + 3]);
          *reinterpret_cast<uint4*>(sDS + off) = make_uint4(dw[4 * v], dw[4 * v + 1], dw[4 * v + 2], dw[4 * v + 3]);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bars->ds_ready);
      if (g == G - 1) {
        mbar_arrive(&bars->b_empty[bst]);
        // single-writer dbias partial of this outer group: rows of query tile i,
        // columns of key tile ktile
        const int q = i * BM + r;
        if (q < N) {
          float* dst = dbias_part + (static_cast<size_t>(grp) * gridDim.z + bh) * static_cast<size_t>(N) * N +
                       static_cast<size_t>(q) * N + static_cast<size_t>(ktile) * BN;
          const int nk = min(BN, N - ktile * BN);
#pragma unroll
          for (int k4 = 0; k4 < BN / 4; ++k4)
            if (k4 * 4 < nk)
              reinterpret_cast<float4*>(dst)[k4] =
                  make_float4(dbacc[4 * k4], dbacc[4 * k4 + 1], dbacc[4 * k4 + 2], dbacc[4 * k4 + 3]);
        }
#pragma unroll
        for (int k = 0; k < BN; ++k) dbacc[k] = 0.f;
      }
      // dQ partial of this key tile
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->mma_done, s & 1, wc, abort))) { ok = false; break; }
      tc_fence_after();
      {
        const int q = i * BM + r;
        const size_t rows_all = static_cast<size_t>(gridDim.z) * N_o * N;  // B*H*N_o*N
        const size_t row = (static_cast<size_t>((b * N_o + o0 + g) * H + h)) * N + q;
        float* out = dq_part + (static_cast<size_t>(ktile) * rows_all + row) * D;
        if constexpr (D == 32) {
          uint32_t qr[32];
          tmem_ld32(tmem + lane_addr + kTDQ, qr);
          tc_wait_ld();
          if (q < N) {
#pragma unroll
            for (int v = 0; v < 8; ++v)
              reinterpret_cast<float4*>(out)[v] =
                  make_float4(__uint_as_float(qr[4 * v]), __uint_as_float(qr[4 * v + 1]),
                              __uint_as_float(qr[4 * v + 2]), __uint_as_float(qr[4 * v + 3]));
          }
        } else {
          uint32_t qr[16];
          tmem_ld16(tmem + lane_addr + kTDQ, qr);
          tc_wait_ld();
          if (q < N) {
#pragma unroll
            for (int v = 0; v < 4; ++v)
              reinterpret_cast<float4*>(out)[v] =
                  make_float4(__uint_as_float(qr[4 * v]), __uint_as_float(qr[4 * v + 1]),
                              __uint_as_float(qr[4 * v + 2]), __uint_as_float(qr[4 * v + 3]));
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&bars->tmem_free);
    }

    // ------------------------------------------------------------ epilogue: dK, dV
    if (ok) {
      // the last mma_done wait above covers every MMA of this CTA
      tc_fence_after();
      const int krow = ktile * BN + r;  // key of this thread's TMEM lane
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const size_t row = (static_cast<size_t>((b * N_o + o0 + g) * H + h)) * N + krow;
#pragma unroll
        for (int which = 0; which < 2; ++which) {
          const uint32_t t = tmem + lane_addr + (which == 0 ? g * D : 4 * D + g * D);
          uint32_t w[D / 2];
          if constexpr (D == 32) {
            uint32_t raw[32];
            tmem_ld32(t, raw);
            tc_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) w[e] = pack_bf16x2(__uint_as_float(raw[2 * e]), __uint_as_float(raw[2 * e + 1]));
          } else {
            uint32_t raw[16];
            tmem_ld16(t, raw);
            tc_wait_ld();
#pragma unroll
            for (int e = 0; e < 8; ++e) w[e] = pack_bf16x2(__uint_as_float(raw[2 * e]), __uint_as_float(raw[2 * e + 1]));
          }
          if (krow < N) {
            uint4* dst = reinterpret_cast<uint4*>((which == 0 ? dv : dk) + row * D);
#pragma unroll
            for (int v = 0; v < D / 8; ++v) dst[v] = make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
          }
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
// dQ[row, :] = sum_{t = 0 .. J_K-1} dq_part[t][row, :]   (ascending t, FP32)
__global__ void __launch_bounds__(256) reduce_dq_kernel(const float4* __restrict__ part, uint2* __restrict__ out,
                                                        size_t n4, int jk) {
  const size_t idx = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= n4) return;
  float4 acc = __ldcs(part + idx);
  for (int t = 1; t < jk; ++t) {
    const float4 v = __ldcs(part + static_cast<size_t>(t) * n4 + idx);
    acc.x += v.x;
    acc.y += v.y;
    acc.z += v.z;
    acc.w += v.w;
  }
  out[idx] = make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
}

// dbias[b,h,q,k] = sum_{l = 0 .. L-1} dbias_part[l][b,h,q,k]   (ascending l, FP32)
__global__ void __launch_bounds__(256) reduce_dbias_kernel(const float4* __restrict__ part, uint2* __restrict__ out,
                                                           size_t n4, int ngroups) {
  const size_t idx = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= n4) return;
  float4 acc = __ldcs(part + idx);
  for (int l = 1; l < ngroups; ++l) {
    const float4 v = __ldcs(part + static_cast<size_t>(l) * n4 + idx);
    acc.x += v.x;
    acc.y += v.y;
    acc.z += v.z;
    acc.w += v.w;
  }
  out[idx] = make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
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
  bwd_main_kernel<D><<<grid, kThreads, BwdSmem<D>::kBytes, stream>>>(
      a.tm_q, a.tm_k, a.tm_v, a.tm_do, a.tm_bias, static_cast<const uint16_t*>(a.mask), a.lse, a.delta,
      static_cast<uint16_t*>(a.dk), static_cast<uint16_t*>(a.dv), a.dq_part, a.dbias_part, a.N_o, a.N, a.H, a.wc);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_bwd_reduce_dq(const BwdArgs& a, cudaStream_t stream) {
  const int JK = (a.N + BN - 1) / BN;
  const size_t n4 = static_cast<size_t>(a.B) * a.N_o * a.H * a.N * D / 4;
  const unsigned grid = static_cast<unsigned>((n4 + 255) / 256);
  reduce_dq_kernel<<<grid, 256, 0, stream>>>(reinterpret_cast<const float4*>(a.dq_part),
                                             static_cast<uint2*>(a.dq), n4, JK);
  return cudaGetLastError();
}

cudaError_t launch_bwd_reduce_dbias(const BwdArgs& a, cudaStream_t stream) {
  const size_t n4 = static_cast<size_t>(a.B) * a.H * a.N * a.N / 4;
  const unsigned grid = static_cast<unsigned>((n4 + 255) / 256);
  reduce_dbias_kernel<<<grid, 256, 0, stream>>>(reinterpret_cast<const float4*>(a.dbias_part),
                                                static_cast<uint2*>(a.dbias), n4, a.N_o / G);
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
