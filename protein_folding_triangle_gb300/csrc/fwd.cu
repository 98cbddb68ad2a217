// Forward kernel of triangular attention on sm_103a.
//
// "TurboPairFormer: Fast and Stable Protein Folding Model Training with an
// Optimized Triangle Attention Kernel": Abstract and Figure 1(a) define the
// operation (N_o slices sharing one pair bias); Table 1 gives the layout
// [B, N_o, H, N, D]; Figure 9 and the Abstract describe the saved BF16
// output-rounding residual used by the backward.
//
// One CTA owns (b, h, a 128-row query tile i, a group of GF = 4 outer slices).
// The four slices of the group use the same bias tile for every key tile, so
// each bias tile is loaded once into shared memory and read by four slices.
//
// Warp roles (10 warps):
//   warp 0     TMA producer: Q tiles once, then per key tile one bias tile and
//              one K and one V tile per slice (rings of 2 / 4 / 4 stages).
//   warp 1     TMEM allocator and tcgen05 MMA issuer (one elected lane of a
//              converged warp, descriptors precomputed): S = Q K^T into score
//              buffer s % 3, then O_g += P V with P read from TMEM (the score
//              buffer's first 64 columns, rewritten as packed BF16 by the
//              softmax warps).  With three score buffers S(s+3) is issued
//              right after P V(s), so a warpgroup's next scores are ready
//              when it finishes a step.
//   warps 2-9  two softmax warpgroups; warpgroup w owns the slices g with
//              g % 2 == w, so while one warpgroup computes a softmax the MMA
//              for the other one runs.  Thread = query row (TMEM lane).
//              One pass over the scores exponentiates (base 2) against the
//              running base m of the row and keeps P (BF16) in registers;
//              if the tile's maximum lies more than 8 (log2 units) above m,
//              or the row has nothing accumulated yet and the maximum lies
//              more than 64 below m, the warp redoes the pass with the new
//              base and O is rescaled in TMEM.  Only then is P written to
//              TMEM.  The epilogue writes O (BF16), the residual
//              E = bf16(O32 - O) and lse = m + ln l.
//
// TMEM (512 columns): score buffers at [0,128), [128,256), [256,384); O_g at
// 384 + g*D.  Step s = j*GF + g uses buffer s % 3.
#include "kernels.cuh"

namespace triattn {

namespace {

constexpr int BM = 128;     // query rows per tile (TMEM lanes)
constexpr int BN = 128;     // keys per tile
constexpr int GF = 4;       // outer slices per CTA (share a bias tile)
constexpr int NSLOT = 4;    // K ring and V ring depth
constexpr int NBIAS = 2;    // bias ring depth
constexpr int kEW = 256;               // softmax threads (two warpgroups)
constexpr int kThreads = 64 + kEW;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThresh = 8.0f;  // log2 units: P stays below 2^8
constexpr float kLowThresh = -64.0f;    // log2 units: rebase an empty row whose maximum is this far below
constexpr int kTO = 384;                // first O column in TMEM

template <int D>
struct FwdSmem {
  static constexpr int kTile = BM * D * 2;           // one Q / K / V tile in bytes
  static constexpr int kQ = 0;                       // GF Q tiles
  static constexpr int kK = kQ + GF * kTile;         // NSLOT K tiles
  static constexpr int kV = kK + NSLOT * kTile;      // NSLOT V tiles
  static constexpr int kBias = kV + NSLOT * kTile;   // NBIAS x 32 KB (1024-aligned)
  static constexpr int kBar = kBias + NBIAS * BM * BN * 2;
  static constexpr int kMask = kBar + 256;           // GF x JK x 128 fp32 (key mask), then GF x JK x 16 flags
  static constexpr int kFixed = kMask + 1024;        // + slack for 1024-byte alignment
  static_assert(kBias % 1024 == 0, "bias tiles need 1024-byte alignment");
  // bytes for a problem with JK key tiles
  static constexpr int bytes(int JK) { return kFixed + GF * JK * (BN * 4 + 16); }
  static constexpr int kMaxJK = (232448 - kFixed) / (GF * (BN * 4 + 16));
};

struct FwdBars {
  uint64_t q_full;
  uint64_t k_full[NSLOT], k_empty[NSLOT];
  uint64_t v_full[NSLOT], v_empty[NSLOT];
  uint64_t b_full[NBIAS], b_empty[NBIAS];
  uint64_t s_full[3], p_full[3];
  uint64_t all_done;
  uint32_t tmem_slot;
  int abort;
};

}  // namespace

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_bias,
               const uint16_t* __restrict__ mask, uint16_t* __restrict__ out_o, float* __restrict__ out_lse,
               uint16_t* __restrict__ out_resid, int N_o, int N, int H, int test_starve, WaitCtl wc) {
  using L = FwdSmem<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  FwdBars* bars = reinterpret_cast<FwdBars*>(sm + L::kBar);
  volatile int* abort = &bars->abort;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int qtile = blockIdx.x;
  const int o0 = blockIdx.y * GF;
  const int bh = blockIdx.z;
  const int b = bh / H;
  const int h = bh - b * H;
  const int JK = (N + BN - 1) / BN;
  const int nsteps = JK * GF;

  if (tid == 0) {
    mbar_init(&bars->q_full, 1);
    for (int i = 0; i < NSLOT; ++i) {
      mbar_init(&bars->k_full[i], 1);
      mbar_init(&bars->k_empty[i], 1);
      mbar_init(&bars->v_full[i], 1);
      mbar_init(&bars->v_empty[i], 1);
    }
    for (int i = 0; i < NBIAS; ++i) {
      mbar_init(&bars->b_full[i], 1);
      mbar_init(&bars->b_empty[i], kEW);
    }
    for (int i = 0; i < 3; ++i) {
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->p_full[i], BM);
    }
    mbar_init(&bars->all_done, 1);
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
      prefetch_tmap(&tm_bias);
      const int row0 = qtile * BM;
      mbar_expect_tx(&bars->q_full, GF * L::kTile);
      for (int g = 0; g < GF; ++g)
        tma_load_3d(sm + L::kQ + g * L::kTile, &tm_q, &bars->q_full, 0, row0, (b * N_o + o0 + g) * H + h);
      for (int j = 0; j < JK && !*abort; ++j) {
        const int st = j % NBIAS;
        if (!mbar_wait(&bars->b_empty[st], ((j / NBIAS) & 1) ^ 1, wc, abort)) break;
        mbar_expect_tx(&bars->b_full[st], BM * BN * 2);
        uint8_t* bdst = sm + L::kBias + st * (BM * BN * 2);
        tma_load_3d(bdst, &tm_bias, &bars->b_full[st], j * BN, row0, bh);
        tma_load_3d(bdst + BM * 128, &tm_bias, &bars->b_full[st], j * BN + 64, row0, bh);
        for (int g = 0; g < GF; ++g) {
          const int s = j * GF + g;
          const int slot = s % NSLOT;
          const uint32_t par = ((s / NSLOT) & 1) ^ 1;
          const int boh = (b * N_o + o0 + g) * H + h;
          if (!mbar_wait(&bars->k_empty[slot], par, wc, abort)) break;
          if (!(test_starve && s == 0)) {
            mbar_expect_tx(&bars->k_full[slot], L::kTile);
            tma_load_3d(sm + L::kK + slot * L::kTile, &tm_k, &bars->k_full[slot], 0, j * BN, boh);
          }
          if (!mbar_wait(&bars->v_empty[slot], par, wc, abort)) break;
          mbar_expect_tx(&bars->v_full[slot], L::kTile);
          tma_load_3d(sm + L::kV + slot * L::kTile, &tm_v, &bars->v_full[slot], 0, j * BN, boh);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t kSwz = (D == 32) ? 4u : 6u;       // 64B / 32B swizzle
    constexpr uint32_t kSbo = 8u * D * 2u;               // 8 rows of D bf16
    constexpr uint32_t idS = idesc_bf16_f32(BM, BN, 0, 0);
    constexpr uint32_t idPV = idesc_bf16_f32(BM, D, 0, 1);
    constexpr uint32_t kTile16 = L::kTile >> 4;          // tile size in descriptor units
    constexpr uint32_t kRowStep = (16 * D * 2) >> 4;     // 16 rows of a D-wide tile
    // base descriptors; per-MMA offsets are added to the start-address field
    const uint64_t dQb = smem_desc(smem_u32(sm + L::kQ), 16, kSbo, kSwz);
    const uint64_t dKb = smem_desc(smem_u32(sm + L::kK), 16, kSbo, kSwz);
    const uint64_t dVb = smem_desc(smem_u32(sm + L::kV), 16, kSbo, kSwz);
    bool ok = __all_sync(0xffffffffu, mbar_wait(&bars->q_full, 0, wc, abort));
    auto issue_s = [&](int s) -> bool {
      const int g = s % GF, slot = s % NSLOT;
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->k_full[slot], (s / NSLOT) & 1, wc, abort))) return false;
      tc_fence_after();
      if (elect_one()) {
        const uint32_t dS = tmem + (s % 3) * BN;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss(dS, dQb + g * kTile16 + 2 * kk, dKb + slot * kTile16 + 2 * kk, idS, kk > 0 ? 1u : 0u);
        mma_commit(&bars->s_full[s % 3]);
        mma_commit(&bars->k_empty[slot]);
      }
      __syncwarp();
      return true;
    };
    for (int s = 0; s < 3 && s < nsteps && ok; ++s) ok = issue_s(s);
    for (int s = 0; s < nsteps && ok; ++s) {
      const int g = s % GF, j = s / GF, slot = s % NSLOT, buf = s % 3;
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->p_full[buf], (s / 3) & 1, wc, abort))) { ok = false; break; }
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->v_full[slot], (s / NSLOT) & 1, wc, abort))) { ok = false; break; }
      tc_fence_after();
      if (elect_one()) {
        const uint32_t dO = tmem + kTO + g * D;
        const uint32_t aP = tmem + buf * BN;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          mma_ts(dO, aP + kk * 8, dVb + slot * kTile16 + kk * kRowStep, idPV, (j > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&bars->v_empty[slot]);
      }
      __syncwarp();
      if (s + 3 < nsteps) ok = issue_s(s + 3);
    }
    if (elect_one()) mma_commit(&bars->all_done);
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax warpgroups
    const int ew = tid - 64;              // 0..255
    const int wg = (warp - 2) >> 2;       // warpgroup: slices g with g % 2 == wg
    const int quarter = warp & 3;         // TMEM lane quarter of this warp
    const int r = quarter * 32 + lane;    // query row within the tile (= TMEM lane)
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const float inv_sqrt_d = rsqrtf(static_cast<float>(D));
    float* mask2 = reinterpret_cast<float*>(sm + L::kMask);
    uint8_t* mflag = sm + L::kMask + nsteps * BN * 4;

    // Key mask of every (key tile, slice) step (natural-log units, -inf past
    // N) and per 8-key chunk a flag "some mask value is nonzero": staged once,
    // before any bounded wait, so the two barriers are always fully entered.
    for (int idx = ew; idx < nsteps * BN; idx += kEW) {
      const int s = idx / BN, key = (s / GF) * BN + (idx % BN), g = s % GF;
      float mv = -INFINITY;
      if (key < N) {
        mv = 0.f;
        if (mask != nullptr)
          mv = __uint_as_float(static_cast<uint32_t>(__ldg(mask + (static_cast<size_t>(b) * N_o + o0 + g) * N + key))
                               << 16);
      }
      mask2[idx] = mv;
    }
    named_bar_sync(1, kEW);
    for (int idx = ew; idx < nsteps * 16; idx += kEW) {
      bool any = false;
#pragma unroll
      for (int e = 0; e < 8; ++e) any |= (mask2[idx * 8 + e] != 0.f);
      mflag[idx] = any ? 1 : 0;
    }
    named_bar_sync(1, kEW);

    // running base m (natural units) and sum l for this warpgroup's two slices
    float m_run[2] = {0.f, 0.f}, l_run[2] = {0.f, 0.f};
    const float2 c2 = make_float2(inv_sqrt_d * kLog2e, inv_sqrt_d * kLog2e);
    const float2 l2e2 = make_float2(kLog2e, kLog2e);
    bool ok = true;

    for (int j = 0; j < JK && ok; ++j) {
      const int st = j % NBIAS;
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->b_full[st], (j / NBIAS) & 1, wc, abort))) { ok = false; break; }
      const uint8_t* bias_s = sm + L::kBias + st * (BM * BN * 2);
#pragma unroll 1
      for (int sl = 0; sl < 2; ++sl) {
        const int g = wg + 2 * sl;
        const int s = j * GF + g;
        const int buf = s % 3;
        if (!__all_sync(0xffffffffu, mbar_wait(&bars->s_full[buf], (s / 3) & 1, wc, abort))) { ok = false; break; }
        tc_fence_after();
        const uint32_t tS = tmem + lane_addr + buf * BN;
        const float* mk = mask2 + s * BN;
        const uint8_t* fl = mflag + s * 16;

        // t = (S / sqrt(D) + bias + mask - base) log2 e; returns max t and,
        // with_exp, p = 2^t packed to BF16 in pw and sum p.  16-key chunks,
        // the TMEM load of chunk c+1 in flight while chunk c is computed.
        uint32_t pw[2][32];
        auto score_pass = [&](float base, bool with_exp, float& tmax, float& lsum) {
          const float2 nb2 = make_float2(-base * kLog2e, -base * kLog2e);
          float2 ls = make_float2(0.f, 0.f);
          float tm = -INFINITY;
          uint32_t sb[2][16];
          tmem_ld16(tS, sb[0]);
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            uint32_t(&raw)[16] = sb[c & 1];
            tc_wait_ld_regs(raw);
            if (c + 1 < 8) tmem_ld16(tS + (c + 1) * 16, sb[(c + 1) & 1]);
#pragma unroll
            for (int v = 0; v < 2; ++v) {
              const int cc = c * 2 + v;  // 8-key chunk (0..15)
              const uint4 bw = *reinterpret_cast<const uint4*>(bias_s + (cc >> 3) * (BM * 128) + sw128(r, cc & 7));
              const uint32_t bws[4] = {bw.x, bw.y, bw.z, bw.w};
              const bool masked = fl[cc] != 0;
              float4 m0 = make_float4(0.f, 0.f, 0.f, 0.f), m1 = m0;
              if (masked) {
                m0 = *reinterpret_cast<const float4*>(mk + cc * 8);
                m1 = *reinterpret_cast<const float4*>(mk + cc * 8 + 4);
              }
              const float2 mm[4] = {make_float2(m0.x, m0.y), make_float2(m0.z, m0.w), make_float2(m1.x, m1.y),
                                    make_float2(m1.z, m1.w)};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int k = v * 8 + 2 * e;
                const float2 s2 = make_float2(__uint_as_float(raw[k]), __uint_as_float(raw[k + 1]));
                const float2 b2 = make_float2(bf16lo_to_f32(bws[e]), bf16hi_to_f32(bws[e]));
                float2 t = ffma2(s2, c2, ffma2(b2, l2e2, nb2));
                if (masked) t = ffma2(mm[e], l2e2, t);
                tm = fmax3(tm, t.x, t.y);
                if (with_exp) {
                  const float2 p = make_float2(ex2_approx(t.x), ex2_approx(t.y));
                  ls = fadd2(ls, p);
                  pw[c >> 2][(c & 3) * 8 + v * 4 + e] = pack_bf16x2(p.x, p.y);
                }
              }
            }
          }
          tmax = tm;
          lsum = ls.x + ls.y;
        };

        float tmax, lsum;
        if (j == 0) {
          // first key tile: the base is the tile's row maximum
          score_pass(0.f, false, tmax, lsum);
          m_run[sl] = tmax == -INFINITY ? 0.f : tmax * kLn2;
        }
        score_pass(m_run[sl], true, tmax, lsum);
        // later tiles keep the base unless the tile maximum overshoots it (P
        // would grow past 2^8), or nothing is accumulated yet and the maximum
        // lies far below it; then the warp redoes the pass with a new base
        const bool up = tmax > kRescaleThresh;
        const bool down = l_run[sl] == 0.f && tmax < kLowThresh && tmax != -INFINITY;
        const bool need = up || down;
        float alpha = 1.f;
        if (__any_sync(0xffffffffu, need)) {
          const float m_old = m_run[sl];
          if (need) m_run[sl] = m_old + tmax * kLn2;
          float t2;
          score_pass(m_run[sl], true, t2, lsum);
          if (need && l_run[sl] > 0.f) alpha = ex2_approx((m_old - m_run[sl]) * kLog2e);
        }
        if (sl == 1) mbar_arrive(&bars->b_empty[st]);  // this warpgroup's last read of the bias tile
        l_run[sl] = l_run[sl] * alpha + lsum;
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
          // O_g's previous P.V (step s - 4) was issued before S(s - 1); the
          // S of this step was issued after it, so s_full implies it finished.
          const uint32_t tO = tmem + lane_addr + kTO + g * D;
#pragma unroll 1
          for (int c0 = 0; c0 < D; c0 += 16) {
            uint32_t ov[16];
            tmem_ld16(tO + c0, ov);
            tc_wait_ld_regs(ov);
#pragma unroll
            for (int e = 0; e < 16; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
            tmem_st16(tO + c0, ov);
          }
        }
        // P of keys [32c, 32c+32) into columns [16c, 16c+16): S is no longer read
        tmem_st32(tS, pw[0]);
        tmem_st32(tS + 32, pw[1]);
        tc_wait_st();
        tc_fence_before();
        mbar_arrive(&bars->p_full[buf]);
      }
    }

    // ------------------------------------------------------------ epilogue
    if (ok && __all_sync(0xffffffffu, mbar_wait(&bars->all_done, 0, wc, abort))) {
      tc_fence_after();
      const int q = qtile * BM + r;
#pragma unroll
      for (int sl = 0; sl < 2; ++sl) {
        const int g = wg + 2 * sl;
        float ov[D];
        {
          const uint32_t tO = tmem + lane_addr + kTO + g * D;
          if constexpr (D == 32) {
            uint32_t raw[32];
            tmem_ld32(tO, raw);
            tc_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) ov[e] = __uint_as_float(raw[e]);
          } else {
            uint32_t raw[16];
            tmem_ld16(tO, raw);
            tc_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) ov[e] = __uint_as_float(raw[e]);
          }
        }
        if (q < N) {
          const float l = l_run[sl];
          const float inv = l > 0.f ? 1.0f / l : 0.f;
          const size_t row = (static_cast<size_t>((b * N_o + o0 + g) * H + h)) * N + q;
          uint32_t ob[D / 2], eb[D / 2];
#pragma unroll
          for (int e = 0; e < D / 2; ++e) {
            const float y0 = ov[2 * e] * inv, y1 = ov[2 * e + 1] * inv;
            const uint32_t w = pack_bf16x2(y0, y1);
            ob[e] = w;
            eb[e] = pack_bf16x2(y0 - bf16lo_to_f32(w), y1 - bf16hi_to_f32(w));
          }
          uint4* op = reinterpret_cast<uint4*>(out_o + row * D);
#pragma unroll
          for (int v4 = 0; v4 < D / 8; ++v4)
            op[v4] = make_uint4(ob[4 * v4], ob[4 * v4 + 1], ob[4 * v4 + 2], ob[4 * v4 + 3]);
          if (out_resid != nullptr) {
            uint4* ep = reinterpret_cast<uint4*>(out_resid + row * D);
#pragma unroll
            for (int v4 = 0; v4 < D / 8; ++v4)
              ep[v4] = make_uint4(eb[4 * v4], eb[4 * v4 + 1], eb[4 * v4 + 2], eb[4 * v4 + 3]);
          }
          out_lse[row] = l > 0.f ? m_run[sl] + __logf(l) : -INFINITY;
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

template <int D>
int fwd_smem_bytes(int N) { return FwdSmem<D>::bytes((N + BN - 1) / BN); }

template <int D>
cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t stream) {
  const int JQ = (a.N + BM - 1) / BM;
  dim3 grid(JQ, a.N_o / GF, a.B * a.H);
  const int JK = (a.N + BN - 1) / BN;
  if (JK > FwdSmem<D>::kMaxJK) return cudaErrorInvalidValue;
  fwd_kernel<D><<<grid, kThreads, FwdSmem<D>::bytes(JK), stream>>>(
      a.tm_q, a.tm_k, a.tm_v, a.tm_bias, static_cast<const uint16_t*>(a.mask), static_cast<uint16_t*>(a.o), a.lse,
      static_cast<uint16_t*>(a.o_resid), a.N_o, a.N, a.H, a.test_starve, a.wc);
  return cudaGetLastError();
}

template <int D>
cudaError_t setup_fwd() {
  return cudaFuncSetAttribute(fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
}

template cudaError_t launch_fwd<16>(const FwdArgs&, cudaStream_t);
template cudaError_t launch_fwd<32>(const FwdArgs&, cudaStream_t);
template cudaError_t setup_fwd<16>();
template cudaError_t setup_fwd<32>();
template int fwd_smem_bytes<16>(int);
template int fwd_smem_bytes<32>(int);

}  // namespace triattn
