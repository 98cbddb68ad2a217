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
//   warp 1     TMEM allocator and single-thread tcgen05 MMA issuer:
//              S = Q K^T into the score buffer of the slice's warpgroup, then
//              O_g += P V with P read from TMEM (the score buffer's first
//              64 columns, rewritten as packed BF16 by the softmax warps).
//   warps 2-9  two softmax warpgroups; warpgroup w owns the slices g with
//              g % 2 == w, so while one warpgroup computes a softmax the MMA
//              for the other one runs.  Thread = query row (TMEM lane).
//              Pass 1 adds bias and key mask and writes the scores back to
//              TMEM while taking the row max; pass 2 exponentiates (base 2),
//              sums, and writes P as BF16 into TMEM.  O is rescaled in TMEM
//              only when the running max grows by more than 2^8.  The
//              epilogue writes O (BF16), the residual E = bf16(O32 - O) and lse.
//
// TMEM (512 columns): score buffers at [0,128) (warpgroup 0) and [128,256)
// (warpgroup 1); O_g at 256 + g*D.  Step s = j*GF + g uses buffer s % 2.
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
constexpr float kRescaleThresh = 8.0f;  // log2 units

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
  uint64_t s_full[2], p_full[2];
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
    for (int i = 0; i < 2; ++i) {
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
    if (lane == 0) {
      constexpr uint32_t kSwz = (D == 32) ? 4u : 6u;       // 64B / 32B swizzle
      constexpr uint32_t kSbo = 8u * D * 2u;               // 8 rows of D bf16
      constexpr uint32_t idS = idesc_bf16_f32(BM, BN, 0, 0);
      constexpr uint32_t idPV = idesc_bf16_f32(BM, D, 0, 1);
      const uint32_t sQ = smem_u32(sm + L::kQ), sK = smem_u32(sm + L::kK), sV = smem_u32(sm + L::kV);
      bool ok = mbar_wait(&bars->q_full, 0, wc, abort);
      auto issue_s = [&](int s) -> bool {
        const int g = s % GF, slot = s % NSLOT;
        if (!mbar_wait(&bars->k_full[slot], (s / NSLOT) & 1, wc, abort)) return false;
        tc_fence_after();
        const uint32_t dS = tmem + (s & 1) * BN;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t a = smem_desc(sQ + g * L::kTile + kk * 32, 16, kSbo, kSwz);
          const uint64_t bdesc = smem_desc(sK + slot * L::kTile + kk * 32, 16, kSbo, kSwz);
          mma_ss(dS, a, bdesc, idS, kk > 0 ? 1u : 0u);
        }
        mma_commit(&bars->s_full[s & 1]);
        mma_commit(&bars->k_empty[slot]);
        return true;
      };
      if (ok) ok = issue_s(0);
      if (ok && nsteps > 1) ok = issue_s(1);
      for (int s = 0; s < nsteps && ok; ++s) {
        const int g = s % GF, j = s / GF, slot = s % NSLOT;
        if (!mbar_wait(&bars->p_full[s & 1], (s >> 1) & 1, wc, abort)) { ok = false; break; }
        if (!mbar_wait(&bars->v_full[slot], (s / NSLOT) & 1, wc, abort)) { ok = false; break; }
        tc_fence_after();
        const uint32_t dO = tmem + 256 + g * D;
        const uint32_t aP = tmem + (s & 1) * BN;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          const uint64_t bdesc = smem_desc(sV + slot * L::kTile + kk * 16 * D * 2, 16, kSbo, kSwz);
          mma_ts(dO, aP + kk * 8, bdesc, idPV, (j > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&bars->v_empty[slot]);
        if (s + 2 < nsteps) ok = issue_s(s + 2);
      }
      mma_commit(&bars->all_done);
    }
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

    // running max (natural units) and sum for this warpgroup's two slices
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
    const float2 isd2 = make_float2(inv_sqrt_d, inv_sqrt_d);
    const float2 l2e2 = make_float2(kLog2e, kLog2e);
    bool ok = true;

    for (int j = 0; j < JK && ok; ++j) {
      const int st = j % NBIAS;
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->b_full[st], (j / NBIAS) & 1, wc, abort))) { ok = false; break; }
      const uint8_t* bias_s = sm + L::kBias + st * (BM * BN * 2);
#pragma unroll
      for (int sl = 0; sl < 2; ++sl) {
        const int g = wg + 2 * sl;
        const int s = j * GF + g;
        if (!__all_sync(0xffffffffu, mbar_wait(&bars->s_full[wg], (s >> 1) & 1, wc, abort))) { ok = false; break; }
        tc_fence_after();
        const uint32_t tS = tmem + lane_addr + wg * BN;
        const float* mk = mask2 + s * BN;
        const uint8_t* fl = mflag + s * 16;

        // pass 1: u = S / sqrt(D) + bias + mask, written back to TMEM; row max.
        // 32-key chunks, the load of chunk c+1 in flight while c is computed.
        float mt = -INFINITY;
        uint32_t buf[2][32];
        tmem_ld32(tS, buf[0]);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t(&raw)[32] = buf[c & 1];
          tc_wait_ld_regs(raw);
          if (c + 1 < 4) {
            if (c >= 1) tc_wait_st();  // buf[(c+1)&1] fed the store of chunk c-1
            tmem_ld32(tS + (c + 1) * 32, buf[(c + 1) & 1]);
          }
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const int cc = c * 4 + v;  // 8-key chunk (0..15)
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
              float2 u = ffma2(s2, isd2, b2);
              if (masked) u = fadd2(u, mm[e]);
              mt = fmax3(mt, u.x, u.y);
              raw[k] = __float_as_uint(u.x);
              raw[k + 1] = __float_as_uint(u.y);
            }
          }
          tmem_st32(tS + c * 32, raw);
        }
        if (sl == 1) mbar_arrive(&bars->b_empty[st]);  // this warpgroup's last read of the bias tile

        // online softmax with lazy rescaling of O (kept in TMEM)
        const float m_new = fmaxf(m_run[sl], mt);
        float alpha = 1.f;
        bool need = false;
        if (j == 0) {
          m_run[sl] = m_new;
        } else {
          need = (m_new - m_run[sl]) * kLog2e > kRescaleThresh;
          if (need) {
            alpha = ex2_approx((m_run[sl] - m_new) * kLog2e);
            m_run[sl] = m_new;
          }
        }
        const float msub = (m_run[sl] == -INFINITY) ? 0.f : m_run[sl];
        const float2 nm2 = make_float2(-msub * kLog2e, -msub * kLog2e);
        tc_wait_st();

        // pass 2: p = 2^((u - m) log2 e); P (BF16) into the first 64 columns
        float2 lsum = make_float2(0.f, 0.f);
        uint32_t pw[2][16];
        tmem_ld32(tS, buf[0]);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t(&raw)[32] = buf[c & 1];
          tc_wait_ld_regs(raw);
          if (c + 1 < 4) tmem_ld32(tS + (c + 1) * 32, buf[(c + 1) & 1]);
          if (c >= 2) tc_wait_st();  // pw[c&1] fed the store of chunk c-2
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float2 u = make_float2(__uint_as_float(raw[2 * e]), __uint_as_float(raw[2 * e + 1]));
            const float2 t = ffma2(u, l2e2, nm2);
            const float2 p = make_float2(ex2_approx(t.x), ex2_approx(t.y));
            lsum = fadd2(lsum, p);
            pw[c & 1][e] = pack_bf16x2(p.x, p.y);
          }
          // P of keys [32c, 32c+32) lands in columns [16c, 16c+16): already read
          tmem_st16(tS + c * 16, pw[c & 1]);
        }
        l_run[sl] = l_run[sl] * alpha + (lsum.x + lsum.y);
        if (__any_sync(0xffffffffu, need)) {
          // O_g's previous P.V (step s - 4) was issued before this warpgroup's
          // previous S (step s - 2); s_full of this step implies it finished.
          const uint32_t tO = tmem + lane_addr + 256 + g * D;
          if constexpr (D == 32) {
            uint32_t ov[32];
            tmem_ld32(tO, ov);
            tc_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
            tmem_st32(tO, ov);
          } else {
            uint32_t ov[16];
            tmem_ld16(tO, ov);
            tc_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
            tmem_st16(tO, ov);
          }
        }
        tc_wait_st();
        tc_fence_before();
        mbar_arrive(&bars->p_full[wg]);
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
          const uint32_t tO = tmem + lane_addr + 256 + g * D;
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
