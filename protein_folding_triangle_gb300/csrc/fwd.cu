// Forward kernel of triangular attention on sm_103a.
//
// "TurboPairFormer: Fast and Stable Protein Folding Model Training with an
// Optimized Triangle Attention Kernel": Abstract and Figure 1(a) define the
// operation (N_o slices sharing one pair bias); Table 1 gives the layout
// [B, N_o, H, N, D]; Figure 9 and the Abstract describe the saved BF16
// output-rounding residual used by the backward.
//
// One CTA owns (b, h, a 128-row query tile, a group of GF = 4 outer slices).
// The four slices use the same bias tile for every key tile, so each bias
// tile is loaded once into shared memory and read by four warpgroups.  Key
// tiles are 64 wide, so the four slices each get their own softmax
// warpgroup and their own score, P and O columns in TMEM.
//
// Warp roles (20 warps):
//   warp 0       TMA producer: the four Q tiles once; per 64-key tile one
//                bias tile and, per slice, one K and one V tile (rings of
//                3 / 2 / 2 stages).
//   warps 1, 2   tcgen05 MMA issuers (converged warps, one elected lane
//                issues, descriptors precomputed), for slices {0,2} and
//                {1,3}: S(j+1) = Q K^T as soon as the warpgroup has loaded
//                S(j) into registers, O += P V(j) once it has written P(j).
//   warp 3       idle (completes warpgroup 0 for the register split).
//   warps 4-19   four softmax warpgroups; warpgroup g owns slice g.
//                Thread = query row (TMEM lane).  A thread loads the 64
//                scores of a tile into registers at once (so the next S can
//                be computed meanwhile), forms t = (S/sqrt(D) + bias + mask
//                - m) log2 e in place and the tile maximum; on the first key
//                tile, or when the maximum lies more than 8 (log2 units)
//                above the base m, or when the row has nothing accumulated
//                yet and the maximum lies more than 64 below m, it shifts t
//                and m to the maximum (O rescaled in TMEM).  Then
//                p = 2^t, the row sum, and P (BF16) into TMEM.  The epilogue
//                writes O (BF16), the residual E = bf16(O32 - O) and
//                lse = m + ln l.
//
// TMEM (512 columns): slice g owns [128g, 128g + 128): scores at +0 (64),
// P at +64 (32), O at +96 (D).
#include <type_traits>

#include "kernels.cuh"

namespace triattn {

namespace {

constexpr int BM = 128;     // query rows per tile (TMEM lanes)
constexpr int BN = 64;      // keys per step
constexpr int GF = 4;       // outer slices per CTA (share a bias tile)
constexpr int NSLOT = 3;    // K ring and V ring depth per slice
constexpr int NBIAS = 3;    // bias ring depth
constexpr int kSoftmax = 128 * GF;      // softmax threads (one warpgroup per slice)
constexpr int kThreads = 128 + kSoftmax;
constexpr int kRegsLaunch = 96;         // per thread at launch (__launch_bounds__(kThreads, 1))
constexpr int kRegsCtl = 32;            // warpgroup 0: producer and MMA issuers
constexpr int kRegsSoftmax = 112;     // softmax warpgroups
static_assert(128 * kRegsCtl + kSoftmax * kRegsSoftmax <= kThreads * kRegsLaunch, "register split");
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThresh = 8.0f;  // log2 units: P stays below 2^8
constexpr float kLowThresh = -64.0f;    // log2 units: rebase an empty row whose maximum is this far below
constexpr float kSumThresh = 65536.0f;  // a later tile whose row sum exceeds this (some p > 2^16) is rebased
constexpr uint32_t kTP = 64;            // P columns within a slice's TMEM block
constexpr uint32_t kTO = 96;            // O columns within a slice's TMEM block

template <int D>
struct FwdSmem {
  static constexpr int kTileQ = BM * D * 2;                  // one Q tile (128 rows x D bf16)
  static constexpr int kTileKV = BN * D * 2;                 // one K / V tile (64 keys x D bf16)
  static constexpr int kQ = 0;                               // GF Q tiles
  static constexpr int kK = kQ + GF * kTileQ;                // GF x NSLOT K tiles
  static constexpr int kV = kK + GF * NSLOT * kTileKV;       // GF x NSLOT V tiles
  static constexpr int kBias = kV + GF * NSLOT * kTileKV;    // NBIAS x [128 q][64 k] bf16, SW128
  static constexpr int kBar = kBias + NBIAS * BM * BN * 2;
  static constexpr int kMask = kBar + 1024;  // GF x (JK*64) bf16 key mask, GF x JK x 8 chunk flags, GF x JK tile flags
  static constexpr int kFixed = kMask + 1024;                // + slack for 1024-byte alignment
  static_assert(kBias % 1024 == 0, "bias tiles need 1024-byte alignment");
  static constexpr int bytes(int JK) { return kFixed + GF * JK * (BN * 2 + BN / 8 + 1); }
  static constexpr int kMaxJK = (232448 - kFixed) / (GF * (BN * 2 + BN / 8 + 1));
};

struct FwdBars {
  uint64_t k_full[GF][NSLOT], k_empty[GF][NSLOT];
  uint64_t v_full[GF][NSLOT], v_empty[GF][NSLOT];
  uint64_t b_full[NBIAS], b_empty[NBIAS];
  uint64_t s_full[GF], s_cons[GF], p_full[GF], pv_done[GF];
  uint64_t q_full, all_done;
  uint32_t tmem_slot;
  int abort;
};
static_assert(sizeof(FwdBars) <= 1024, "barrier block");

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

  if (tid == 0) {
    for (int g = 0; g < GF; ++g) {
      for (int i = 0; i < NSLOT; ++i) {
        mbar_init(&bars->k_full[g][i], 1);
        mbar_init(&bars->k_empty[g][i], 1);
        mbar_init(&bars->v_full[g][i], 1);
        mbar_init(&bars->v_empty[g][i], 1);
      }
      mbar_init(&bars->s_full[g], 1);
      mbar_init(&bars->s_cons[g], 128);
      mbar_init(&bars->p_full[g], 128);
      mbar_init(&bars->pv_done[g], 1);
    }
    for (int i = 0; i < NBIAS; ++i) {
      mbar_init(&bars->b_full[i], 1);
      mbar_init(&bars->b_empty[i], kSoftmax);
    }
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->all_done, 2);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(&bars->tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_slot;

  if (warp < 4) regs_dec<kRegsCtl>();
  else regs_inc<kRegsSoftmax>();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      prefetch_tmap(&tm_bias);
      const int row0 = qtile * BM;
      mbar_expect_tx(&bars->q_full, GF * L::kTileQ);
      for (int g = 0; g < GF; ++g)
        tma_load_3d(sm + L::kQ + g * L::kTileQ, &tm_q, &bars->q_full, 0, row0, (b * N_o + o0 + g) * H + h);
      for (int j = 0; j < JK && !*abort; ++j) {
        const int bst = j % NBIAS;
        if (!mbar_wait(&bars->b_empty[bst], ((j / NBIAS) & 1) ^ 1, wc, abort)) break;
        mbar_expect_tx(&bars->b_full[bst], BM * BN * 2);
        tma_load_3d(sm + L::kBias + bst * (BM * BN * 2), &tm_bias, &bars->b_full[bst], j * BN, row0, bh);
        const int slot = j % NSLOT;
        const uint32_t par = ((j / NSLOT) & 1) ^ 1;
        bool go = true;
        for (int g = 0; g < GF && go; ++g) {
          const int boh = (b * N_o + o0 + g) * H + h;
          if (!mbar_wait(&bars->k_empty[g][slot], par, wc, abort)) { go = false; break; }
          if (!(test_starve && j == 0 && g == 0)) {
            mbar_expect_tx(&bars->k_full[g][slot], L::kTileKV);
            tma_load_3d(sm + L::kK + (g * NSLOT + slot) * L::kTileKV, &tm_k, &bars->k_full[g][slot], 0, j * BN, boh);
          }
          if (!mbar_wait(&bars->v_empty[g][slot], par, wc, abort)) { go = false; break; }
          mbar_expect_tx(&bars->v_full[g][slot], L::kTileKV);
          tma_load_3d(sm + L::kV + (g * NSLOT + slot) * L::kTileKV, &tm_v, &bars->v_full[g][slot], 0, j * BN, boh);
        }
        if (!go) break;
      }
    }
  } else if (warp <= 2) {
    // ------------------------------------------------------------ MMA issuers (slices 2(warp-1), 2(warp-1)+1)
    constexpr uint32_t kSwz = (D == 32) ? 4u : 6u;       // 64B / 32B swizzle of D-wide rows
    constexpr uint32_t kSbo = 8u * D * 2u;               // 8 rows of D bf16
    constexpr uint32_t idS = idesc_bf16_f32(BM, BN, 0, 0);   // S = Q K^T: A (Q), B (K) K-major
    constexpr uint32_t idPV = idesc_bf16_f32(BM, D, 0, 1);   // O += P V: A (P) in TMEM, B (V) MN-major
    constexpr uint32_t kTileQ16 = L::kTileQ >> 4;
    constexpr uint32_t kTile16 = L::kTileKV >> 4;
    constexpr uint32_t kRowStep = (16 * D * 2) >> 4;     // 16 rows of a D-wide tile
    const uint64_t dQb = smem_desc(smem_u32(sm + L::kQ), 16, kSbo, kSwz);
    const uint64_t dKb = smem_desc(smem_u32(sm + L::kK), 16, kSbo, kSwz);
    const uint64_t dVb = smem_desc(smem_u32(sm + L::kV), 16, kSbo, kSwz);
    const int g0 = warp - 1;  // slices g0 and g0 + 2 (one warpgroup pair)
    auto issue_s = [&](int g, int slot) {  // S_g = Q_g K^T into the slice's score columns
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss(tmem + 128 * g, dQb + g * kTileQ16 + 2 * kk, dKb + (g * NSLOT + slot) * kTile16 + 2 * kk, idS,
                 kk > 0 ? 1u : 0u);
        mma_commit(&bars->s_full[g]);
        mma_commit(&bars->k_empty[g][slot]);
      }
      __syncwarp();
    };
    bool ok = __all_sync(0xffffffffu, mbar_wait(&bars->q_full, 0, wc, abort));
    for (int g = g0; g < GF && ok; g += 2) {  // S_g(0)
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->k_full[g][0], 0, wc, abort))) { ok = false; break; }
      tc_fence_after();
      issue_s(g, 0);
    }
    for (int j = 0; j < JK && ok; ++j) {
      const int slot = j % NSLOT, slot1 = (j + 1) % NSLOT;
      if (j + 1 < JK) {
        for (int g = g0; g < GF; g += 2) {
          // S(j) of slice g is in registers; K(j+1) loaded
          const uint32_t wb[2] = {smem_u32(&bars->s_cons[g]), smem_u32(&bars->k_full[g][slot1])};
          const uint32_t wp[2] = {static_cast<uint32_t>(j & 1), static_cast<uint32_t>(((j + 1) / NSLOT) & 1)};
          if (!mbar_wait_all(wb, wp, wc, abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_s(g, slot1);
        }
        if (!ok) break;
      }
      for (int g = g0; g < GF; g += 2) {
        // P(j) of slice g in TMEM; V(j) loaded
        const uint32_t wb[2] = {smem_u32(&bars->p_full[g]), smem_u32(&bars->v_full[g][slot])};
        const uint32_t wp[2] = {static_cast<uint32_t>(j & 1), static_cast<uint32_t>((j / NSLOT) & 1)};
        if (!mbar_wait_all(wb, wp, wc, abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            mma_ts(tmem + 128 * g + kTO, tmem + 128 * g + kTP + 8 * kk, dVb + (g * NSLOT + slot) * kTile16 + kk * kRowStep,
                   idPV, (j > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&bars->pv_done[g]);
          mma_commit(&bars->v_empty[g][slot]);
        }
        __syncwarp();
      }
    }
    if (elect_one()) mma_commit(&bars->all_done);
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax warpgroups
    const int ew = tid - 128;             // 0..511
    const int g = (warp - 4) >> 2;        // slice of this warpgroup
    const int quarter = warp & 3;         // TMEM lane quarter of this warp
    const int r = quarter * 32 + lane;    // query row within the tile (= TMEM lane)
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const float inv_sqrt_d = rsqrtf(static_cast<float>(D));
    const int nkeys = JK * BN;
    uint16_t* mask2 = reinterpret_cast<uint16_t*>(sm + L::kMask);  // [GF][nkeys] bf16, -inf past N
    uint8_t* mflag = sm + L::kMask + GF * nkeys * 2;              // [GF][JK*8]: 8-key chunk has a nonzero value
    uint8_t* tflag = mflag + GF * JK * (BN / 8);                  // [GF][JK]: tile has a nonzero value

    // Key mask of the four slices and its chunk / tile flags, staged once,
    // before any bounded wait, so the barriers are always fully entered.
    for (int idx = ew; idx < GF * nkeys; idx += kSoftmax) {
      const int gg = idx / nkeys, key = idx - gg * nkeys;
      uint16_t mv = 0xFF80u;  // -inf
      if (key < N) {
        mv = 0;
        if (mask != nullptr) mv = __ldg(mask + (static_cast<size_t>(b) * N_o + o0 + gg) * N + key);
      }
      mask2[idx] = mv;
    }
    named_bar_sync(1, kSoftmax);
    for (int idx = ew; idx < GF * JK * (BN / 8); idx += kSoftmax) {
      bool any = false;
#pragma unroll
      for (int e = 0; e < 8; ++e) any |= (mask2[idx * 8 + e] & 0x7FFFu) != 0;  // a nonzero value
      mflag[idx] = any ? 1 : 0;
    }
    named_bar_sync(1, kSoftmax);
    for (int idx = ew; idx < GF * JK; idx += kSoftmax) {
      bool any = false;
      for (int e = 0; e < BN / 8; ++e) any |= (mflag[idx * (BN / 8) + e] != 0);
      tflag[idx] = any ? 1 : 0;
    }
    named_bar_sync(1, kSoftmax);

    const int q = qtile * BM + r;
    const size_t row = (static_cast<size_t>((b * N_o + o0 + g) * H + h)) * N + q;

    // running base m (natural units) and sum l of this row
    float m_run = 0.f, l_run = 0.f;
    const float2 c2 = make_float2(inv_sqrt_d * kLog2e, inv_sqrt_d * kLog2e);
    const float2 l2e2 = make_float2(kLog2e, kLog2e);
    const uint32_t tS = tmem + lane_addr + 128 * g;
    bool ok = true;

    for (int j = 0; j < JK && ok; ++j) {
      const int bst = j % NBIAS;
      const uint32_t wb[2] = {smem_u32(&bars->b_full[bst]), smem_u32(&bars->s_full[g])};
      const uint32_t wp[2] = {static_cast<uint32_t>((j / NBIAS) & 1), static_cast<uint32_t>(j & 1)};
      if (!mbar_wait_all(wb, wp, wc, abort)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // the tile's 64 scores into registers; the score columns are free again
      // sv0 holds keys [0, 32), sv1 keys [32, 64)
      uint32_t sv0[32], sv1[32];
      tmem_ld32x2_wait(tS, sv0, tS + 32, sv1);
      tc_fence_before();
      mbar_arrive(&bars->s_cons[g]);

      // P.V(j-1) is complete: the P columns are free and O is up to date
      if (j > 0 && !__all_sync(0xffffffffu, mbar_wait(&bars->pv_done[g], (j - 1) & 1, wc, abort))) {
        ok = false;
        break;
      }
      tc_fence_after();

      // t = (S / sqrt(D) + bias + mask - m) log2 e in place.  The exact
      // path (first key tile, or a row of the warp with nothing accumulated
      // yet) also takes the tile maximum and moves the base to it; later
      // tiles keep the base and only look at the maximum when the row sum
      // of the tile exceeds 2^16 (some p > 2^16).
      const uint8_t* bias_s = sm + L::kBias + bst * (BM * BN * 2);
      const uint16_t* mk = mask2 + (g * nkeys + j * BN);
      const bool tile_masked = tflag[g * JK + j] != 0;
      const bool exact = j == 0 || __any_sync(0xffffffffu, l_run == 0.f);
      const float2 nb2 = make_float2(-m_run * kLog2e, -m_run * kLog2e);
      float tm = -INFINITY;
      // MASKED selects, per key tile (warp-uniform), the version of the loop
      // that adds the key mask; WITH_MAX also takes the maximum of t
      auto scores = [&](uint32_t (&sv)[32], const int cc0, auto masked_tile, auto with_max) {
        constexpr bool MASKED = decltype(masked_tile)::value;
        constexpr bool WITH_MAX = decltype(with_max)::value;
#pragma unroll
        for (int c = 0; c < 4; ++c) {  // 8-key chunks
          const int cc = cc0 + c;
          const uint4 bw = *reinterpret_cast<const uint4*>(bias_s + sw128(r, cc));
          const uint32_t bws[4] = {bw.x, bw.y, bw.z, bw.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int k = c * 8 + 2 * e;
            const float2 s2 = make_float2(__uint_as_float(sv[k]), __uint_as_float(sv[k + 1]));
            const float2 b2 = make_float2(bf16lo_to_f32(bws[e]), bf16hi_to_f32(bws[e]));
            float2 t = ffma2(s2, c2, ffma2(b2, l2e2, nb2));
            if constexpr (MASKED) {  // the pair's two mask values, loaded where they are used
              const uint32_t mw = *reinterpret_cast<const uint32_t*>(mk + cc * 8 + 2 * e);
              t = ffma2(make_float2(bf16lo_to_f32(mw), bf16hi_to_f32(mw)), l2e2, t);
            }
            if constexpr (WITH_MAX) tm = fmax3(tm, t.x, t.y);
            sv[k] = __float_as_uint(t.x);
            sv[k + 1] = __float_as_uint(t.y);
          }
        }
      };
      auto pass1 = [&](auto with_max) {
        if (tile_masked) {
          scores(sv0, 0, std::true_type{}, with_max);
          scores(sv1, 4, std::true_type{}, with_max);
        } else {
          scores(sv0, 0, std::false_type{}, with_max);
          scores(sv1, 4, std::false_type{}, with_max);
        }
      };
      if (exact) pass1(std::true_type{});
      else pass1(std::false_type{});
      mbar_arrive(&bars->b_empty[bst]);  // this thread's last read of the bias tile


      // p = 2^(t - sh), the row sum, and P (BF16) into the P columns, 32
      // keys at a time; returns the row sum
      auto expo = [&](const float sh, auto shifted) -> float {
        constexpr bool SHIFT = decltype(shifted)::value;
        const float2 sh2 = make_float2(-sh, -sh);
        float2 ls = make_float2(0.f, 0.f);
        {
          uint32_t pw[16];
#pragma unroll
          for (int k = 0; k < 32; k += 2) {
            float2 t = make_float2(__uint_as_float(sv0[k]), __uint_as_float(sv0[k + 1]));
            if constexpr (SHIFT) t = fadd2(t, sh2);
            const float2 p = make_float2(ex2_approx(t.x), ex2_approx(t.y));
            ls = fadd2(ls, p);
            pw[k / 2] = pack_bf16x2(p.x, p.y);
          }
          tmem_st16(tS + kTP, pw);
        }
        {
          uint32_t pw[16];
#pragma unroll
          for (int k = 0; k < 32; k += 2) {
            float2 t = make_float2(__uint_as_float(sv1[k]), __uint_as_float(sv1[k + 1]));
            if constexpr (SHIFT) t = fadd2(t, sh2);
            const float2 p = make_float2(ex2_approx(t.x), ex2_approx(t.y));
            ls = fadd2(ls, p);
            pw[k / 2] = pack_bf16x2(p.x, p.y);
          }
          tmem_st16(tS + kTP + 16, pw);
        }
        return ls.x + ls.y;
      };
      // Rebase this row to sh (the maximum of its t values, or 0): m moves
      // by sh, O and l are scaled by 2^-sh when something is accumulated.
      // Returns the scale.
      auto rebase = [&](const float sh) -> float {
        const float a = (l_run > 0.f && sh != 0.f) ? ex2_approx(-sh) : 1.f;
        m_run += sh * kLn2;
        if (__any_sync(0xffffffffu, a != 1.f)) {
          const uint32_t tO = tS + kTO;
#pragma unroll 1
          for (int c0 = 0; c0 < D; c0 += 16) {
            uint32_t ov[16];
            tmem_ld16_wait(tO + c0, ov);
#pragma unroll
            for (int e = 0; e < 16; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * a);
            tmem_st16(tO + c0, ov);
          }
        }
        return a;
      };
      float alpha = 1.f, lsum;
      if (exact) {
        // new base at the tile maximum: on the first tile, when the maximum
        // overshoots the base (P would grow past 2^8), or when nothing is
        // accumulated yet and it lies far below the base
        const float sh =
            (tm != -INFINITY && (j == 0 || tm > kRescaleThresh || (l_run == 0.f && tm < kLowThresh))) ? tm : 0.f;
        alpha = rebase(sh);
        lsum = expo(sh, std::true_type{});
      } else {
        lsum = expo(0.f, std::false_type{});
        const bool need = !(lsum <= kSumThresh);
        if (__any_sync(0xffffffffu, need)) {
          // rare: rebase the rows whose sum overflowed to their tile maximum
          float mx = -INFINITY;
#pragma unroll
          for (int k = 0; k < 32; k += 2) mx = fmax3(mx, __uint_as_float(sv0[k]), __uint_as_float(sv0[k + 1]));
#pragma unroll
          for (int k = 0; k < 32; k += 2) mx = fmax3(mx, __uint_as_float(sv1[k]), __uint_as_float(sv1[k + 1]));
          const float sh = need ? mx : 0.f;
          alpha = rebase(sh);
          lsum = expo(sh, std::true_type{});
        }
      }
      l_run = l_run * alpha + lsum;
      tc_wait_st();
      tc_fence_before();
      mbar_arrive(&bars->p_full[g]);
    }

    // ------------------------------------------------------------ epilogue
    if (ok && __all_sync(0xffffffffu, mbar_wait(&bars->all_done, 0, wc, abort))) {
      tc_fence_after();
      float ov[D];
      {
        const uint32_t tO = tmem + lane_addr + 128 * g + kTO;
        if constexpr (D == 32) {
          uint32_t raw[32];
          tmem_ld32_wait(tO, raw);
#pragma unroll
          for (int e = 0; e < 32; ++e) ov[e] = __uint_as_float(raw[e]);
        } else {
          uint32_t raw[16];
          tmem_ld16_wait(tO, raw);
#pragma unroll
          for (int e = 0; e < 16; ++e) ov[e] = __uint_as_float(raw[e]);
        }
      }
      if (q < N) {
        const float inv = l_run > 0.f ? 1.0f / l_run : 0.f;
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
        for (int v4 = 0; v4 < D / 8; ++v4) op[v4] = make_uint4(ob[4 * v4], ob[4 * v4 + 1], ob[4 * v4 + 2], ob[4 * v4 + 3]);
        if (out_resid != nullptr) {
          uint4* ep = reinterpret_cast<uint4*>(out_resid + row * D);
#pragma unroll
          for (int v4 = 0; v4 < D / 8; ++v4)
            ep[v4] = make_uint4(eb[4 * v4], eb[4 * v4 + 1], eb[4 * v4 + 2], eb[4 * v4 + 3]);
        }
        out_lse[row] = l_run > 0.f ? m_run + __logf(l_run) : -INFINITY;
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
      a.tm_q, a.tm_k, a.tm_v, a.tm_bias, static_cast<const uint16_t*>(a.mask),
      static_cast<uint16_t*>(a.o), a.lse, static_cast<uint16_t*>(a.o_resid), a.N_o, a.N, a.H, a.test_starve, a.wc);
  return cudaGetLastError();
}

template <int D>
cudaError_t setup_fwd() {
  // setmaxnreg.inc waits until the registers it asks for are free in the
  // block's launch allocation: refuse to run a build whose launch register
  // count could not cover the split.
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, fwd_kernel<D>);
  if (e != cudaSuccess) return e;
  if (fa.numRegs < kRegsLaunch) return cudaErrorInvalidConfiguration;
  return cudaFuncSetAttribute(fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
}

bool fwd_attrs_current() {
  // The attribute set by setup_fwd is lost with the context (a device
  // reset); the library then sets every attribute again.
  cudaFuncAttributes fa;
  return cudaFuncGetAttributes(&fa, fwd_kernel<32>) == cudaSuccess && fa.maxDynamicSharedSizeBytes >= 232448;
}

template cudaError_t launch_fwd<16>(const FwdArgs&, cudaStream_t);
template cudaError_t launch_fwd<32>(const FwdArgs&, cudaStream_t);
template cudaError_t setup_fwd<16>();
template cudaError_t setup_fwd<32>();
template int fwd_smem_bytes<16>(int);
template int fwd_smem_bytes<32>(int);

}  // namespace triattn
