// Forward kernel of triangular attention on sm_103a.
//
// "TurboPairFormer: Fast and Stable Protein Folding Model Training with an
// Optimized Triangle Attention Kernel": Abstract and Figure 1(a) define the
// operation (N_o slices sharing one pair bias); Table 1 gives the layout
// [B, N_o, H, N, D]; Figure 9 and the Abstract describe the saved BF16
// output-rounding residual used by the backward.
//
// A work item is (b, h, a 128-row query tile, a group of GF = 4 outer
// slices).  The four slices use the same bias tile for every key tile, so
// each bias tile is loaded once into shared memory and read by four
// warpgroups.  Key tiles are 64 wide, so the four slices each get their own
// softmax warpgroup and their own score, P and O columns in TMEM.
//
// The kernel is persistent: one CTA per SM takes items blockIdx.x,
// blockIdx.x + gridDim.x, ... (the order a plain grid would run them in, so
// neighbouring CTAs still share K, V and bias tiles in L2).  The rings run on
// across items: the producer loads the next item's Q tiles (two stages) and
// first key tiles while the softmax warps finish the current item, and the
// next item's S MMAs start as soon as their operands are there; only its
// first P.V waits until the epilogue has read the current item's O out of
// TMEM.  A CTA per item spent a quarter of its time filling and draining
// its pipeline.
//
// Warp roles (20 warps):
//   warp 0       TMA producer: per item the four Q tiles; per 64-key tile one
//                bias tile with the four slices' key-mask records of that
//                tile, and per slice one K and one V tile (rings of 3 stages).
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
//
// Key mask: a small kernel writes, per (64-key tile, slice), a 144-byte
// record (the tile's 64 additive mask values in BF16, -inf past N, then a
// 16-byte header whose first word is nonzero when any value is), tile-major
// so that the four slices' records of a tile are one bulk copy, loaded with
// the tile's bias.  Without a mask and with N a multiple of 64 there
// are no records and no tile is masked.  Nothing depends on N in shared
// memory, so N is bounded only by the grid and the tensor maps.
//
// A group may extend past N_o (N_o not a multiple of 4): its extra slices
// read records that mask every key, and nothing of theirs is stored.
#include <algorithm>
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
  static constexpr int kQ = 0;                               // 2 stages x GF Q tiles
  static constexpr int kK = kQ + 2 * GF * kTileQ;            // GF x NSLOT K tiles
  static constexpr int kV = kK + GF * NSLOT * kTileKV;       // GF x NSLOT V tiles
  static constexpr int kBias = kV + GF * NSLOT * kTileKV;    // NBIAS x [128 q][64 k] bf16, SW128
  static constexpr int kRec = kBias + NBIAS * BM * BN * 2;   // NBIAS x GF key-mask records
  static constexpr int kBar = kRec + NBIAS * GF * kFwdMaskRec;
  static constexpr int kBytes = kBar + 1024 + 1024;          // + slack for 1024-byte alignment
  static_assert(kBias % 1024 == 0, "bias tiles need 1024-byte alignment");
  static_assert(kFwdMaskRec % 16 == 0 && kRec % 16 == 0, "records are bulk copies");
  static_assert(kBytes <= 232448, "shared memory budget");
};

struct FwdBars {
  uint64_t k_full[GF][NSLOT], k_empty[GF][NSLOT];
  uint64_t v_full[GF][NSLOT], v_empty[GF][NSLOT];
  uint64_t b_full[NBIAS], b_empty[NBIAS];
  uint64_t s_full[GF], s_cons[GF], p_full[GF], pv_done[GF];
  uint64_t o_free[GF];          // the item's O read out of TMEM by the epilogue
  uint64_t q_full[2], q_empty[2];
  uint64_t never;               // completes no phase: a parity-1 wait on it always passes
  uint32_t tmem_slot;
  int abort;
};
static_assert(sizeof(FwdBars) <= 1024, "barrier block");

}  // namespace

// GENERAL = false: q, k, v, o and its residual in the contiguous layout
// [B, N_o, H, N, D] (3-D tensor maps, row indices).  GENERAL = true: any row
// layouts (the maps of q, k, v follow lq.hn, o and the residual lo's
// strides), and the items run heads first, so that the items running
// together read or write neighbouring heads of the same rows.
template <int D, bool GENERAL>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_bias,
               const uint8_t* __restrict__ mrec, uint16_t* __restrict__ out_o, float* __restrict__ out_lse,
               uint16_t* __restrict__ out_resid, int N_o, int N, int H, int BH, int test_starve, RowLayout lq,
               RowLayout lo, WaitCtl wc) {
  using L = FwdSmem<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  FwdBars* bars = reinterpret_cast<FwdBars*>(sm + L::kBar);
  volatile int* abort = &bars->abort;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int JQ = (N + BM - 1) / BM;
  const int NG = (N_o + GF - 1) / GF;                     // outer groups
  const int JK = (N + BN - 1) / BN;
  const int rec_slices = (BH / H) * N_o + GF;             // records per key tile
  // Work items, in the order of a (JQ, NG, B*H) grid (heads first when they
  // lie inside the rows of q, k, v): this CTA takes items
  // blockIdx.x, blockIdx.x + gridDim.x, ...; nitems of them.
  const int total = JQ * NG * BH;
  const int nitems = blockIdx.x < total ? (total - 1 - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1 : 0;
  const int ntiles = nitems * JK;                         // key tiles over all of this CTA's items
  struct Item { int qtile, o0, bh, b, h; };
  auto item_of = [&](int k) {
    const int it = static_cast<int>(blockIdx.x) + k * static_cast<int>(gridDim.x);
    Item r;
    if constexpr (GENERAL) {
      r.h = it % H;
      const int rest = it / H;
      r.qtile = rest % JQ;
      r.o0 = ((rest / JQ) % NG) * GF;
      r.b = rest / (JQ * NG);
      r.bh = r.b * H + r.h;
    } else {
      r.qtile = it % JQ;
      r.o0 = ((it / JQ) % NG) * GF;
      r.bh = it / (JQ * NG);
      r.b = r.bh / H;
      r.h = r.bh - r.b * H;
    }
    return r;
  };

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
      mbar_init(&bars->o_free[g], 128);
    }
    for (int i = 0; i < NBIAS; ++i) {
      mbar_init(&bars->b_full[i], 1);
      mbar_init(&bars->b_empty[i], kSoftmax);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->q_full[i], 1);
      mbar_init(&bars->q_empty[i], 2);  // both issuers, after an item's last S
    }
    mbar_init(&bars->never, 1);
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
      bool go = true;
      int bst = 0, bpar = 0, slot = 0, spar = 0;  // ring positions of the current key tile
      for (int k = 0; k < nitems && go && !*abort; ++k) {
        const Item w = item_of(k);
        const int row0 = w.qtile * BM;
        const int qs = k & 1;
        if (!mbar_wait(&bars->q_empty[qs], ((k >> 1) & 1) ^ 1, wc, abort)) break;
        mbar_expect_tx(&bars->q_full[qs], GF * L::kTileQ);
        for (int g = 0; g < GF; ++g)
          tma_load_rows(sm + L::kQ + (qs * GF + g) * L::kTileQ, &tm_q, &bars->q_full[qs], GENERAL && lq.hn, row0, w.h,
                        w.b * N_o + w.o0 + g, H);
        for (int j = 0; j < JK && go; ++j) {
          if (!mbar_wait(&bars->b_empty[bst], bpar ^ 1, wc, abort)) { go = false; break; }
          mbar_expect_tx(&bars->b_full[bst], BM * BN * 2 + (mrec != nullptr ? GF * kFwdMaskRec : 0));
          tma_load_3d(sm + L::kBias + bst * (BM * BN * 2), &tm_bias, &bars->b_full[bst], j * BN, row0, w.bh);
          if (mrec != nullptr)  // the four slices' records of tile j are contiguous
            bulk_load(sm + L::kRec + bst * (GF * kFwdMaskRec),
                      mrec + (static_cast<size_t>(j) * rec_slices + w.b * N_o + w.o0) * kFwdMaskRec, GF * kFwdMaskRec,
                      &bars->b_full[bst]);
          const uint32_t par = spar ^ 1;
          for (int g = 0; g < GF && go; ++g) {
            const int bo = w.b * N_o + w.o0 + g;
            if (!mbar_wait(&bars->k_empty[g][slot], par, wc, abort)) { go = false; break; }
            if (!(test_starve && k == 0 && j == 0 && g == 0)) {
              mbar_expect_tx(&bars->k_full[g][slot], L::kTileKV);
              tma_load_rows(sm + L::kK + (g * NSLOT + slot) * L::kTileKV, &tm_k, &bars->k_full[g][slot], GENERAL && lq.hn,
                            j * BN, w.h, bo, H);
            }
            if (!mbar_wait(&bars->v_empty[g][slot], par, wc, abort)) { go = false; break; }
            mbar_expect_tx(&bars->v_full[g][slot], L::kTileKV);
            tma_load_rows(sm + L::kV + (g * NSLOT + slot) * L::kTileKV, &tm_v, &bars->v_full[g][slot], GENERAL && lq.hn, j * BN,
                          w.h, bo, H);
          }
          if (++bst == NBIAS) { bst = 0; bpar ^= 1; }
          if (++slot == NSLOT) { slot = 0; spar ^= 1; }
        }
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
    // S_g of a key tile (ring slot `slot`, Q stage `qs`; `last` = the item's
    // last key tile) into the slice's score columns
    auto issue_s = [&](int g, int slot, int qs, bool last) {
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss(tmem + 128 * g, dQb + (qs * GF + g) * kTileQ16 + 2 * kk, dKb + (g * NSLOT + slot) * kTile16 + 2 * kk,
                 idS, kk > 0 ? 1u : 0u);
        mma_commit(&bars->s_full[g]);
        mma_commit(&bars->k_empty[g][slot]);
        // the item's last S read its Q stage
        if (last && g == g0 + 2) mma_commit(&bars->q_empty[qs]);
      }
      __syncwarp();
    };
    bool ok = ntiles > 0;
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bars->q_full[0], 0, wc, abort));
    for (int g = g0; g < GF && ok; g += 2) {  // S_g of tile 0
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->k_full[g][0], 0, wc, abort))) { ok = false; break; }
      tc_fence_after();
      issue_s(g, 0, 0, JK == 1);
    }
    // (item k, tile j) of key tile t, its ring slot and phase; the same for t + 1
    int j = 0, k = 0, slot = 0, spar = 0;
    int j1 = 1, k1 = 0, slot1 = 1, spar1 = 0;
    if (j1 == JK) { j1 = 0; k1 = 1; }
    if (slot1 == NSLOT) { slot1 = 0; spar1 = 1; }
    for (int t = 0; t < ntiles && ok; ++t) {
      if (t + 1 < ntiles) {
        if (j1 == 0) {  // the next item's Q tiles
          if (!__all_sync(0xffffffffu, mbar_wait(&bars->q_full[k1 & 1], (k1 >> 1) & 1, wc, abort))) {
            ok = false;
            break;
          }
        }
        for (int g = g0; g < GF; g += 2) {
          // S(t) of slice g is in registers; K(t+1) loaded
          const uint32_t wb[2] = {smem_u32(&bars->s_cons[g]), smem_u32(&bars->k_full[g][slot1])};
          const uint32_t wp[2] = {static_cast<uint32_t>(t & 1), static_cast<uint32_t>(spar1)};
          if (!mbar_wait_all(wb, wp, wc, abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_s(g, slot1, k1 & 1, j1 == JK - 1);
        }
        if (!ok) break;
      }
      for (int g = g0; g < GF; g += 2) {
        // P(t) of slice g in TMEM; V(t) loaded; on an item's first tile the
        // previous item's O has been read out (parity 1 passes for item 0)
        const uint32_t wb[3] = {smem_u32(&bars->p_full[g]), smem_u32(&bars->v_full[g][slot]),
                                smem_u32(j == 0 && k > 0 ? &bars->o_free[g] : &bars->never)};
        const uint32_t wp[3] = {static_cast<uint32_t>(t & 1), static_cast<uint32_t>(spar),
                                j == 0 && k > 0 ? static_cast<uint32_t>((k - 1) & 1) : 1u};
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
      // advance both tile positions by one
      j = j1; k = k1; slot = slot1; spar = spar1;
      if (++j1 == JK) { j1 = 0; ++k1; }
      if (++slot1 == NSLOT) { slot1 = 0; spar1 ^= 1; }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax warpgroups
    const int g = (warp - 4) >> 2;        // slice of this warpgroup
    const int quarter = warp & 3;         // TMEM lane quarter of this warp
    const int r = quarter * 32 + lane;    // query row within the tile (= TMEM lane)
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const float inv_sqrt_d = rsqrtf(static_cast<float>(D));

    const bool has_rec = mrec != nullptr;
    const float2 c2 = make_float2(inv_sqrt_d * kLog2e, inv_sqrt_d * kLog2e);
    const float2 l2e2 = make_float2(kLog2e, kLog2e);
    const uint32_t tS = tmem + lane_addr + 128 * g;
    bool ok = true;

    for (int k = 0; k < nitems && ok; ++k) {
      // running base m (natural units) and sum l of this row
      float m_run = 0.f, l_run = 0.f;

      for (int j = 0; j < JK && ok; ++j) {
        const int jj = k * JK + j;  // key tile over all of this CTA's items (ring phases)
        const int bst = jj % NBIAS;
        const uint32_t wb[2] = {smem_u32(&bars->b_full[bst]), smem_u32(&bars->s_full[g])};
        const uint32_t wp[2] = {static_cast<uint32_t>((jj / NBIAS) & 1), static_cast<uint32_t>(jj & 1)};
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

        // P.V(jj-1) is complete: the P columns are free and O is up to date
        if (jj > 0 && !__all_sync(0xffffffffu, mbar_wait(&bars->pv_done[g], (jj - 1) & 1, wc, abort))) {
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
        const uint8_t* rec_s = sm + L::kRec + (bst * GF + g) * kFwdMaskRec;
        const uint16_t* mk = reinterpret_cast<const uint16_t*>(rec_s);  // this tile's 64 mask values
        const bool tile_masked = has_rec && *reinterpret_cast<const uint32_t*>(rec_s + BN * 2) != 0u;
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

      // ------------------------------------------------------------ epilogue of item k
      // the item's last P.V is complete
      if (ok && __all_sync(0xffffffffu, mbar_wait(&bars->pv_done[g], (k * JK + JK - 1) & 1, wc, abort))) {
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
        // O is in registers: the next item's first P.V may overwrite it
        tc_fence_before();
        mbar_arrive(&bars->o_free[g]);
        const Item w = item_of(k);  // the item's rows: computed here, no registers held in the loop
        const int q = w.qtile * BM + r;
        const int bo = w.b * N_o + w.o0 + g;
        const size_t row = (static_cast<size_t>(bo) * H + w.h) * N + q;  // lse row
        if (q < N && w.o0 + g < N_o) {
          const float inv = l_run > 0.f ? 1.0f / l_run : 0.f;
          uint32_t ob[D / 2], eb[D / 2];
  #pragma unroll
          for (int e = 0; e < D / 2; ++e) {
            const float y0 = ov[2 * e] * inv, y1 = ov[2 * e + 1] * inv;
            const uint32_t w = pack_bf16x2(y0, y1);
            ob[e] = w;
            eb[e] = pack_bf16x2(y0 - bf16lo_to_f32(w), y1 - bf16hi_to_f32(w));
          }
          const size_t off = GENERAL ? static_cast<size_t>(lo.offset(bo, w.h, q)) : row * D;
          uint4* op = reinterpret_cast<uint4*>(out_o + off);
  #pragma unroll
          for (int v4 = 0; v4 < D / 8; ++v4) op[v4] = make_uint4(ob[4 * v4], ob[4 * v4 + 1], ob[4 * v4 + 2], ob[4 * v4 + 3]);
          if (out_resid != nullptr) {
            uint4* ep = reinterpret_cast<uint4*>(out_resid + off);
  #pragma unroll
            for (int v4 = 0; v4 < D / 8; ++v4)
              ep[v4] = make_uint4(eb[4 * v4], eb[4 * v4 + 1], eb[4 * v4 + 2], eb[4 * v4 + 3]);
          }
          out_lse[row] = l_run > 0.f ? m_run + __logf(l_run) : -INFINITY;
        }
      }
    }  // item k
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Key-mask records of the forward, [J_K][B*N_o + GF] (tile-major): one warp
// per (64-key tile, slice), lane l covering keys 2l and 2l + 1.  Slices
// b * N_o + o take the caller's mask (0 without one), -inf past N; the GF
// slices after the last example's are padding (every key -inf) for a group
// that extends past N_o.
__global__ void __launch_bounds__(256) fwd_mask_records_kernel(const uint16_t* __restrict__ mask, uint8_t* __restrict__ rec,
                                                               int N, int rec_slices, int real_slices, size_t total) {
  const size_t w = (static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= total) return;  // whole warps: total is per warp
  const int j = static_cast<int>(w / rec_slices), slice = static_cast<int>(w % rec_slices);
  uint32_t word = 0xFF80FF80u;  // two -inf
  if (slice < real_slices) {
    uint16_t v[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int key = j * BN + 2 * lane + e;
      v[e] = 0xFF80u;
      if (key < N) v[e] = mask != nullptr ? __ldg(mask + static_cast<size_t>(slice) * N + key) : static_cast<uint16_t>(0);
    }
    word = static_cast<uint32_t>(v[0]) | (static_cast<uint32_t>(v[1]) << 16);
  }
  uint8_t* r = rec + static_cast<size_t>(w) * kFwdMaskRec;
  reinterpret_cast<uint32_t*>(r)[lane] = word;
  const bool nonzero = (word & 0x7FFF7FFFu) != 0u;  // a value other than +-0
  const unsigned any = __ballot_sync(0xffffffffu, nonzero);
  if (lane == 0) *reinterpret_cast<uint4*>(r + BN * 2) = make_uint4(any != 0u ? 1u : 0u, 0u, 0u, 0u);
}

// biasP[bh][q][k] = bias[bh][q][k] for k < N, 0 for N <= k < Np (Np = N rounded
// up to a multiple of 8), so that TMA can read rows with a 16-byte stride.
__global__ void __launch_bounds__(256) fwd_pad_bias_kernel(const uint16_t* __restrict__ bias, uint16_t* __restrict__ biasP,
                                                           int N, int Np, size_t rows) {
  const size_t t = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int chunks = Np / 8;
  const size_t row = t / chunks;
  if (row >= rows) return;
  const int k0 = static_cast<int>(t % chunks) * 8;
  uint32_t w[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int k = k0 + 2 * e;
    const uint32_t lo = k < N ? __ldg(bias + row * N + k) : 0u;
    const uint32_t hi = k + 1 < N ? __ldg(bias + row * N + k + 1) : 0u;
    w[e] = lo | (hi << 16);
  }
  *reinterpret_cast<uint4*>(biasP + row * Np + k0) = make_uint4(w[0], w[1], w[2], w[3]);
}

cudaError_t launch_fwd_prep(const FwdArgs& a, cudaStream_t stream) {
  if (a.mrec != nullptr) {
    const int JK = (a.N + BN - 1) / BN;
    const int rec_slices = a.B * a.N_o + GF;
    const size_t total = static_cast<size_t>(rec_slices) * JK;
    fwd_mask_records_kernel<<<static_cast<unsigned>((total * 32 + 255) / 256), 256, 0, stream>>>(
        static_cast<const uint16_t*>(a.mask), a.mrec, a.N, rec_slices, a.B * a.N_o, total);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (a.bias_padded != nullptr) {
    const int Np = (a.N + 7) / 8 * 8;
    const size_t rows = static_cast<size_t>(a.B) * a.H * a.N;
    const size_t items = rows * (Np / 8);
    fwd_pad_bias_kernel<<<static_cast<unsigned>((items + 255) / 256), 256, 0, stream>>>(
        static_cast<const uint16_t*>(a.bias), static_cast<uint16_t*>(a.bias_padded), a.N, Np, rows);
    return cudaGetLastError();
  }
  return cudaSuccess;
}

template <int D>
int fwd_smem_bytes() { return FwdSmem<D>::kBytes; }

template <int D>
cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t stream) {
  // persistent: one CTA per SM (the shared memory allows one), each taking
  // every gridDim.x-th item of the (query tile, outer group, b*h) items
  const long long total = static_cast<long long>((a.N + BM - 1) / BM) * ((a.N_o + GF - 1) / GF) * a.B * a.H;
  if (total >= (1ll << 31)) return cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const unsigned grid = static_cast<unsigned>(std::min<long long>(total, sms));
  const RowLayout c = contiguous_layout(a.N, a.H, D);
  auto same = [&](const RowLayout& l) { return l.slice == c.slice && l.head == c.head && l.row == c.row; };
  auto kernel = (same(a.lq) && same(a.lo)) ? fwd_kernel<D, false> : fwd_kernel<D, true>;
  kernel<<<grid, kThreads, FwdSmem<D>::kBytes, stream>>>(
      a.tm_q, a.tm_k, a.tm_v, a.tm_bias, a.mrec, static_cast<uint16_t*>(a.o), a.lse,
      static_cast<uint16_t*>(a.o_resid), a.N_o, a.N, a.H, a.B * a.H, a.test_starve, a.lq, a.lo, a.wc);
  return cudaGetLastError();
}

template <int D>
cudaError_t setup_fwd() {
  // setmaxnreg.inc waits until the registers it asks for are free in the
  // block's launch allocation: refuse to run a build whose launch register
  // count could not cover the split.
  for (auto kernel : {fwd_kernel<D, false>, fwd_kernel<D, true>}) {
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, kernel);
    if (e != cudaSuccess) return e;
    if (fa.numRegs < kRegsLaunch) return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

bool fwd_attrs_current() {
  // The attribute set by setup_fwd is lost with the context (a device
  // reset); the library then sets every attribute again.
  cudaFuncAttributes fa;
  return cudaFuncGetAttributes(&fa, fwd_kernel<32, false>) == cudaSuccess && fa.maxDynamicSharedSizeBytes >= 232448;
}

template cudaError_t launch_fwd<16>(const FwdArgs&, cudaStream_t);
template cudaError_t launch_fwd<32>(const FwdArgs&, cudaStream_t);
template cudaError_t setup_fwd<16>();
template cudaError_t setup_fwd<32>();
template int fwd_smem_bytes<16>();
template int fwd_smem_bytes<32>();

}  // namespace triattn
