// BF16 GEMM on the tcgen05 tensor cores (sm_103a), for the pair-feature
// projections and the per-channel contraction of the triangle multiplicative
// update ("TurboPairFormer", Figure 12, Table 10) and the projections of the
// triangle-attention module (Figure 6).
//
// Row-major C[M, N] = op(A) op(B) with A [M, K] (or [K, M]) and B [K, N] (or
// [N, K]), BF16 operands, FP32 accumulation, C in BF16 or FP32; batched over
// matrices a fixed stride apart; optionally split along K into FP32 partials
// that a second kernel adds in ascending split order (deterministic, no
// atomics), for the weight gradients whose K is the pair count.
//
// Persistent kernel, one CTA per SM, 6 warps:
//   warp 0     TMA producer: per 64-deep K stage one 128 x 64 A tile and one
//              BN x 64 B tile (128-byte swizzle; an operand whose M or N runs
//              contiguously in memory is loaded as 64-wide column blocks), a
//              ring of 4 stages.
//   warp 1     MMA issuer: four M = 128, N = BN, K = 16 MMAs per stage into one
//              of two TMEM accumulators (BN columns each), so the epilogue of
//              one tile overlaps the MMAs of the next.
//   warps 2-5  epilogue: thread = accumulator row (TMEM lane); 32-column
//              chunks converted (BF16 or FP32), staged in swizzled shared
//              memory and written by TMA stores (ragged rows and columns
//              clipped by the output tensor map).
//
// Two further epilogues serve the input projection of the triangle
// multiplicative update, p = x W_p with W_p's columns [a_v | a_g | b_v | b_g |
// g] (C_h, C_h, C_h, C_h, C_z wide), so that p itself never goes to memory:
//   gated      tile n < ceil(C_h / 64) loads the four 64-column blocks of
//              channels [64n, 64n + 64) of the four branch projections side
//              by side (accumulator columns [a_v | a_g | b_v | b_g]); the
//              epilogue forms a = m sigmoid(a_g) a_v and b = m sigmoid(b_g) b_v
//              (m the optional pair mask) and stores them channel-major,
//              [B][C_h][N*N], through a transposed staging block (channel
//              rows of 32 pairs); the remaining tiles hold the g columns,
//              stored pair-major [M][C_z] like a plain tile.
//   gate bwd   the same gated tiles, recomputed in the backward; the epilogue
//              reads dA, dB (channel-major) and writes the four blocks of
//              dp = d(a, b)/d(a_v, a_g, b_v, b_g) pair-major.
//
// A fourth serves the projections of the triangle-attention module, whose
// rows are the pairs (b, i, j) of [B, N, N] and whose columns are nblk blocks
// of H heads of D features (q, k, v, or dO), then H bias columns:
//   heads      each 32-row quarter of a tile (32 consecutive j of one (b, i);
//              N a multiple of 32) goes out per head as a D x 32 box into
//              the core's layout [nblk][B, N, H, N, D] (5-D tensor map), and
//              the bias columns as 32-element rows into the planes
//              [B, H, N, N] (4-D map); padding columns are dropped.
// Every mbarrier wait is bounded (WaitCtl): a wait that runs out records a
// timeout in the device status word and the CTA stops.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "kernels.cuh"

namespace triattn {
namespace {

constexpr int GB_M = 128;   // rows of a tile (TMEM lanes)
constexpr int GB_K = 64;    // K depth of a stage (one 128-byte swizzle row of BF16)
constexpr int GB_SMAX = 4;  // stages (plain tiles; the gated tiles, with twice the epilogue warps, use 3)

struct GemmBars {
  uint64_t full[GB_SMAX], empty[GB_SMAX];
  uint64_t acc_full[2], acc_empty[2];
  uint32_t tmem_slot;
  int abort;
};

struct GemmParams {
  int M, N, K;
  int batch, ksplit, kchunk;  // K range of split ks: [ks * kchunk, min(K, (ks + 1) * kchunk))
  int tiles_m, tiles_n;
  void* C;                    // output (BF16 or FP32), or FP32 partials [ksplit][batch][M][N]
  long long ldc, strideC;     // elements
  int c_f32, partial;
  // gated epilogues
  int Ch, gated_tiles;        // channels per branch; tiles of the four branch blocks
  long long NN;               // pairs per example
  const uint16_t* mask;       // optional pair mask [M] (BF16)
  const uint16_t* dA;         // gate bwd: channel-major gradients of a and b
  const uint16_t* dB;
  int nblk, H, D, Ntok, nbias;  // heads epilogue: head blocks, heads, features, tokens, bias columns
  WaitCtl wc;
};

enum GemmMode { kPlain = 0, kGated = 1, kGateBwd = 2, kHeads = 3 };



// Per mode: epilogue warps (4; 16 for the gated tiles, whose epilogue does
// the gating arithmetic: four warps per TMEM lane quarter, one per (branch,
// 32-channel chunk), and for the heads epilogue, whose many small stores of
// a short-K (HBM-bound) GEMM are latency-bound with 4), ring stages, and bytes
// per staging buffer (FP32 or BF16 32 x 32 blocks; the gated and heads modes
// write BF16 only).
template <int MODE> struct GemmCfg {
  static constexpr int kEpi = MODE == 0 ? 4 : 16;
  static constexpr int kS = MODE == 0 ? 4 : 3;
  static constexpr int kBuf = MODE == 0 ? 4096 : 2048;
  static constexpr int kThreads = (2 + kEpi) * 32;
};

template <int BN, int MODE>
struct GemmSmem {
  static constexpr int kA = GB_M * GB_K * 2;       // 16 KB
  static constexpr int kB = BN * GB_K * 2;         // 16 / 32 KB
  static constexpr int kStage = kA + kB;
  static constexpr int kBar = GemmCfg<MODE>::kS * kStage;
  static constexpr int kStg = kBar + 1024;          // epilogue staging: two buffers per warp
  static constexpr int kBytes = kStg + GemmCfg<MODE>::kEpi * 2 * GemmCfg<MODE>::kBuf + 1024;  // + alignment slack
  static_assert(kBytes <= 232448, "shared memory budget");
  static_assert(kStage % 1024 == 0, "swizzled tiles need 1024-byte alignment");
};

template <int BN, bool A_MN, bool B_MN, int MODE>
__global__ void __launch_bounds__(GemmCfg<MODE>::kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                const __grid_constant__ CUtensorMap tm_c, const __grid_constant__ CUtensorMap tm_x,
                const __grid_constant__ CUtensorMap tm_y, GemmParams p) {
  static_assert(MODE == kPlain || MODE == kHeads || (BN == 256 && !A_MN && B_MN), "gated tiles: K-major x, N-major W_p");
  static_assert(MODE != kHeads || !A_MN, "heads epilogue: K-major A");
  using L = GemmSmem<BN, MODE>;
  constexpr int GB_S = GemmCfg<MODE>::kS;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  GemmBars* bars = reinterpret_cast<GemmBars*>(sm + L::kBar);
  volatile int* abort = &bars->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const WaitCtl& wc = p.wc;

  const int tiles_mn = p.tiles_m * p.tiles_n;
  const long long total = static_cast<long long>(tiles_mn) * p.batch * p.ksplit;
  // tile t: n fastest, then m, then batch, then the K split
  auto decode = [&](long long t, int& mt, int& nt, int& bt, int& ks) {
    nt = static_cast<int>(t % p.tiles_n);
    mt = static_cast<int>((t / p.tiles_n) % p.tiles_m);
    bt = static_cast<int>((t / tiles_mn) % p.batch);
    ks = static_cast<int>(t / (static_cast<long long>(tiles_mn) * p.batch));
  };
  auto kstages = [&](int ks) {
    const int kb = ks * p.kchunk, ke = min(p.K, kb + p.kchunk);
    return (ke - kb + GB_K - 1) / GB_K;
  };

  if (threadIdx.x == 0) {
    for (int i = 0; i < GB_S; ++i) {
      mbar_init(&bars->full[i], 1);
      mbar_init(&bars->empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->acc_full[i], 1);
      mbar_init(&bars->acc_empty[i], GemmCfg<MODE>::kEpi * 32);
    }
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
      prefetch_tmap(&tm_a);
      prefetch_tmap(&tm_b);
      int stage = 0, phase = 0;
      for (long long t = blockIdx.x; t < total && !*abort; t += gridDim.x) {
        int mt, nt, bt, ks;
        decode(t, mt, nt, bt, ks);
        const int ns = kstages(ks);
        const int m0 = mt * GB_M, n0 = nt * BN;
        bool go = true;
        for (int kk = 0; kk < ns; ++kk) {
          if (!mbar_wait(&bars->empty[stage], phase ^ 1, wc, abort)) { go = false; break; }
          const int k0 = ks * p.kchunk + kk * GB_K;
          uint8_t* sa = sm + stage * L::kStage;
          uint8_t* sb = sa + L::kA;
          mbar_expect_tx(&bars->full[stage], L::kStage);
          if constexpr (A_MN) {  // A stored [K][M]: two 64-wide M blocks
            tma_load_3d(sa, &tm_a, &bars->full[stage], m0, k0, bt);
            tma_load_3d(sa + 64 * 128, &tm_a, &bars->full[stage], m0 + 64, k0, bt);
          } else {
            tma_load_3d(sa, &tm_a, &bars->full[stage], k0, m0, bt);
          }
          if constexpr (MODE == kGated || MODE == kGateBwd) {  // the four branch blocks of channels [64 nt, 64 nt + 64), or g
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int col = nt < p.gated_tiles ? j * p.Ch + 64 * nt : 4 * p.Ch + 256 * (nt - p.gated_tiles) + 64 * j;
              tma_load_3d(sb + j * 64 * 128, &tm_b, &bars->full[stage], col, k0, bt);
            }
          } else if constexpr (B_MN) {  // B stored [K][N]: BN / 64 blocks of 64 N
#pragma unroll
            for (int j = 0; j < BN / 64; ++j) tma_load_3d(sb + j * 64 * 128, &tm_b, &bars->full[stage], n0 + 64 * j, k0, bt);
          } else {
            tma_load_3d(sb, &tm_b, &bars->full[stage], k0, n0, bt);
          }
          if (++stage == GB_S) { stage = 0; phase ^= 1; }
        }
        if (!go) break;
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc = idesc_bf16_f32(GB_M, BN, A_MN ? 1 : 0, B_MN ? 1 : 0);
    int stage = 0, phase = 0, local = 0;
    bool ok = true;
    for (long long t = blockIdx.x; t < total && ok; t += gridDim.x, ++local) {
      int mt, nt, bt, ks;
      decode(t, mt, nt, bt, ks);
      const int ns = kstages(ks);
      const int ab = local & 1;
      // the epilogue has read this accumulator's previous tile (parity 1 passes at first)
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->acc_empty[ab], ((local >> 1) & 1) ^ 1, wc, abort))) break;
      tc_fence_after();
      for (int kk = 0; kk < ns; ++kk) {
        if (!__all_sync(0xffffffffu, mbar_wait(&bars->full[stage], phase, wc, abort))) { ok = false; break; }
        tc_fence_after();
        const uint32_t sa = smem_u32(sm + stage * L::kStage), sb = sa + L::kA;
        if (elect_one()) {
#pragma unroll
          for (int k16 = 0; k16 < GB_K / 16; ++k16) {
            // K-major: the next 16 K columns are 32 bytes further along each
            // swizzled 128-byte row; MN-major: 16 K rows of 128 bytes further
            const uint64_t da = A_MN ? smem_desc(sa + k16 * 2048, 64 * 128, 1024, 2) : smem_desc(sa + k16 * 32, 16, 1024, 2);
            const uint64_t db = B_MN ? smem_desc(sb + k16 * 2048, 64 * 128, 1024, 2) : smem_desc(sb + k16 * 32, 16, 1024, 2);
            mma_ss(tmem + ab * BN, da, db, idesc, (kk > 0 || k16 > 0) ? 1u : 0u);
          }
          mma_commit(&bars->empty[stage]);
          if (kk == ns - 1) mma_commit(&bars->acc_full[ab]);
        }
        __syncwarp();
        if (++stage == GB_S) { stage = 0; phase ^= 1; }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 2-5)
    // Each warp owns 32 accumulator rows (its TMEM lane quarter).  Per
    // 32-column chunk a lane converts its row, writes it into a swizzled
    // staging buffer (64-byte rows for BF16, 128-byte rows for FP32), and one
    // lane stores the 32 x 32 block with TMA (rows and columns past the
    // matrix are clipped by the tensor map); two buffers per warp.
    constexpr int kBuf = GemmCfg<MODE>::kBuf;
    const int quarter = warp & 3;       // TMEM lanes a warp may read: 32 * (warp id mod 4) on
    const int part = (warp - 2) >> 2;   // gated tiles: (branch, chunk) unit; plain: column range
    const int r = quarter * 32 + lane;  // accumulator row = TMEM lane
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const bool f32 = p.partial || p.c_f32;
    uint8_t* stg = sm + L::kStg + (warp - 2) * (2 * kBuf);
    int nst = 0;  // TMA stores issued by this warp
    // the next staging buffer, once the store that last used it has read it
    auto next_buf = [&]() -> uint8_t* {
      uint8_t* buf = stg + (nst & 1) * kBuf;
      if (lane == 0) bulk_wait_read_allow1();
      __syncwarp();
      return buf;
    };
    // one accumulator row of 32 FP32 values as BF16 into a 64-byte-swizzled 32 x 32 block
    auto put_bf16 = [&](uint8_t* buf, const uint32_t (&v)[32]) {
      uint32_t w[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) w[e] = pack_bf16x2(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]));
#pragma unroll
      for (int c = 0; c < 4; ++c)
        *reinterpret_cast<uint4*>(buf + lane * 64 + ((c ^ ((lane >> 1) & 3)) << 4)) =
            make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
    };
    auto issue = [&](const CUtensorMap* map, uint8_t* buf, int x, int y, int z) {
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) tma_store_3d(map, buf, x, y, z);
      ++nst;
    };
    // heads epilogue: 32 columns from `col` of this warp's 32 rows (pairs
    // m0 .. m0 + 31, consecutive j of one (b, i)), routed to the core's layout
    // or to the bias planes
    auto heads_chunk = [&](int m0, int col, const uint32_t (&v)[32]) {
      if (m0 >= p.M) return;
      const int bi = m0 / p.Ntok, j0 = m0 - bi * p.Ntok;
      const int HD = p.H * p.D, nh = p.nblk * HD;
      if (col < nh) {
        uint8_t* buf = next_buf();
        if (p.D == 32) {  // one head (H D is a multiple of 32): 32 x 64-byte rows, 64-byte swizzle
          const int t = col / HD, h = (col - t * HD) / 32;
          put_bf16(buf, v);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_5d_nc(&tm_c, buf, 0, j0, h, bi, t);
            bulk_commit();
          }
        } else {  // two 16-column halves, each one head of 16 features (of its own block: H D may be
                  // an odd multiple of 16), as 32 x 32-byte blocks without swizzle; an upper half past
                  // the head columns is bias
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            uint32_t w[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
              w[e] = pack_bf16x2(__uint_as_float(v[16 * hf + 2 * e]), __uint_as_float(v[16 * hf + 2 * e + 1]));
            uint4* row = reinterpret_cast<uint4*>(buf + hf * 1024 + lane * 32);
            row[0] = make_uint4(w[0], w[1], w[2], w[3]);
            row[1] = make_uint4(w[4], w[5], w[6], w[7]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
              const int ch = col + 16 * hf;
              if (ch < nh) {
                const int th = ch / HD;
                tma_store_5d_nc(&tm_c, buf + hf * 1024, 0, j0, (ch - th * HD) / 16, bi, th);
              }
            }
            bulk_commit();
          }
        }
        ++nst;
        if (col + 32 <= nh) return;  // else the chunk's upper half holds bias columns
      }
      // bias columns [nh, nh + nbias) of this chunk: one 32-element row per head
      const int c_lo = max(col, nh), c_hi = min(col + 32, nh + p.nbias);
      if (c_lo >= c_hi) return;
      // the chunk row-major (64-byte swizzled rows) in one staging buffer,
      // then each bias column as one 32-pair row in the other, 16 rows at a
      // time at a 128-byte pitch (TMA sources are 128-byte aligned)
      uint8_t* buf = next_buf();
      put_bf16(buf, v);
      ++nst;
      uint8_t* rows = stg + (nst & 1) * kBuf;
      const int b = bi / p.Ntok, i = bi - b * p.Ntok;
      for (int cs = c_lo; cs < c_hi; cs += 16) {
        const int ce = min(cs + 16, c_hi);
        if (lane == 0) bulk_wait_read();  // every earlier store has read its buffer
        __syncwarp();
        for (int c = cs; c < ce; ++c) {
          const int e = c - col;
          *reinterpret_cast<uint16_t*>(rows + (c - cs) * 128 + lane * 2) =
              *reinterpret_cast<const uint16_t*>(buf + lane * 64 + (((e >> 3) ^ ((lane >> 1) & 3)) << 4) + (e & 7) * 2);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          for (int c = cs; c < ce; ++c) tma_store_4d_nc(&tm_x, rows + (c - cs) * 128, j0, i, c - nh, b);
          bulk_commit();
        }
      }
      ++nst;
    };
    // A gated tile: accumulator columns [a_v | a_g | b_v | b_g] of channels
    // [64 nt, 64 nt + 64).  The four warps of a TMEM lane quarter take one
    // (branch, 32-channel chunk) unit each; a warp's 32 rows are 32
    // consecutive pairs of one example (N*N is a multiple of 32).  With
    // sigmoid(x) = (1 + tanh(x / 2)) / 2:  m sigmoid(g) v = h + h tanh(g / 2),
    // h = m v / 2;  its derivatives are m sigmoid(g) (value) and
    // m v (1 - tanh(g / 2)^2) / 4 (gate).
    const int unit_br = part >> 1, unit_c0 = 32 * (part & 1);
    auto unit_rows = [&](int mt) { return static_cast<long long>(mt) * GB_M + quarter * 32; };
    // gate bwd: this lane's 32 values of dA or dB (BF16 pairs), loaded before
    // the accumulator wait
    auto load_d = [&](int mt, int nt, uint32_t (&d)[16]) {
      const long long mq = unit_rows(mt);
      const int ch = 64 * nt + unit_c0;
      if (mq >= p.M || ch >= p.Ch) return;
      const long long bq = mq / p.NN, pos0 = mq % p.NN;
      const uint16_t* src = (unit_br ? p.dB : p.dA) + (bq * p.Ch + ch) * p.NN + pos0 + lane;
#pragma unroll
      for (int e = 0; e < 16; ++e)
        d[e] = static_cast<uint32_t>(src[2 * e * p.NN]) | (static_cast<uint32_t>(src[(2 * e + 1) * p.NN]) << 16);
    };
    auto gated_tile = [&](int mt, int nt, int ab, const uint32_t (&d)[16]) {
      const long long mq = unit_rows(mt);
      const int ch = 64 * nt + unit_c0;
      if (mq >= p.M || ch >= p.Ch) return;
      const int bq = static_cast<int>(mq / p.NN);
      const int pos0 = static_cast<int>(mq % p.NN);
      const float mk = p.mask != nullptr ? bf16lo_to_f32(p.mask[mq + lane]) : 1.f;
      const uint32_t tv = tmem + lane_addr + ab * BN + 128 * unit_br + unit_c0;  // value columns; gate at +64
      if constexpr (MODE == kGated) {
        // channel rows of 32 pairs (64 bytes, no swizzle), stored channel-major
        uint8_t* buf = next_buf();
        uint16_t* hb = reinterpret_cast<uint16_t*>(buf);
        const float hm = 0.5f * mk;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t v[16], gv[16];
          tmem_ld16x2_wait(tv + 16 * hf, v, tv + 64 + 16 * hf, gv);
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float h = hm * __uint_as_float(v[e]);
            const float o = fmaf(h, tanh_approx(0.5f * __uint_as_float(gv[e])), h);
            hb[(16 * hf + e) * 32 + lane] = static_cast<uint16_t>(pack_bf16x2(o, 0.f) & 0xFFFFu);
          }
        }
        issue(unit_br ? &tm_y : &tm_x, buf, pos0, ch, bq);
      } else {
        // the value and gate blocks in the warp's two buffers
        if (lane == 0) bulk_wait_read();  // every earlier store has read its buffer
        __syncwarp();
        uint8_t* bval = stg;
        uint8_t* bgate = stg + kBuf;
        // 8 columns (one 16-byte chunk of each 64-byte-swizzled block) at a time
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t v[8], gv[8], wv[4], wg[4];
          tmem_ld8x2_wait(tv + 8 * c, v, tv + 64 + 8 * c, gv);
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            float dv2[2], dg2[2];
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              const uint32_t dw = d[4 * c + (e >> 1)];
              const float dd = (k ? bf16hi_to_f32(dw) : bf16lo_to_f32(dw)) * mk;
              const float t = tanh_approx(0.5f * __uint_as_float(gv[e + k]));
              dv2[k] = dd * fmaf(0.5f, t, 0.5f);
              dg2[k] = (0.25f * dd * __uint_as_float(v[e + k])) * fmaf(-t, t, 1.f);
            }
            wv[e >> 1] = pack_bf16x2(dv2[0], dv2[1]);
            wg[e >> 1] = pack_bf16x2(dg2[0], dg2[1]);
          }
          const int off = lane * 64 + ((c ^ ((lane >> 1) & 3)) << 4);
          *reinterpret_cast<uint4*>(bval + off) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
          *reinterpret_cast<uint4*>(bgate + off) = make_uint4(wg[0], wg[1], wg[2], wg[3]);
        }
        issue(&tm_c, bval, 2 * unit_br * p.Ch + ch, static_cast<int>(mq), 0);
        issue(&tm_c, bgate, (2 * unit_br + 1) * p.Ch + ch, static_cast<int>(mq), 0);
      }
    };
    int local = 0;
    for (long long t = blockIdx.x; t < total; t += gridDim.x, ++local) {
      int mt, nt, bt, ks;
      decode(t, mt, nt, bt, ks);
      const int ab = local & 1;
      uint32_t dpre[16];
      if constexpr (MODE == kGateBwd) load_d(mt, nt, dpre);
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->acc_full[ab], (local >> 1) & 1, wc, abort))) break;
      tc_fence_after();
      if constexpr (MODE == kGated || MODE == kGateBwd) {
        if (nt < p.gated_tiles) {
          gated_tile(mt, nt, ab, dpre);
          tc_fence_before();
          mbar_arrive(&bars->acc_empty[ab]);
          continue;
        }
      }
      const int m0 = mt * GB_M + quarter * 32;
      const int n0 = (MODE == kGated ? nt - p.gated_tiles : nt) * BN;
      const int zc = p.partial ? ks * p.batch + bt : bt;
      constexpr int kCols = BN * 4 / GemmCfg<MODE>::kEpi;  // columns per warp of a plain tile
#pragma unroll 1
      for (int c0 = part * kCols; c0 < (part + 1) * kCols; c0 += 32) {
        uint32_t v[32];
        tmem_ld32_wait(tmem + lane_addr + ab * BN + c0, v);
        if (n0 + c0 >= p.N) continue;  // the whole chunk is past N (the same for every lane)
        if constexpr (MODE == kHeads) {
          heads_chunk(m0, n0 + c0, v);
          continue;
        }
        uint8_t* buf = next_buf();
        if (f32) {
#pragma unroll
          for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4*>(buf + sw128(lane, c)) = make_uint4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
        } else {
          put_bf16(buf, v);
        }
        issue(&tm_c, buf, n0 + c0, m0, zc);
      }
      (void)r;
      tc_fence_before();
      mbar_arrive(&bars->acc_empty[ab]);
    }
    if (lane == 0) bulk_wait_all();  // the last stores have landed before the kernel ends
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// out[b][m][n] = sum over ks ascending of part[ks][b][m][n], in FP32, stored
// BF16 or FP32 with row stride ldc and batch stride strideC.
__global__ void __launch_bounds__(256) gemm_splitk_reduce_kernel(const float* __restrict__ part, int ksplit, int batch,
                                                                 int M, int N, void* __restrict__ C, long long ldc,
                                                                 long long strideC, int c_f32) {
  const long long n_el = static_cast<long long>(batch) * M * N;
  for (long long e = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; e < n_el;
       e += static_cast<long long>(gridDim.x) * blockDim.x) {
    float acc = part[e];
    for (int k = 1; k < ksplit; ++k) acc += part[static_cast<long long>(k) * n_el + e];
    const int n = static_cast<int>(e % N);
    const long long m = (e / N) % M, b = e / (static_cast<long long>(N) * M);
    const long long o = b * strideC + m * ldc + n;
    if (c_f32) static_cast<float*>(C)[o] = acc;
    else static_cast<uint16_t*>(C)[o] = static_cast<uint16_t>(pack_bf16x2(acc, 0.f) & 0xFFFFu);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 gemm_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// 3-D map over [batch][rows][ld] BF16 (inner extent `inner` of each row),
// box = box_inner x box_rows, 128-byte swizzle.
bool gemm_map(CUtensorMap* m, const void* base, long long inner, long long rows, int batch, long long ld,
              long long stride, unsigned box_inner, unsigned box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = gemm_encoder();
  if (enc == nullptr) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(batch)};
  const long long bs = batch > 1 ? stride : rows * ld;
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld) * 2, static_cast<cuuint64_t>(bs) * 2};
  const cuuint32_t box[3] = {box_inner, box_rows, 1u};
  const cuuint32_t es[3] = {1u, 1u, 1u};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Output map: [planes][M][ld] BF16 (64-byte swizzle) or FP32 (128-byte
// swizzle), box = 32 columns x 32 rows.
bool gemm_out_map(CUtensorMap* m, void* base, long long N, long long M, long long planes, long long ld,
                  long long stride, bool f32) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = gemm_encoder();
  if (enc == nullptr) return false;
  const int esz = f32 ? 4 : 2;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(M), static_cast<cuuint64_t>(planes)};
  const long long bs = planes > 1 ? stride : M * ld;
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld) * esz, static_cast<cuuint64_t>(bs) * esz};
  const cuuint32_t box[3] = {32u, 32u, 1u};
  const cuuint32_t es[3] = {1u, 1u, 1u};
  return enc(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, f32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN, bool A_MN, bool B_MN, int MODE = kPlain>
cudaError_t gemm_launch_t(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc, const CUtensorMap& tx,
                          const CUtensorMap& ty, const GemmParams& p, int grid, cudaStream_t s) {
  using L = GemmSmem<BN, MODE>;
  static std::once_flag once;
  static cudaError_t attr = cudaSuccess;
  std::call_once(once, [] {
    attr = cudaFuncSetAttribute(gemm_kernel<BN, A_MN, B_MN, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                L::kBytes);
  });
  if (attr != cudaSuccess) return attr;
  gemm_kernel<BN, A_MN, B_MN, MODE><<<grid, GemmCfg<MODE>::kThreads, L::kBytes, s>>>(ta, tb, tc, tx, ty, p);
  return cudaGetLastError();
}
template <int BN, bool A_MN, bool B_MN>
cudaError_t gemm_launch_t(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc, const GemmParams& p,
                          int grid, cudaStream_t s) {
  return gemm_launch_t<BN, A_MN, B_MN, kPlain>(ta, tb, tc, tc, tc, p, grid, s);
}

int gemm_sms() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 148;
  return sms;
}

struct SplitPlan {
  int ksplit, kchunk;
};
// Split K only when the output tiles cannot fill the GPU: enough splits to
// give every SM a tile, each at least 8 stages deep.
SplitPlan split_plan(int M, int N, int K, int batch, int BN, int sms) {
  const long long tiles = static_cast<long long>(batch) * ((M + GB_M - 1) / GB_M) * ((N + BN - 1) / BN);
  int ks = 1;
  if (tiles < sms) ks = static_cast<int>(std::min<long long>((sms + tiles - 1) / tiles, std::max(1, K / (8 * GB_K))));
  int kchunk = (K + ks - 1) / ks;
  kchunk = (kchunk + GB_K - 1) / GB_K * GB_K;
  ks = (K + kchunk - 1) / kchunk;
  return {ks, kchunk};
}

}  // namespace

size_t gemm_splitk_bytes(int M, int N, int K, int batch) {
  const int BN = N > 128 ? 256 : 128;
  const SplitPlan sp = split_plan(M, N, K, batch, BN, gemm_sms());
  return sp.ksplit > 1 ? static_cast<size_t>(sp.ksplit) * batch * M * N * 4 : 0;
}

cudaError_t launch_gemm(bool ta, bool tb, int M, int N, int K, const void* A, long long lda, const void* B,
                        long long ldb, void* C, long long ldc, bool c_f32, int batch, long long sA, long long sB,
                        long long sC, void* ws, size_t ws_bytes, const WaitCtl& wc, cudaStream_t s) {
  if (M < 1 || N < 1 || K < 1 || batch < 1) return cudaErrorInvalidValue;
  // TMA: 16-byte aligned bases and row strides
  if ((reinterpret_cast<uintptr_t>(A) & 15u) || (reinterpret_cast<uintptr_t>(B) & 15u) || (lda & 7) || (ldb & 7) ||
      (batch > 1 && ((sA & 7) || (sB & 7))))
    return cudaErrorInvalidValue;
  const int BN = N > 128 ? 256 : 128;
  const int sms = gemm_sms();
  SplitPlan sp = split_plan(M, N, K, batch, BN, sms);
  const size_t need = static_cast<size_t>(sp.ksplit) * batch * M * N * 4;
  if (sp.ksplit > 1 && (ws == nullptr || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 15u) || (N & 3))) {
    sp.ksplit = 1;
    sp.kchunk = (K + GB_K - 1) / GB_K * GB_K;
  }
  // the epilogue's vector stores need 16-byte aligned rows
  if (sp.ksplit == 1 && ((reinterpret_cast<uintptr_t>(C) & 15u) || (ldc & (c_f32 ? 3 : 7)) ||
                         (batch > 1 && (sC & (c_f32 ? 3 : 7)))))
    return cudaErrorInvalidValue;
  CUtensorMap tma, tmb;
  const bool okA = ta ? gemm_map(&tma, A, M, K, batch, lda, sA, 64, 64) : gemm_map(&tma, A, K, M, batch, lda, sA, 64, 128);
  const bool okB = tb ? gemm_map(&tmb, B, K, N, batch, ldb, sB, 64, static_cast<unsigned>(BN))
                      : gemm_map(&tmb, B, N, K, batch, ldb, sB, 64, 64);
  CUtensorMap tmc;
  const bool okC = sp.ksplit > 1 ? gemm_out_map(&tmc, ws, N, M, static_cast<long long>(sp.ksplit) * batch, N,
                                                static_cast<long long>(M) * N, true)
                                 : gemm_out_map(&tmc, C, N, M, batch, ldc, sC, c_f32);
  if (!okA || !okB || !okC) return cudaErrorInvalidValue;
  GemmParams p;
  p.M = M;
  p.N = N;
  p.K = K;
  p.batch = batch;
  p.ksplit = sp.ksplit;
  p.kchunk = sp.kchunk;
  p.tiles_m = (M + GB_M - 1) / GB_M;
  p.tiles_n = (N + BN - 1) / BN;
  p.partial = sp.ksplit > 1 ? 1 : 0;
  p.C = p.partial ? ws : C;
  p.ldc = ldc;
  p.strideC = sC;
  p.c_f32 = c_f32 ? 1 : 0;
  p.Ch = 0;
  p.gated_tiles = 0;
  p.NN = 1;
  p.mask = p.dA = p.dB = nullptr;
  p.wc = wc;
  const long long total = static_cast<long long>(p.tiles_m) * p.tiles_n * batch * sp.ksplit;
  const int grid = static_cast<int>(std::min<long long>(total, sms));
  const bool amn = ta, bmn = !tb;  // [K][M] A, [K][N] B: M / N contiguous
  cudaError_t e;
  if (BN == 256) {
    if (amn) e = bmn ? gemm_launch_t<256, true, true>(tma, tmb, tmc, p, grid, s) : gemm_launch_t<256, true, false>(tma, tmb, tmc, p, grid, s);
    else e = bmn ? gemm_launch_t<256, false, true>(tma, tmb, tmc, p, grid, s) : gemm_launch_t<256, false, false>(tma, tmb, tmc, p, grid, s);
  } else {
    if (amn) e = bmn ? gemm_launch_t<128, true, true>(tma, tmb, tmc, p, grid, s) : gemm_launch_t<128, true, false>(tma, tmb, tmc, p, grid, s);
    else e = bmn ? gemm_launch_t<128, false, true>(tma, tmb, tmc, p, grid, s) : gemm_launch_t<128, false, false>(tma, tmb, tmc, p, grid, s);
  }
  if (e != cudaSuccess || !p.partial) return e;
  const long long n_el = static_cast<long long>(batch) * M * N;
  const unsigned blocks = static_cast<unsigned>(std::min<long long>((n_el + 255) / 256, static_cast<long long>(sms) * 16));
  gemm_splitk_reduce_kernel<<<blocks, 256, 0, s>>>(static_cast<const float*>(ws), sp.ksplit, batch, M, N, C, ldc,
                                                   batch > 1 ? sC : 0, c_f32 ? 1 : 0);
  return cudaGetLastError();
}

namespace {
// Channel-major output map: [B][C_h][N*N] BF16, box = 32 pairs x 32 channels,
// no swizzle (the staging block holds channel rows of 64 bytes).
bool gemm_cm_map(CUtensorMap* m, void* base, long long NN, int Ch, int B) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = gemm_encoder();
  if (enc == nullptr) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(NN), static_cast<cuuint64_t>(Ch), static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(NN) * 2, static_cast<cuuint64_t>(NN) * Ch * 2};
  const cuuint32_t box[3] = {32u, 32u, 1u};
  const cuuint32_t es[3] = {1u, 1u, 1u};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool al16p(const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; }

// The gated tiles' common parameters and operand maps (x [M][C_z] K-major,
// W_p [C_z][4 C_h + C_z] N-major).
bool gated_setup(int B, long long NN, int Cz, int Ch, const void* x, const void* w_p, const void* mask,
                 CUtensorMap* tma, CUtensorMap* tmb, GemmParams* p) {
  const long long M = B * NN;
  if (B < 1 || NN < 32 || NN % 32 != 0 || M > 0x7fffffffLL || Cz < 32 || Cz % 32 != 0 || Ch < 32 || Ch % 32 != 0 ||
      !al16p(x) || !al16p(w_p) || (mask != nullptr && !al16p(mask)))
    return false;
  const int F = 4 * Ch + Cz;
  if (!gemm_map(tma, x, Cz, M, 1, Cz, 0, 64, 128) || !gemm_map(tmb, w_p, F, Cz, 1, F, 0, 64, 64)) return false;
  p->M = static_cast<int>(M);
  p->K = Cz;
  p->batch = 1;
  p->ksplit = 1;
  p->kchunk = (Cz + GB_K - 1) / GB_K * GB_K;
  p->tiles_m = static_cast<int>((M + GB_M - 1) / GB_M);
  p->partial = 0;
  p->c_f32 = 0;
  p->ldc = 0;
  p->strideC = 0;
  p->Ch = Ch;
  p->gated_tiles = (Ch + 63) / 64;
  p->NN = NN;
  p->mask = static_cast<const uint16_t*>(mask);
  p->dA = p->dB = nullptr;
  return true;
}
}  // namespace

cudaError_t launch_gated_proj(int B, long long NN, int Cz, int Ch, const void* x, const void* w_p, const void* mask,
                              void* a, void* b, void* g, const WaitCtl& wc, cudaStream_t s) {
  CUtensorMap tma, tmb, tmc, tmx, tmy;
  GemmParams p;
  if (!gated_setup(B, NN, Cz, Ch, x, w_p, mask, &tma, &tmb, &p) || !al16p(a) || !al16p(b) || !al16p(g))
    return cudaErrorInvalidValue;
  const long long M = B * NN;
  if (!gemm_out_map(&tmc, g, Cz, M, 1, Cz, 0, false) || !gemm_cm_map(&tmx, a, NN, Ch, B) ||
      !gemm_cm_map(&tmy, b, NN, Ch, B))
    return cudaErrorInvalidValue;
  p.N = Cz;  // the g tiles' columns
  p.tiles_n = p.gated_tiles + (Cz + 255) / 256;
  p.C = g;
  p.wc = wc;
  const long long total = static_cast<long long>(p.tiles_m) * p.tiles_n;
  const int grid = static_cast<int>(std::min<long long>(total, gemm_sms()));
  return gemm_launch_t<256, false, true, kGated>(tma, tmb, tmc, tmx, tmy, p, grid, s);
}

cudaError_t launch_gate_bwd_proj(int B, long long NN, int Cz, int Ch, const void* x, const void* w_p,
                                 const void* mask, const void* dA, const void* dB, void* dp, long long ldp,
                                 const WaitCtl& wc, cudaStream_t s) {
  CUtensorMap tma, tmb, tmc;
  GemmParams p;
  if (!gated_setup(B, NN, Cz, Ch, x, w_p, mask, &tma, &tmb, &p) || !al16p(dA) || !al16p(dB) || !al16p(dp) ||
      ldp < 4 * Ch || ldp % 8 != 0)
    return cudaErrorInvalidValue;
  const long long M = B * NN;
  if (!gemm_out_map(&tmc, dp, 4 * Ch, M, 1, ldp, 0, false)) return cudaErrorInvalidValue;
  p.N = 4 * Ch;
  p.tiles_n = p.gated_tiles;
  p.C = dp;
  p.dA = static_cast<const uint16_t*>(dA);
  p.dB = static_cast<const uint16_t*>(dB);
  p.wc = wc;
  const long long total = static_cast<long long>(p.tiles_m) * p.tiles_n;
  const int grid = static_cast<int>(std::min<long long>(total, gemm_sms()));
  return gemm_launch_t<256, false, true, kGateBwd>(tma, tmb, tmc, tmc, tmc, p, grid, s);
}

cudaError_t launch_gemm_heads(bool tb, int M, int N, int K, const void* A, long long lda, const void* B, long long ldb,
                              int nblk, int H, int D, int Ntok, int Bx, void* heads, void* bias_planes, int nbias,
                              const WaitCtl& wc, cudaStream_t s) {
  if (M < 1 || N < 1 || K < 1 || (D != 16 && D != 32) || H < 1 || nblk < 1 || Ntok < 32 || Ntok % 32 != 0 ||
      static_cast<long long>(Bx) * Ntok * Ntok != M || nblk * H * D + nbias > N || (nbias > 0 && bias_planes == nullptr))
    return cudaErrorInvalidValue;
  if (!al16p(A) || !al16p(B) || !al16p(heads) || (bias_planes != nullptr && !al16p(bias_planes)) || (lda & 7) ||
      (ldb & 7))
    return cudaErrorInvalidValue;
  PFN_cuTensorMapEncodeTiled_v12000 enc = gemm_encoder();
  if (enc == nullptr) return cudaErrorInvalidValue;
  const int BN = N > 128 ? 256 : 128;
  CUtensorMap tma, tmb, tmc, tmx;
  const bool okA = gemm_map(&tma, A, K, M, 1, lda, 0, 64, 128);
  const bool okB = tb ? gemm_map(&tmb, B, K, N, 1, ldb, 0, 64, static_cast<unsigned>(BN))
                      : gemm_map(&tmb, B, N, K, 1, ldb, 0, 64, 64);
  if (!okA || !okB) return cudaErrorInvalidValue;
  {  // heads: [nblk][B*Ntok (b, i)][H][Ntok (j)][D], box D x 32 rows of one (b, i, h, t)
    const cuuint64_t dims[5] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(Ntok), static_cast<cuuint64_t>(H),
                                static_cast<cuuint64_t>(Bx) * Ntok, static_cast<cuuint64_t>(nblk)};
    const cuuint64_t row = static_cast<cuuint64_t>(D) * 2, head = row * Ntok, slice = head * H,
                     blk = slice * Bx * Ntok;
    const cuuint64_t strides[4] = {row, head, slice, blk};
    const cuuint32_t box[5] = {static_cast<cuuint32_t>(D), 32u, 1u, 1u, 1u};
    const cuuint32_t es[5] = {1u, 1u, 1u, 1u, 1u};
    if (enc(&tmc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, heads, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            D == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  tmx = tmc;
  if (nbias > 0) {  // bias planes [B][H][Ntok (i)][Ntok (j)], box 32 j of one (b, h, i)
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(Ntok), static_cast<cuuint64_t>(Ntok),
                                static_cast<cuuint64_t>(nbias), static_cast<cuuint64_t>(Bx)};
    const cuuint64_t row = static_cast<cuuint64_t>(Ntok) * 2, plane = row * Ntok, ex = plane * nbias;
    const cuuint64_t strides[3] = {row, plane, ex};
    const cuuint32_t box[4] = {32u, 1u, 1u, 1u};
    const cuuint32_t es[4] = {1u, 1u, 1u, 1u};
    if (enc(&tmx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, bias_planes, dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  GemmParams p;
  std::memset(&p, 0, sizeof(p));
  p.M = M;
  p.N = N;
  p.K = K;
  p.batch = 1;
  p.ksplit = 1;
  p.kchunk = (K + GB_K - 1) / GB_K * GB_K;
  p.tiles_m = (M + GB_M - 1) / GB_M;
  p.tiles_n = (N + BN - 1) / BN;
  p.NN = 1;
  p.nblk = nblk;
  p.H = H;
  p.D = D;
  p.Ntok = Ntok;
  p.nbias = nbias;
  p.wc = wc;
  const long long total = static_cast<long long>(p.tiles_m) * p.tiles_n;
  const int grid = static_cast<int>(std::min<long long>(total, gemm_sms()));
  const bool bmn = !tb;
  if (BN == 256)
    return bmn ? gemm_launch_t<256, false, true, kHeads>(tma, tmb, tmc, tmx, tmx, p, grid, s)
               : gemm_launch_t<256, false, false, kHeads>(tma, tmb, tmc, tmx, tmx, p, grid, s);
  return bmn ? gemm_launch_t<128, false, true, kHeads>(tma, tmb, tmc, tmx, tmx, p, grid, s)
             : gemm_launch_t<128, false, false, kHeads>(tma, tmb, tmc, tmx, tmx, p, grid, s);
}

}  // namespace triattn
