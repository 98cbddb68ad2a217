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
#include <algorithm>

#include "kernels.cuh"

namespace triattn {

namespace {

constexpr int BM = kTileQ;   // query rows per tile
constexpr int BN = kTileK;   // keys per CTA (TMEM lanes of S^T, dP^T, dK, dV)
constexpr float kLog2e = 1.4426950408889634f;
// Per query row the backward keeps an 8-wide BF16 record
//   [x0, x1, x2, 0, y0, y1, y2, 0],  x0 + x1 + x2 = -lse sqrt(D),  y0 + y1 + y2 = -delta
// (each value split into three BF16 terms, together about FP32 precision).
// It is the B operand of one extra K = 16 step of the S^T and dP^T MMAs,
// whose A operand is a constant [1, 1, 1, 0, 0, 0, 0, 0] (S^T) or
// [0, 0, 0, 0, 1, 1, 1, 0] (dP^T) per key, with the upper 8 K columns zero,
// so the tensor core adds -lse sqrt(D) to every score and -delta to every
// dP value of the query.  A row without any key gets x0 = -1e30 (P = 0).
constexpr int kRecRow = 16;            // bytes per query row
constexpr int kRecTile = BM * kRecRow;  // bytes per (slice, query tile)
// Stages of the Q / dO / record ring.  A stage is refilled once dK of its
// step is done, and the next-but-one step's S^T needs it: three stages leave
// more than a step of time for the load.
constexpr int NQ = 3;

// ---------------------------------------------------------------- preprocess
// One 16-byte record per query row (rows padded to whole 128-row tiles):
// BF16 [x0 x1 x2 0 y0 y1 y2 0] with x0 + x1 + x2 = -lse[q] sqrt(D) (x0 = -1e30
// for a fully masked row and for q >= N) and y0 + y1 + y2 = -delta[q],
// delta[q] = sum_d dO[q,d] (O[q,d] + E[q,d]) in FP32 (E omitted when null;
// 0 for q >= N).
template <int D>
__global__ void __launch_bounds__(256) preprocess_kernel(const uint16_t* __restrict__ dO,
                                                         const uint16_t* __restrict__ o,
                                                         const uint16_t* __restrict__ e,
                                                         const float* __restrict__ lse, uint4* __restrict__ rec,
                                                         int N, int H, int JQ, size_t padded_rows, RowLayout lo,
                                                         RowLayout ldo) {
  // One 16-byte chunk (8 features) of one row per thread, so that a warp's
  // loads cover consecutive rows contiguously; the D/8 lanes of a row add
  // their partial sums with a fixed butterfly.
  constexpr int kCpr = D / 8;  // chunks per row
  const size_t t = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const size_t pr = t / kCpr;  // (slice * JQ + i) * 128 + qq
  const int c = static_cast<int>(t % kCpr);
  const size_t tile = pr / BM;
  const int qq = static_cast<int>(pr % BM);
  const int i = static_cast<int>(tile % JQ);
  const size_t slice = tile / JQ;
  const int q = i * BM + qq;
  const bool live = pr < padded_rows && q < N;
  float xs = -1e30f, acc = 0.f;
  if (live) {
    const size_t row = slice * N + q;
    const long long bo = static_cast<long long>(slice / H);
    const int hh = static_cast<int>(slice - bo * H);
    const long long off = lo.offset(bo, hh, q);
    const uint4 gw = __ldg(reinterpret_cast<const uint4*>(dO + ldo.offset(bo, hh, q)) + c);
    const uint4 ow = __ldg(reinterpret_cast<const uint4*>(o + off) + c);
    uint4 ew = make_uint4(0, 0, 0, 0);
    if (e != nullptr) ew = __ldg(reinterpret_cast<const uint4*>(e + off) + c);
    const uint32_t g4[4] = {gw.x, gw.y, gw.z, gw.w}, o4[4] = {ow.x, ow.y, ow.z, ow.w},
                   e4[4] = {ew.x, ew.y, ew.z, ew.w};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      acc = fmaf(bf16lo_to_f32(g4[u]), bf16lo_to_f32(o4[u]) + bf16lo_to_f32(e4[u]), acc);
      acc = fmaf(bf16hi_to_f32(g4[u]), bf16hi_to_f32(o4[u]) + bf16hi_to_f32(e4[u]), acc);
    }
    const float l = __ldg(lse + row);
    if (l != -INFINITY) xs = -l * sqrtf(static_cast<float>(D));
  }
#pragma unroll
  for (int off = kCpr / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (pr >= padded_rows || c != 0) return;
  // three-term BF16 splits: v = h + m + lo to about 24 significant bits
  auto split3 = [](float v, uint32_t& w01, uint32_t& w2) {
    const uint32_t h = pack_bf16x2(v, 0.f) & 0xFFFFu;
    const float r1 = v - bf16lo_to_f32(h);
    const uint32_t m = pack_bf16x2(r1, 0.f) & 0xFFFFu;
    const uint32_t lo = pack_bf16x2(r1 - bf16lo_to_f32(m), 0.f) & 0xFFFFu;
    w01 = h | (m << 16);
    w2 = lo;
  };
  uint4 w;
  split3(xs, w.x, w.y);
  split3(-acc, w.z, w.w);
  rec[pr] = w;
}

// biasT[bh][k][q] = bias[bh][q][k]: 64 x 64 tiles through shared memory.
// biasT rows have Np = N rounded up to a multiple of 8 elements (16-byte
// strides for TMA); columns q >= N of a row are written as zeros.  When N is
// a multiple of 8 an 8-element group of a bias row is all inside or all
// outside and moves as one 16-byte load; otherwise elements are read one by
// one (bias rows are then not 16-byte aligned).
__global__ void __launch_bounds__(256) transpose_bias_kernel(const uint16_t* __restrict__ bias,
                                                             uint16_t* __restrict__ biasT, int N, int Np) {
  __shared__ __align__(16) uint16_t tile[64][72];
  const int q0 = blockIdx.y * 64, k0 = blockIdx.x * 64;
  const size_t base = static_cast<size_t>(blockIdx.z) * N * N;
  const size_t baseT = static_cast<size_t>(blockIdx.z) * N * Np;
  const bool vec = (N & 7) == 0;
  for (int e = threadIdx.x; e < 64 * 8; e += blockDim.x) {
    const int rr = e >> 3, c8 = e & 7;
    const int q = q0 + rr, k = k0 + 8 * c8;
    uint4 w = make_uint4(0, 0, 0, 0);
    if (q < N && k < N) {
      const uint16_t* src = bias + base + static_cast<size_t>(q) * N + k;
      if (vec) {
        w = __ldg(reinterpret_cast<const uint4*>(src));
      } else {
        uint32_t h[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) h[j] = k + j < N ? __ldg(src + j) : 0u;
        w = make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16), h[6] | (h[7] << 16));
      }
    }
    *reinterpret_cast<uint4*>(&tile[rr][8 * c8]) = w;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < 64 * 8; e += blockDim.x) {
    const int rr = e >> 3, c8 = e & 7;
    const int k = k0 + rr, q = q0 + 8 * c8;
    if (k >= N || q >= Np) continue;
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      w[j] = static_cast<uint32_t>(tile[8 * c8 + 2 * j][rr]) | (static_cast<uint32_t>(tile[8 * c8 + 2 * j + 1][rr]) << 16);
    *reinterpret_cast<uint4*>(biasT + baseT + static_cast<size_t>(k) * Np + q) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// ---------------------------------------------------------------- main kernel
//
// The tile is held transposed: TMEM lane = key of this CTA's key tile,
// column = query, so P^T and dS^T land in TMEM where the dV and dK MMAs read
// them as their A operand, and the key mask of a slice is one value per thread.
//
// Thread roles (20 warps):
// G = 4 slices per CTA at D = 32, 8 at D = 16 (TMEM: dV and dK of every slice
// in 2 G D columns, S^T and dP^T in 256).
//
//   warp 0       TMA producer: K, V of the G slices once; per query tile one
//                transposed bias tile; per (query tile, slice) the Q and dO
//                tiles and the record of -lse log2 e and -delta.
//   warps 1-3    three tcgen05 MMA issuers (converged warps, one elected lane
//                issues one group per step; descriptors are precomputed).  A
//                single issuing thread spends ~27 cycles per N = 32 MMA and
//                ~100 per group boundary, so the step's 28 MMAs are split:
//                warp 1 (also TMEM owner): dV_g += P^T dO, then S^T(s+1);
//                warp 2: dK_g += dS^T Q, then dP^T(s+1);
//                warp 3: the dQ tile dS K.
//                Each pair stays in one thread, so dV (dK) reads P^T (dS^T)
//                before S^T (dP^T) of the next step overwrites it.
//   warps 4-19   four elementwise warpgroups.  Each covers all 128 TMEM lanes
//                (thread = key row for S^T / dP^T / dK / dV, query row for the
//                dQ tile); warpgroup w handles query columns [32w, 32w + 32).
//
// Per step s = (query tile i, slice g), two elementwise phases:
//   P-phase   P^T = 2^((S^T - lse sqrt(D)) log2e/sqrt(D) + (bias^T + mask) log2e),
//             FP32 P kept in registers, BF16 P^T written into half of the
//             S^T columns the warpgroup has just read.
//   dS-phase  dS^T = P^T (dP^T - delta); dbias accumulator += dS^T (FP32
//             registers); BF16 dS^T into this warpgroup's own dP^T columns
//             and into shared memory (the A operand of the dQ MMA).
// MMA order per step: dV_g += P^T dO (A from TMEM) and S^T(s+1) after the
// P-phase; dK_g += dS^T Q (A from TMEM) and dP^T(s+1) after the dS-phase; the
// dQ tile dS K (into S^T columns [48, 48 + D)) after the dS-phase, once every
// warp has loaded S^T(s+1).  Warpgroup 0 (one warp per TMEM lane quarter)
// stores that dQ tile as soon as it completes; S^T(s+2) waits for that.  dK
// is scaled by 1/sqrt(D) when it leaves TMEM, the dQ tile when it is stored.  After slice
// G-1 of a query tile the FP32 dbias partial of the outer group is written
// once.
template <int D>
struct BwdSmem {
  static constexpr int G = kGroupBwdFor(D);             // outer slices per CTA
  static constexpr int kTile = BM * D * 2;              // 128 rows x D bf16
  static constexpr int kDS = 0;                         // dS^T [2 query blocks][128 k][64 q] bf16, SW128
  static constexpr int kBias = kDS + BN * BM * 2;       // 2 stages of bias^T, same layout
  static constexpr int kK = kBias + 2 * BN * BM * 2;    // G K tiles (stationary)
  static constexpr int kV = kK + G * kTile;             // G V tiles (stationary)
  static constexpr int kQ = kV + G * kTile;             // NQ stages of Q tiles
  static constexpr int kDO = kQ + NQ * kTile;           // NQ stages of dO tiles
  static constexpr int kAugS = kDO + NQ * kTile;        // constant A of the record step of S^T
  static constexpr int kAugP = kAugS + kRecTile;        // constant A of the record step of dP^T
  static constexpr int kRec = kAugP + kRecTile;         // NQ stages of the query-row record
  static constexpr int kZero = kRec + NQ * kRecTile;    // zeros: K columns 8-15 of the record step
  static constexpr int kMask = kZero + kRecTile;        // G x 128 fp32: base-2 key mask
  static constexpr int kBar = kMask + G * BN * 4;
  static constexpr int kBytes = kBar + 256;
  static_assert(kBytes <= 232448, "shared memory budget");
};

constexpr int kNWG = 4;                // elementwise warpgroups
constexpr int kCols = BM / kNWG;       // query columns per warpgroup
constexpr int kEW = 128 * kNWG;        // elementwise threads
constexpr int kMainThreads = 128 + kEW;

struct BwdBars {
  uint64_t kv_full;
  uint64_t qdo_full[NQ], qdo_empty[NQ];
  uint64_t b_full[2], b_empty[2];
  uint64_t s_full, dp_full, s_cons, p_ready, ds_ready, dq_full, dq_read, all_done;
  uint64_t never;  // completes no phase: a parity-1 wait on it always passes
  // bulk-reduction ablation only: the dQ tile staged in shared memory
  // (staged), and its bulk read finished so the staging area is free (stage_free)
  uint64_t staged, stage_free;
  uint32_t tmem_slot;
  int abort;
};

// kAtomic (non-deterministic ablation only; 0 in the product path): bit 0
// adds the dQ tiles into an FP32 [slices][J_Q*128][D] accumulator, bit 1 the
// dbias tiles into an FP32 [B*H][J_K*128 (k)][J_Q*128 (q)] accumulator, with
// FP32 atomics instead of writing single-writer partials; bit 2 adds the dQ
// tiles into the same accumulator with the TMA engine's bulk reduction
// (cp.reduce.async.bulk, this GPU's memory only): warpgroup 0 stages the
// FP32 tile in the dS buffer once the dQ MMA has read it, one thread issues
// the reduction, and the next dS waits until the engine has read the tile.
// HF (the ordered path only): the grid runs heads first, so that the CTAs
// running together read or write neighbouring heads of the same rows --
// chosen when q, k, v, dO or dq, dk, dv have their heads inside their rows
// (RowLayout::hn).  The tensor maps follow lq.hn and ldo.hn.
template <int D, int kAtomic = 0, bool HF = false>
__global__ void __launch_bounds__(kMainThreads, 1)
    bwd_main_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_biasT, const uint16_t* __restrict__ mask,
                    const uint4* __restrict__ rec, uint16_t* __restrict__ dk, uint16_t* __restrict__ dv,
                    float* __restrict__ dq_part, float* __restrict__ dbias_part, int N_o, int N, int H, RowLayout lq,
                    RowLayout ldo, RowLayout lg, WaitCtl wc) {
  using L = BwdSmem<D>;
  constexpr int G = L::G;  // outer slices per CTA
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw;
  BwdBars* bars = reinterpret_cast<BwdBars*>(sm + L::kBar);
  volatile int* abort = &bars->abort;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  // grid (J_K, groups, B * H), or (H * J_K, groups, B) with HF
  const int ktile = HF ? static_cast<int>(blockIdx.x) / H : static_cast<int>(blockIdx.x);
  const int grp = blockIdx.y;
  const int o0 = grp * G;
  const int bh = HF ? static_cast<int>(blockIdx.z) * H + static_cast<int>(blockIdx.x) % H : static_cast<int>(blockIdx.z);
  const int b = bh / H;
  const int h = bh - b * H;
  const int nkt = HF ? static_cast<int>(gridDim.x) / H : static_cast<int>(gridDim.x);  // key tiles
  const int nbh = HF ? static_cast<int>(gridDim.z) * H : static_cast<int>(gridDim.z);  // B * H
  const int JQ = (N + BM - 1) / BM;
  const int nsteps = JQ * G;
  // The last group may extend past N_o: its extra slices see every key
  // masked (P = 0, so they add nothing), their records are read from the
  // last real slice, and nothing of theirs is stored.
  const int last_rec_slice = nbh * N_o - 1;

  // The swizzled tiles below need a 1024-byte aligned base.
  if ((smem_u32(sm) & 1023u) != 0) {
    if (tid == 0) atomicOr(wc.status, 2u);
    return;
  }

  // TMEM columns: dV_g at g*D, dK_g at G*D + g*D, S^T (128), dP^T (128).
  // Warpgroup w reads S^T and dP^T columns [32w, 32w + 32) and writes its
  // BF16 P^T (16 columns) back into half of them: the upper half for w = 0,
  // 2, the lower half for w = 1, 3 (columns 16, 32, 80, 96).  Every column
  // a thread overwrites it has read itself, so no other warp has to be
  // waited for, and S^T columns [48, 80) stay free for the dQ tile (D
  // columns).  BF16 dS^T of warpgroup w goes into dP^T columns [32w, 32w + 16).
  constexpr uint32_t kTS = 2 * G * D;
  constexpr uint32_t kTDP = kTS + 128;
  constexpr uint32_t kTDQ = kTS + 48;
  auto p_col = [](int w) { return static_cast<uint32_t>(16 + 16 * w + 32 * (w >> 1)); };
  static_assert(kTDP + 128 <= 512, "TMEM budget");

  if (tid == 0) {
    mbar_init(&bars->kv_full, 1);
    for (int i = 0; i < NQ; ++i) {
      mbar_init(&bars->qdo_full[i], 1);
      mbar_init(&bars->qdo_empty[i], 2);  // issuers A (S, dV) and C (dP, dK)
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->b_full[i], 1);
      mbar_init(&bars->b_empty[i], kEW);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->s_cons, kEW);
    mbar_init(&bars->p_ready, kEW);
    mbar_init(&bars->ds_ready, kEW);
    mbar_init(&bars->dq_full, 1);
    mbar_init(&bars->dq_read, 128);
    mbar_init(&bars->all_done, 3);
    mbar_init(&bars->never, 1);
    mbar_init(&bars->staged, 128);
    mbar_init(&bars->stage_free, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(&bars->tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_slot;

  // Warpgroup 0 (producer and the three issuers: one warp per TMEM lane
  // quarter) drains each dQ tile: warp w stores rows [32w, 32w + 32), all D
  // columns scaled by 1/sqrt(D), as this key tile's FP32 partial, chunk-major
  // per 128-row tile: [J_K][slices][J_Q][D/8 chunks][128 rows] x 8 floats,
  // with 32-byte stores.  Then S^T(t+2), which overwrites those columns, may
  // be issued.
  auto drain_dq = [&](int t) -> bool {
    if (!__all_sync(0xffffffffu, mbar_wait(&bars->dq_full, t & 1, wc, abort))) return false;
    tc_fence_after();
    const int ti = t / G, tg = t % G;
    const int r = (warp & 3) * 32 + lane;
    const bool live = o0 + tg < N_o;
    const size_t slice = static_cast<size_t>((b * N_o + o0 + tg) * H + h);
    const size_t nslices = static_cast<size_t>(nbh) * N_o;
    float* out = dq_part + ((static_cast<size_t>(ktile) * nslices + slice) * JQ + ti) * (BM * D) + r * 8;
    const uint32_t taddr = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + kTDQ;
    const float isd = rsqrtf(static_cast<float>(D));
    uint32_t qr[D];
    if constexpr (D == 32) tmem_ld32_wait(taddr, qr);
    else tmem_ld16_wait(taddr, qr);
    if (!live) {
      // a padded slice of the last group: nothing to store
    } else if constexpr ((kAtomic & 4) != 0) {
      // FP32 row r of the tile into the staging area (row-major, the
      // accumulator's layout), 16-byte chunks in a rotated order so that a
      // quarter warp's stores hit distinct banks
      uint8_t* stg = sm + L::kDS + r * (D * 4);
#pragma unroll
      for (int cc = 0; cc < D / 4; ++cc) {
        const int c = (cc + r) & (D / 4 - 1);
        *reinterpret_cast<float4*>(stg + c * 16) =
            make_float4(__uint_as_float(qr[4 * c]) * isd, __uint_as_float(qr[4 * c + 1]) * isd,
                        __uint_as_float(qr[4 * c + 2]) * isd, __uint_as_float(qr[4 * c + 3]) * isd);
      }
    } else if constexpr ((kAtomic & 1) != 0) {
      float* acc = dq_part + ((slice * JQ + ti) * BM + r) * D;
#pragma unroll
      for (int c = 0; c < D / 4; ++c)
        red_add_v4(acc + 4 * c, __uint_as_float(qr[4 * c]) * isd, __uint_as_float(qr[4 * c + 1]) * isd,
                   __uint_as_float(qr[4 * c + 2]) * isd, __uint_as_float(qr[4 * c + 3]) * isd);
    } else {
#pragma unroll
      for (int c = 0; c < D / 8; ++c)
        st_global_v8(out + c * BM * 8, __uint_as_float(qr[8 * c]) * isd, __uint_as_float(qr[8 * c + 1]) * isd,
                     __uint_as_float(qr[8 * c + 2]) * isd, __uint_as_float(qr[8 * c + 3]) * isd,
                     __uint_as_float(qr[8 * c + 4]) * isd, __uint_as_float(qr[8 * c + 5]) * isd,
                     __uint_as_float(qr[8 * c + 6]) * isd, __uint_as_float(qr[8 * c + 7]) * isd);
    }
    tc_fence_before();
    mbar_arrive(&bars->dq_read);
    if constexpr ((kAtomic & 4) != 0) {
      fence_proxy_async_smem();  // the staged rows, before the engine reads them
      mbar_arrive(&bars->staged);
      if (warp == 3 && lane == 0) {
        if (!mbar_wait(&bars->staged, t & 1, wc, abort)) return false;
        if (live) bulk_reduce_add_f32(dq_part + (slice * JQ + ti) * (BM * D), sm + L::kDS, BM * D * 4);
        bulk_wait_read();
        mbar_arrive(&bars->stage_free);  // the next dS may overwrite the staging area
      }
    }
    return true;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer (converged warp)
    // constant A operands of the record step and the zero K columns, made
    // visible to the tensor core before kv_full (which the issuers wait for)
    {
      const uint32_t one2 = 0x3F803F80u, one1 = 0x00003F80u;  // BF16 1.0 pairs
      uint4* augS = reinterpret_cast<uint4*>(sm + L::kAugS);
      uint4* augP = reinterpret_cast<uint4*>(sm + L::kAugP);
      uint4* zero = reinterpret_cast<uint4*>(sm + L::kZero);
      for (int rr = lane; rr < BM; rr += 32) {
        augS[rr] = make_uint4(one2, one1, 0u, 0u);
        augP[rr] = make_uint4(0u, 0u, one2, one1);
        zero[rr] = make_uint4(0u, 0u, 0u, 0u);
      }
      fence_proxy_async_smem();
      __syncwarp();
    }
    if (elect_one()) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      prefetch_tmap(&tm_do);
      prefetch_tmap(&tm_biasT);
      mbar_expect_tx(&bars->kv_full, 2 * G * L::kTile);
      for (int g = 0; g < G; ++g) {
        const int bo = b * N_o + o0 + g;
        tma_load_rows(sm + L::kK + g * L::kTile, &tm_k, &bars->kv_full, lq.hn, ktile * BN, h, bo, H);
        tma_load_rows(sm + L::kV + g * L::kTile, &tm_v, &bars->kv_full, lq.hn, ktile * BN, h, bo, H);
      }
    }
    __syncwarp();
    bool ok = true;
    for (int s = 0; s < nsteps && ok; ++s) {
      const int i = s / G, g = s % G;
      if (g == 0) {
        const int st = i & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(&bars->b_empty[st], ((i >> 1) & 1) ^ 1, wc, abort))) {
          ok = false;
          break;
        }
        if (elect_one()) {
          mbar_expect_tx(&bars->b_full[st], BM * BN * 2);
          uint8_t* bdst = sm + L::kBias + st * (BM * BN * 2);
          tma_load_3d(bdst, &tm_biasT, &bars->b_full[st], i * BM, ktile * BN, bh);
          tma_load_3d(bdst + BN * 128, &tm_biasT, &bars->b_full[st], i * BM + 64, ktile * BN, bh);
        }
        __syncwarp();
      }
      const int st = s % NQ;
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->qdo_empty[st], ((s / NQ) & 1) ^ 1, wc, abort))) {
        ok = false;
        break;
      }
      if (elect_one()) {
        const int boh = (b * N_o + o0 + g) * H + h;
        mbar_expect_tx(&bars->qdo_full[st], 2 * L::kTile + kRecTile);
        tma_load_rows(sm + L::kQ + st * L::kTile, &tm_q, &bars->qdo_full[st], lq.hn, i * BM, h, b * N_o + o0 + g, H);
        tma_load_rows(sm + L::kDO + st * L::kTile, &tm_do, &bars->qdo_full[st], ldo.hn, i * BM, h, b * N_o + o0 + g,
                      H);
        bulk_load(sm + L::kRec + st * kRecTile, rec + (static_cast<size_t>(min(boh, last_rec_slice)) * JQ + i) * BM,
                  kRecTile, &bars->qdo_full[st]);
      }
      __syncwarp();
      if (s >= 2) ok = drain_dq(s - 2);
    }
    for (int t = nsteps >= 2 ? nsteps - 2 : 0; t < nsteps && ok; ++t) ok = drain_dq(t);
  } else if (warp <= 3) {
    // ------------------------------------------------------------ MMA issuers
    constexpr uint32_t kSwz = (D == 32) ? 4u : 6u;  // 64B / 32B swizzle for D-wide rows
    constexpr uint32_t kSbo = 8u * D * 2u;
    constexpr uint32_t idSS = idesc_bf16_f32(BN, BM, 0, 0);     // S^T, dP^T: A, B K-major
    constexpr uint32_t idKV = idesc_bf16_f32(BN, D, 0, 1);      // dV, dK: A in TMEM, B MN-major
    constexpr uint32_t idQ = idesc_bf16_f32(BM, D, 1, 1);       // dQ: A MN-major, B MN-major
    constexpr uint32_t kTile16 = L::kTile >> 4;                 // tile size in descriptor units
    constexpr uint32_t kRowStep = (16 * D * 2) >> 4;            // 16 rows of a D-wide tile
    // base descriptors; per-MMA offsets are added to the start-address field
    const uint64_t dQb = smem_desc(smem_u32(sm + L::kQ), 16, kSbo, kSwz);
    const uint64_t dDOb = smem_desc(smem_u32(sm + L::kDO), 16, kSbo, kSwz);
    const uint64_t dKb = smem_desc(smem_u32(sm + L::kK), 16, kSbo, kSwz);
    const uint64_t dVb = smem_desc(smem_u32(sm + L::kV), 16, kSbo, kSwz);
    const uint64_t dDSmn = smem_desc(smem_u32(sm + L::kDS), 16384, 1024, 2);  // dS (queries contiguous)
    // record step (no swizzle, K-major: 8-row core matrices 128 B apart,
    // K columns 8-15 in the zero block)
    const uint64_t dAugS = smem_desc(smem_u32(sm + L::kAugS), L::kZero - L::kAugS, 128, 0);
    const uint64_t dAugP = smem_desc(smem_u32(sm + L::kAugP), L::kZero - L::kAugP, 128, 0);
    auto rec_desc = [&](int stage) {
      const uint32_t off = L::kRec + stage * kRecTile;
      return smem_desc(smem_u32(sm + off), L::kZero - off, 128, 0);
    };
    bool ok = __all_sync(0xffffffffu, mbar_wait(&bars->kv_full, 0, wc, abort)) &&
              (warp == 3 || __all_sync(0xffffffffu, mbar_wait(&bars->qdo_full[0], 0, wc, abort)));
    if (warp == 1) {
      // ---- issuer A: dV_g += P^T dO, then S^T(s+1) = K Q^T
      if (ok) {
        tc_fence_after();
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) mma_ss(tmem + kTS, dKb + 2 * kk, dQb + 2 * kk, idSS, kk > 0 ? 1u : 0u);
          mma_ss(tmem + kTS, dAugS, rec_desc(0), idSS, 1u);  // + (-lse sqrt(D))
          mma_commit(&bars->s_full);
        }
        __syncwarp();
      }
      for (int s = 0; s < nsteps && ok; ++s) {
        const int i = s / G, g = s % G, st = s % NQ, st1 = (s + 1) % NQ;
        const bool next = s + 1 < nsteps;
        // P-phase of s done (P^T in TMEM); Q(s+1) loaded; the dQ tile of s-1,
        // which S^T(s+1) overwrites, drained (parity 1 passes at s = 0)
        const uint32_t wb[3] = {smem_u32(&bars->p_ready), smem_u32(next ? &bars->qdo_full[st1] : &bars->never),
                               smem_u32(next ? &bars->dq_read : &bars->never)};
        const uint32_t wp[3] = {static_cast<uint32_t>(s & 1), next ? ((s + 1) / NQ) & 1 : 1u,
                                next ? (s - 1) & 1 : 1u};
        if (!mbar_wait_all(wb, wp, wc, abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t dod = dDOb + st * kTile16;
        const uint64_t qn = dQb + st1 * kTile16, kn = dKb + ((s + 1) % G) * kTile16;
        if (elect_one()) {
          const uint32_t tdv = tmem + g * D;
#pragma unroll
          for (int kk = 0; kk < BM / 16; ++kk)  // dV_g += P^T dO
            mma_ts(tdv, tmem + kTS + p_col(kk >> 1) + 8 * (kk & 1), dod + kk * kRowStep, idKV,
                   (i > 0 || kk > 0) ? 1u : 0u);
          if (next) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) mma_ss(tmem + kTS, kn + 2 * kk, qn + 2 * kk, idSS, kk > 0 ? 1u : 0u);
            mma_ss(tmem + kTS, dAugS, rec_desc(st1), idSS, 1u);
            mma_commit(&bars->s_full);
          }
          mma_commit(&bars->qdo_empty[st]);
        }
        __syncwarp();
        if (!drain_dq(s)) { ok = false; break; }
      }
    } else if (warp == 2) {
      // ---- issuer C: dK_g += dS^T Q, then dP^T(s+1) = V dO^T
      if (ok) {
        tc_fence_after();
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) mma_ss(tmem + kTDP, dVb + 2 * kk, dDOb + 2 * kk, idSS, kk > 0 ? 1u : 0u);
          mma_ss(tmem + kTDP, dAugP, rec_desc(0), idSS, 1u);  // + (-delta)
          mma_commit(&bars->dp_full);
        }
        __syncwarp();
      }
      for (int s = 0; s < nsteps && ok; ++s) {
        const int i = s / G, st = s % NQ, st1 = (s + 1) % NQ;
        const bool next = s + 1 < nsteps;
        // dS-phase of s done (dS^T in TMEM); dO(s+1) loaded
        const uint32_t wb[2] = {smem_u32(&bars->ds_ready), smem_u32(next ? &bars->qdo_full[st1] : &bars->never)};
        const uint32_t wp[2] = {static_cast<uint32_t>(s & 1), next ? ((s + 1) / NQ) & 1 : 1u};
        if (!mbar_wait_all(wb, wp, wc, abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t qd = dQb + st * kTile16;
        const uint64_t don = dDOb + st1 * kTile16, vn = dVb + ((s + 1) % G) * kTile16;
        if (elect_one()) {
          const uint32_t tdk = tmem + G * D + (s % G) * D;
#pragma unroll
          for (int kk = 0; kk < BM / 16; ++kk)  // dK_g += dS^T Q
            mma_ts(tdk, tmem + kTDP + 32 * (kk >> 1) + 8 * (kk & 1), qd + kk * kRowStep, idKV,
                   (i > 0 || kk > 0) ? 1u : 0u);
          if (next) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) mma_ss(tmem + kTDP, vn + 2 * kk, don + 2 * kk, idSS, kk > 0 ? 1u : 0u);
            mma_ss(tmem + kTDP, dAugP, rec_desc(st1), idSS, 1u);
            mma_commit(&bars->dp_full);
          }
          mma_commit(&bars->qdo_empty[st]);
        }
        __syncwarp();
        if (!drain_dq(s)) { ok = false; break; }
      }
    } else {
      // ---- issuer B: the dQ tile dS K into S^T columns [48, 48 + D)
      // S^T(0) loaded, so that the s_cons poll below never sees the barrier
      // two phases behind
      ok = ok && __all_sync(0xffffffffu, mbar_wait(&bars->s_cons, 0, wc, abort));
      for (int s = 0; s < nsteps && ok; ++s) {
        // dS of s in shared memory; every warp has loaded S^T(s+1)
        const bool next = s + 1 < nsteps;
        const uint32_t wb[2] = {smem_u32(&bars->ds_ready), smem_u32(next ? &bars->s_cons : &bars->never)};
        const uint32_t wp[2] = {static_cast<uint32_t>(s & 1), next ? (s + 1) & 1 : 1u};
        if (!mbar_wait_all(wb, wp, wc, abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t kd = dKb + (s % G) * kTile16;
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)  // A = dS (queries contiguous), B = K MN-major
            mma_ss(tmem + kTDQ, dDSmn + kk * 128, kd + kk * kRowStep, idQ, kk > 0 ? 1u : 0u);
          mma_commit(&bars->dq_full);
        }
        __syncwarp();
        if (!drain_dq(s)) { ok = false; break; }
      }
    }
    // the last bulk reduction has landed before the kernel ends
    if constexpr ((kAtomic & 4) != 0) {
      if (warp == 3 && lane == 0) bulk_wait_all();
    }
    // every MMA this issuer started is complete when all_done fires
    if (elect_one()) mma_commit(&bars->all_done);
    __syncwarp();
  } else {
    // ------------------------------------------------------------ elementwise warpgroups
    const int quarter = warp & 3;             // TMEM lane quarter of this warp
    const int wg = (warp - 4) >> 2;           // query-column quarter handled by this warpgroup
    const int r = quarter * 32 + lane;        // TMEM lane: key row (S^T, dP^T, dK, dV) / query row (dQ)
    const int col0 = wg * kCols;
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const float scale_log2 = kLog2e * rsqrtf(static_cast<float>(D));
    const float inv_sqrt_d = rsqrtf(static_cast<float>(D));
    uint8_t* sDS = sm + L::kDS;

    // base-2 key mask of each slice of the group (-inf past N): warpgroup w
    // stages slices w, w + 4, ...  Staged before any bounded wait, so the
    // barrier below is always entered by every elementwise thread.
    const int key = ktile * BN + r;
    float* mask_s = reinterpret_cast<float*>(sm + L::kMask);
    for (int gg = wg; gg < G; gg += kNWG) {
      float mv = -INFINITY;
      if (key < N && o0 + gg < N_o) {
        mv = 0.f;
        if (mask != nullptr)
          mv = __uint_as_float(static_cast<uint32_t>(__ldg(mask + (static_cast<size_t>(b) * N_o + o0 + gg) * N + key))
                               << 16) *
               kLog2e;
      }
      mask_s[gg * BN + r] = mv;
    }
    named_bar_sync(1, kEW);

    float2 dbacc[kCols / 2];  // dbias accumulators of this thread's key for its query columns
#pragma unroll
    for (int k = 0; k < kCols / 2; ++k) dbacc[k] = make_float2(0.f, 0.f);
    const float2 c2 = make_float2(scale_log2, scale_log2);
    const float2 l2e2 = make_float2(kLog2e, kLog2e);
    bool ok = true;

    for (int s = 0; s < nsteps && ok; ++s) {
      const int i = s / G, g = s % G;
      const int bst = i & 1;
      // bias^T tile of query tile i and S^T(s) (-lse sqrt(D) already added)
      if (g == 0 && !__all_sync(0xffffffffu, mbar_wait(&bars->b_full[bst], (i >> 1) & 1, wc, abort))) {
        ok = false;
        break;
      }
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->s_full, s & 1, wc, abort))) {
        ok = false;
        break;
      }
      const uint8_t* bias_s = sm + L::kBias + bst * (BM * BN * 2);

      // ---------------- P-phase
      tc_fence_after();
      float2 p[kCols / 2];
      uint32_t pw[kCols / 2];
      {
        uint32_t sv[kCols];
        tmem_ld32_wait(tmem + lane_addr + kTS + col0, sv);
        tc_fence_before();
        mbar_arrive(&bars->s_cons);
        const float m = mask_s[g * BN + r];  // 0 for most keys, -inf for masked keys and keys past N
        const float2 m2 = make_float2(m, m);
#pragma unroll
        for (int v = 0; v < kCols / 8; ++v) {  // 8 queries per 16-byte chunk
          const int cc = (col0 >> 3) + v;
          const uint32_t off = (cc >> 3) * (BN * 128) + sw128(r, cc & 7);
          const uint4 bw = *reinterpret_cast<const uint4*>(bias_s + off);
          const uint32_t bws[4] = {bw.x, bw.y, bw.z, bw.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 s2 = make_float2(__uint_as_float(sv[v * 8 + 2 * e]), __uint_as_float(sv[v * 8 + 2 * e + 1]));
            const float2 b2 = make_float2(bf16lo_to_f32(bws[e]), bf16hi_to_f32(bws[e]));
            const float2 t = ffma2(s2, c2, ffma2(b2, l2e2, m2));
            const float2 pp = make_float2(ex2_approx(t.x), ex2_approx(t.y));
            p[v * 4 + e] = pp;
            pw[v * 4 + e] = pack_bf16x2(pp.x, pp.y);
          }
        }
      }
      if (g == G - 1) mbar_arrive(&bars->b_empty[bst]);  // last read of this bias tile
      // BF16 P^T into columns this thread has read itself
      tmem_st16(tmem + lane_addr + kTS + col0 + ((wg & 1) ? 0 : 16), pw);  // = p_col(wg)
      tc_wait_st();
      tc_fence_before();
      mbar_arrive(&bars->p_ready);

      // ---------------- dS-phase (dS in shared memory is free once the previous dQ tile is done)
      {
        // dP^T(s); the dQ tile of s-1 has read dS (parity 1 passes at s = 0);
        // with the bulk reduction the staged tile of s-1 has been read too
        const uint32_t wb[2] = {smem_u32(&bars->dp_full),
                                smem_u32((kAtomic & 4) != 0 ? &bars->stage_free : &bars->dq_full)};
        const uint32_t wp[2] = {static_cast<uint32_t>(s & 1), static_cast<uint32_t>((s - 1) & 1)};
        if (!mbar_wait_all(wb, wp, wc, abort)) {
          ok = false;
          break;
        }
      }
      tc_fence_after();
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {  // 16 queries at a time
        uint32_t a[8], bq[8];
        tmem_ld8x2_wait(tmem + lane_addr + kTDP + col0 + hh * 16, a, tmem + lane_addr + kTDP + col0 + hh * 16 + 8, bq);
        uint32_t dw[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const uint32_t x0 = e < 4 ? a[2 * e] : bq[2 * e - 8];
          const uint32_t x1 = e < 4 ? a[2 * e + 1] : bq[2 * e - 7];
          const float2 dp2 = make_float2(__uint_as_float(x0), __uint_as_float(x1));
          const float2 ds = fmul2(p[hh * 8 + e], dp2);  // dP^T - delta from the MMA
          dbacc[hh * 8 + e] = fadd2(dbacc[hh * 8 + e], ds);
          dw[e] = pack_bf16x2(ds.x, ds.y);
        }
        // dS^T of queries [col0 + 16hh, +16) -> this warpgroup's own dP^T columns
        tmem_st8(tmem + lane_addr + kTDP + col0 + 8 * hh, dw);
#pragma unroll
        for (int v = 0; v < 2; ++v) {
          const int cc = (col0 >> 3) + hh * 2 + v;
          const uint32_t off = (cc >> 3) * (BN * 128) + sw128(r, cc & 7);
          *reinterpret_cast<uint4*>(sDS + off) = make_uint4(dw[4 * v], dw[4 * v + 1], dw[4 * v + 2], dw[4 * v + 3]);
        }
      }
      fence_proxy_async_smem();
      tc_wait_st();
      tc_fence_before();
      mbar_arrive(&bars->ds_ready);
      if (g == G - 1) {
        // single-writer dbias partial of this outer group for tile (i, ktile),
        // stored chunk-major ([16 chunks of 8 queries][128 keys] x 8 floats)
        // with 32-byte stores, so that each warp store covers 1 KB
        if constexpr ((kAtomic & 2) != 0) {
          float* acc = dbias_part + ((static_cast<size_t>(bh) * nkt * BN + ktile * BN + r) * JQ + i) * BM + col0;
#pragma unroll
          for (int k4 = 0; k4 < kCols / 4; ++k4)
            red_add_v4(acc + 4 * k4, dbacc[2 * k4].x, dbacc[2 * k4].y, dbacc[2 * k4 + 1].x, dbacc[2 * k4 + 1].y);
        } else {
          float* dst = dbias_part +
                       ((((static_cast<size_t>(grp) * nbh + bh) * JQ + i) * nkt + ktile) * (BM * BN)) +
                       ((col0 / 8) * BN + r) * 8;
#pragma unroll
          for (int k8 = 0; k8 < kCols / 8; ++k8)
            st_global_v8(dst + k8 * BN * 8, dbacc[4 * k8].x, dbacc[4 * k8].y, dbacc[4 * k8 + 1].x,
                         dbacc[4 * k8 + 1].y, dbacc[4 * k8 + 2].x, dbacc[4 * k8 + 2].y, dbacc[4 * k8 + 3].x,
                         dbacc[4 * k8 + 3].y);
        }
#pragma unroll
        for (int k = 0; k < kCols / 2; ++k) dbacc[k] = make_float2(0.f, 0.f);
      }
    }

    // ------------------------------------------------------------ epilogue: dV_g and dK_g of slices g = wg, wg + 4, ...
    if (ok && __all_sync(0xffffffffu, mbar_wait(&bars->all_done, 0, wc, abort))) {
      tc_fence_after();
#pragma unroll 1
      for (int g = wg; g < G; g += kNWG)
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const long long off = lg.offset(b * N_o + o0 + g, h, key);
        const uint32_t t = tmem + lane_addr + which * G * D + g * D;
        const float sc = which == 0 ? 1.f : inv_sqrt_d;
        uint32_t w[D / 2];
        if constexpr (D == 32) {
          uint32_t raw[32];
          tmem_ld32_wait(t, raw);
#pragma unroll
          for (int e = 0; e < 16; ++e)
            w[e] = pack_bf16x2(__uint_as_float(raw[2 * e]) * sc, __uint_as_float(raw[2 * e + 1]) * sc);
        } else {
          uint32_t raw[16];
          tmem_ld16_wait(t, raw);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            w[e] = pack_bf16x2(__uint_as_float(raw[2 * e]) * sc, __uint_as_float(raw[2 * e + 1]) * sc);
        }
        if (key < N && o0 + g < N_o) {
          uint4* dst = reinterpret_cast<uint4*>((which == 0 ? dv : dk) + off);
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
// chunk-major partials (four partials' loads in flight per thread), FP32 sums
// in fixed order, transpose through shared memory, coalesced BF16 row writes.
template <int D>
__global__ void __launch_bounds__(256) reduce_dq_kernel(const float4* __restrict__ part, uint16_t* __restrict__ dq,
                                                        int N, int H, int JQ, int JK, size_t tiles, RowLayout lg) {
  constexpr int kChunks = BM * D / 4;      // float4 per tile
  constexpr int kStride = D + 4;           // padded row stride (floats) of the transpose buffer
  __shared__ float tile[BM * kStride];
  const size_t t = blockIdx.x;             // tile = slice * JQ + i
  const int i = static_cast<int>(t % JQ);
  const size_t slice = t / JQ;
  const long long bo = static_cast<long long>(slice / H);
  const int h = static_cast<int>(slice - bo * H);
  const size_t kstep = tiles * kChunks;    // float4 between key tiles' partials
  for (int e = threadIdx.x; e < kChunks; e += blockDim.x) {
    const float4* p = part + t * kChunks + e;
    float4 acc = __ldcs(p);
    // the loads of four consecutive partials issued together, the adds in
    // ascending order
    int kt = 1;
    for (; kt + 4 <= JK; kt += 4) {
      float4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) v[u] = __ldcs(p + static_cast<size_t>(kt + u) * kstep);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        acc.x += v[u].x;
        acc.y += v[u].y;
        acc.z += v[u].z;
        acc.w += v[u].w;
      }
    }
    for (; kt < JK; ++kt) {
      const float4 v = __ldcs(p + static_cast<size_t>(kt) * kstep);
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    const int rem = e % (2 * BM), c = 2 * (e / (2 * BM)) + (rem & 1), r = rem >> 1;
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
    *reinterpret_cast<uint4*>(dq + lg.offset(bo, h, q) + 8 * c8) = w;
  }
}

// dbias[b,h,q,k] = sum_{l = 0 .. L-1} dbias_part[l][b,h,q,k]   (ascending l, FP32).
// A partial tile is stored [16 chunks of 8 queries][128 keys] x 8 floats, so
// an 8-query slab is 4 KB contiguous.  One block per slab of a 128 x 128 tile
// (b*h, query tile i, key tile t), one float4 per thread (key e/2, queries
// 4(e&1) .. +4); the loads of four consecutive partials are issued together,
// the adds stay in ascending order.  Small blocks keep the SMs evenly loaded
// to the end (16-query slabs left the last wave ragged).
constexpr int kSlab = 8;
constexpr int kRedThreads = kSlab / 4 * BN;  // one float4 chunk per thread
// OutT = uint16_t: BF16 dbias; float: the FP32 sum itself (one GPU's part of
// an outer axis split across GPUs).
template <typename OutT>
__global__ void __launch_bounds__(kRedThreads) reduce_dbias_kernel(const float4* __restrict__ part,
                                                           OutT* __restrict__ dbias, int N, int JQ, int JK,
                                                           int ngroups, size_t tiles) {
  constexpr bool kF32 = sizeof(OutT) == 4;
  constexpr int kChunks = BM * BN / 4;     // float4 per tile
  constexpr int kSlabChunks = kSlab / 4 * BN;
  constexpr int kStride = BN + 16 / sizeof(OutT);  // padded row stride of the transpose buffer
  __shared__ __align__(16) OutT tile[kSlab * kStride];
  const size_t t = blockIdx.x / (BM / kSlab);
  const int slab = blockIdx.x % (BM / kSlab);
  const int kt = static_cast<int>(t % JK);
  const int i = static_cast<int>((t / JK) % JQ);
  const size_t bh = t / (static_cast<size_t>(JK) * JQ);
  const size_t lstride = tiles * kChunks;
  static_assert(kSlab == 8, "a slab is one 8-query chunk of the partial tile");
  for (int e = threadIdx.x; e < kSlabChunks; e += blockDim.x) {
    const int cl = e & 1, k = e >> 1;      // 4-query half of the chunk, key
    const float4* p = part + t * kChunks + slab * kSlabChunks + e;
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
    if constexpr (kF32) {
      tile[(4 * cl + 0) * kStride + k] = acc.x;
      tile[(4 * cl + 1) * kStride + k] = acc.y;
      tile[(4 * cl + 2) * kStride + k] = acc.z;
      tile[(4 * cl + 3) * kStride + k] = acc.w;
    } else {
      const uint32_t w01 = pack_bf16x2(acc.x, acc.y), w23 = pack_bf16x2(acc.z, acc.w);
      tile[(4 * cl + 0) * kStride + k] = static_cast<uint16_t>(w01 & 0xFFFFu);
      tile[(4 * cl + 1) * kStride + k] = static_cast<uint16_t>(w01 >> 16);
      tile[(4 * cl + 2) * kStride + k] = static_cast<uint16_t>(w23 & 0xFFFFu);
      tile[(4 * cl + 3) * kStride + k] = static_cast<uint16_t>(w23 >> 16);
    }
  }
  __syncthreads();
  constexpr int kPer = 16 / sizeof(OutT);  // elements per 16-byte item
  constexpr int kItems = kSlab * BN / kPer;
  const bool vec = N % kPer == 0;          // rows 16-byte aligned, an item all in or all out
  for (int e = threadIdx.x; e < kItems; e += blockDim.x) {
    const int rr = e / (BN / kPer), c = e % (BN / kPer);
    const int q = i * BM + slab * kSlab + rr, k = kt * BN + kPer * c;
    if (q >= N || k >= N) continue;
    OutT* dst = dbias + (bh * N + q) * N + k;
    const OutT* src = &tile[rr * kStride + kPer * c];
    if (vec) {
      *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
    } else {
      for (int u = 0; u < kPer && k + u < N; ++u) dst[u] = src[u];
    }
  }
}

// dbias = bf16(sum_r parts[r]) in ascending r: four elements per thread when
// every part starts 16-byte aligned (elems a multiple of 4), else one.
__global__ void __launch_bounds__(256) dbias_combine_kernel(const float* __restrict__ parts, int R, size_t elems,
                                                            uint16_t* __restrict__ dbias) {
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  const size_t t0 = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (elems % 4 == 0) {
    const float4* p4 = reinterpret_cast<const float4*>(parts);
    const size_t n4 = elems / 4;
    for (size_t e = t0; e < n4; e += stride) {
      float4 acc = __ldcs(p4 + e);
      for (int r = 1; r < R; ++r) {
        const float4 v = __ldcs(p4 + static_cast<size_t>(r) * n4 + e);
        acc.x += v.x;
        acc.y += v.y;
        acc.z += v.z;
        acc.w += v.w;
      }
      reinterpret_cast<uint2*>(dbias)[e] = make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
    }
  } else {
    for (size_t e = t0; e < elems; e += stride) {
      float acc = parts[e];
      for (int r = 1; r < R; ++r) acc += parts[static_cast<size_t>(r) * elems + e];
      dbias[e] = static_cast<uint16_t>(pack_bf16x2(acc, 0.f) & 0xFFFFu);
    }
  }
}

// ---------------------------------------------------------------- ablation only
// The non-deterministic variant of the backward adds dQ and / or dbias into
// FP32 accumulators with atomics; these two kernels round them to BF16.

// dQ accumulator [slices][J_Q*128][D] FP32 -> dq [slices][N][D] BF16; one
// thread per 8 outputs.
template <int D>
__global__ void __launch_bounds__(256) finish_dq_kernel(const float4* __restrict__ acc, uint16_t* __restrict__ dq,
                                                        int N, int H, int JQ, size_t rows, RowLayout lg) {
  const size_t e = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (e >= rows * (D / 8)) return;
  const size_t row = e / (D / 8);
  const int c8 = static_cast<int>(e % (D / 8));
  const size_t slice = row / N;
  const int q = static_cast<int>(row % N);
  const float4* src = acc + ((slice * JQ * BM + q) * D + 8 * c8) / 4;
  const float4 x = src[0], y = src[1];
  const long long bo = static_cast<long long>(slice / H);
  *reinterpret_cast<uint4*>(dq + lg.offset(bo, static_cast<int>(slice - bo * H), q) + 8 * c8) =
      make_uint4(pack_bf16x2(x.x, x.y), pack_bf16x2(x.z, x.w), pack_bf16x2(y.x, y.y), pack_bf16x2(y.z, y.w));
}

// dbias accumulator [B*H][J_K*128 (k)][J_Q*128 (q)] FP32 -> dbias [B*H][N][N]
// BF16, transposed through 64 x 64 shared-memory tiles.
__global__ void __launch_bounds__(256) finish_dbias_kernel(const float* __restrict__ acc, uint16_t* __restrict__ dbias,
                                                           int N, int JK, int JQ) {
  __shared__ float tile[64][65];
  const int q0 = blockIdx.y * 64, k0 = blockIdx.x * 64;
  const size_t ld = static_cast<size_t>(JQ) * BM;
  const float* base = acc + static_cast<size_t>(blockIdx.z) * JK * BN * ld;
  for (int e = threadIdx.x; e < 64 * 64; e += blockDim.x) {
    const int kk = e / 64, qq = e % 64;  // inside the padded accumulator
    tile[kk][qq] = base[static_cast<size_t>(k0 + kk) * ld + q0 + qq];
  }
  __syncthreads();
  for (int e = threadIdx.x; e < 64 * 32; e += blockDim.x) {
    const int qq = e / 32, kp = e % 32;
    const int q = q0 + qq, k = k0 + 2 * kp;
    if (q >= N || k >= N) continue;
    uint16_t* dst = dbias + (static_cast<size_t>(blockIdx.z) * N + q) * N + k;
    const uint32_t w = pack_bf16x2(tile[2 * kp][qq], tile[2 * kp + 1][qq]);
    if ((N & 1) == 0) {
      *reinterpret_cast<uint32_t*>(dst) = w;  // even N: 4-byte aligned, k + 1 < N
    } else {
      dst[0] = static_cast<uint16_t>(w & 0xFFFFu);
      if (k + 1 < N) dst[1] = static_cast<uint16_t>(w >> 16);
    }
  }
}

}  // namespace

template <int D>
int bwd_smem_bytes() { return BwdSmem<D>::kBytes; }

template <int D>
cudaError_t setup_bwd() {
  cudaError_t e = cudaFuncSetAttribute(bwd_main_kernel<D, 0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       BwdSmem<D>::kBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(bwd_main_kernel<D, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, BwdSmem<D>::kBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(bwd_main_kernel<D, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, BwdSmem<D>::kBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(bwd_main_kernel<D, 3>, cudaFuncAttributeMaxDynamicSharedMemorySize, BwdSmem<D>::kBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(bwd_main_kernel<D, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize, BwdSmem<D>::kBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(bwd_main_kernel<D, 6>, cudaFuncAttributeMaxDynamicSharedMemorySize, BwdSmem<D>::kBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(bwd_main_kernel<D, 0, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             BwdSmem<D>::kBytes);
  return e;
}

template <int D>
cudaError_t launch_bwd_preprocess(const BwdArgs& a, cudaStream_t stream) {
  const int JQ = (a.N + BM - 1) / BM;
  const size_t padded = static_cast<size_t>(a.B) * a.N_o * a.H * JQ * BM;
  const unsigned grid = static_cast<unsigned>((padded * (D / 8) + 255) / 256);
  preprocess_kernel<D><<<grid, 256, 0, stream>>>(static_cast<const uint16_t*>(a.dO), static_cast<const uint16_t*>(a.o),
                                                 static_cast<const uint16_t*>(a.o_resid), a.lse, a.rec, a.N, a.H,
                                                 JQ, padded, a.lo, a.ldo);
  return cudaGetLastError();
}

cudaError_t launch_bwd_transpose_bias(const BwdArgs& a, cudaStream_t stream) {
  const unsigned t = static_cast<unsigned>((a.N + 63) / 64);
  transpose_bias_kernel<<<dim3(t, t, a.B * a.H), 256, 0, stream>>>(static_cast<const uint16_t*>(a.bias),
                                                                   static_cast<uint16_t*>(a.biasT), a.N,
                                                                   (a.N + 7) / 8 * 8);
  return cudaGetLastError();
}

template <int D, int kAtomic>
cudaError_t launch_main_variant(const BwdArgs& a, cudaStream_t stream) {
  const int JK = (a.N + BN - 1) / BN;
  const int NG = (a.N_o + BwdSmem<D>::G - 1) / BwdSmem<D>::G;
  const bool hn = a.lq.hn || a.ldo.hn || a.lg.hn;
  if (hn && kAtomic != 0) return cudaErrorInvalidValue;  // the ablation takes the contiguous layout
  const dim3 grid = hn ? dim3(JK * a.H, NG, a.B) : dim3(JK, NG, a.B * a.H);
  auto kernel = hn ? bwd_main_kernel<D, kAtomic, true> : bwd_main_kernel<D, kAtomic, false>;
  kernel<<<grid, kMainThreads, BwdSmem<D>::kBytes, stream>>>(
      a.tm_q, a.tm_k, a.tm_v, a.tm_do, a.tm_biasT, static_cast<const uint16_t*>(a.mask), a.rec,
      static_cast<uint16_t*>(a.dk), static_cast<uint16_t*>(a.dv), a.dq_part, a.dbias_part, a.N_o, a.N, a.H, a.lq,
      a.ldo, a.lg, a.wc);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_bwd_main(const BwdArgs& a, cudaStream_t stream) {
  return launch_main_variant<D, 0>(a, stream);
}

template <int D>
cudaError_t launch_bwd_main_atomic(const BwdArgs& a, int atomic_mask, cudaStream_t stream) {
  if (atomic_mask == 1) return launch_main_variant<D, 1>(a, stream);
  if (atomic_mask == 2) return launch_main_variant<D, 2>(a, stream);
  if (atomic_mask == 3) return launch_main_variant<D, 3>(a, stream);
  if (atomic_mask == 4) return launch_main_variant<D, 4>(a, stream);
  if (atomic_mask == 6) return launch_main_variant<D, 6>(a, stream);
  return cudaErrorInvalidValue;
}

template <int D>
cudaError_t launch_bwd_finish_dq(const BwdArgs& a, cudaStream_t stream) {
  const int JQ = (a.N + BM - 1) / BM;
  const size_t rows = static_cast<size_t>(a.B) * a.N_o * a.H * a.N;
  const size_t items = rows * (D / 8);
  finish_dq_kernel<D><<<static_cast<unsigned>((items + 255) / 256), 256, 0, stream>>>(
      reinterpret_cast<const float4*>(a.dq_part), static_cast<uint16_t*>(a.dq), a.N, a.H, JQ, rows, a.lg);
  return cudaGetLastError();
}

cudaError_t launch_bwd_finish_dbias(const BwdArgs& a, cudaStream_t stream) {
  const int JK = (a.N + BN - 1) / BN, JQ = (a.N + BM - 1) / BM;
  const unsigned t = static_cast<unsigned>((a.N + 63) / 64);
  finish_dbias_kernel<<<dim3(t, t, a.B * a.H), 256, 0, stream>>>(a.dbias_part, static_cast<uint16_t*>(a.dbias), a.N,
                                                                 JK, JQ);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_bwd_reduce_dq(const BwdArgs& a, cudaStream_t stream) {
  const int JK = (a.N + BN - 1) / BN, JQ = (a.N + BM - 1) / BM;
  const size_t tiles = static_cast<size_t>(a.B) * a.N_o * a.H * JQ;
  reduce_dq_kernel<D><<<static_cast<unsigned>(tiles), 256, 0, stream>>>(
      reinterpret_cast<const float4*>(a.dq_part), static_cast<uint16_t*>(a.dq), a.N, a.H, JQ, JK, tiles, a.lg);
  return cudaGetLastError();
}

cudaError_t launch_bwd_reduce_dbias(const BwdArgs& a, cudaStream_t stream) {
  const int JK = (a.N + BN - 1) / BN, JQ = (a.N + BM - 1) / BM;
  const size_t tiles = static_cast<size_t>(a.B) * a.H * JQ * JK;
  const unsigned blocks = static_cast<unsigned>(tiles * (BM / kSlab));
  const int groups = (a.N_o + kGroupBwdFor(a.D) - 1) / kGroupBwdFor(a.D);
  if (a.dbias_fp32)
    reduce_dbias_kernel<float><<<blocks, kRedThreads, 0, stream>>>(
        reinterpret_cast<const float4*>(a.dbias_part), static_cast<float*>(a.dbias), a.N, JQ, JK, groups, tiles);
  else
    reduce_dbias_kernel<uint16_t><<<blocks, kRedThreads, 0, stream>>>(
        reinterpret_cast<const float4*>(a.dbias_part), static_cast<uint16_t*>(a.dbias), a.N, JQ, JK, groups,
        tiles);
  return cudaGetLastError();
}

cudaError_t launch_dbias_combine(const float* parts, int R, size_t elems, void* dbias, cudaStream_t stream) {
  const size_t n4 = elems / 4;
  const unsigned blocks = static_cast<unsigned>(std::max<size_t>(1, std::min<size_t>((n4 + 255) / 256, 152 * 16)));
  dbias_combine_kernel<<<blocks, 256, 0, stream>>>(parts, R, elems, static_cast<uint16_t*>(dbias));
  return cudaGetLastError();
}

template cudaError_t setup_bwd<16>();
template cudaError_t setup_bwd<32>();
template cudaError_t launch_bwd_main_atomic<16>(const BwdArgs&, int, cudaStream_t);
template cudaError_t launch_bwd_main_atomic<32>(const BwdArgs&, int, cudaStream_t);
template cudaError_t launch_bwd_finish_dq<16>(const BwdArgs&, cudaStream_t);
template cudaError_t launch_bwd_finish_dq<32>(const BwdArgs&, cudaStream_t);
template cudaError_t launch_bwd_preprocess<16>(const BwdArgs&, cudaStream_t);
template cudaError_t launch_bwd_preprocess<32>(const BwdArgs&, cudaStream_t);
template cudaError_t launch_bwd_main<16>(const BwdArgs&, cudaStream_t);
template cudaError_t launch_bwd_main<32>(const BwdArgs&, cudaStream_t);
template cudaError_t launch_bwd_reduce_dq<16>(const BwdArgs&, cudaStream_t);
template cudaError_t launch_bwd_reduce_dq<32>(const BwdArgs&, cudaStream_t);
template int bwd_smem_bytes<16>();
template int bwd_smem_bytes<32>();

}  // namespace triattn
