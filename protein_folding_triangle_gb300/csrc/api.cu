// C ABI of libtriattn: argument validation, TMA descriptor construction and
// kernel launches.  Declared in include/triattn.h.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "triattn.h"
#include "kernels.cuh"

namespace triattn {
namespace {

__device__ uint32_t g_status_word;

constexpr unsigned long long kDefaultWaitNs = 2000000000ull;  // 2 s
std::atomic<unsigned long long> g_wait_limit_ns{kDefaultWaitNs};
std::mutex g_init_mu;
uint64_t g_init_mask = 0;            // devices whose kernel attributes are set
uint32_t* g_status_ptr[64] = {};     // device address of g_status_word per device
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned_to(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

triattn_status init_device(int* dev_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return TRIATTN_ERR_CUDA;
  *dev_out = dev;
  std::lock_guard<std::mutex> lk(g_init_mu);
  if (g_encode == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        fn == nullptr || q != cudaDriverEntryPointSuccess)
      return TRIATTN_ERR_CUDA;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  // The device address of the status word is looked up on every call (it is
  // cheap): after a device reset the module is loaded again and a cached
  // address would be stale.
  void* sp = nullptr;
  if (cudaGetSymbolAddress(&sp, g_status_word) != cudaSuccess || sp == nullptr) return TRIATTN_ERR_CUDA;
  g_status_ptr[dev] = static_cast<uint32_t*>(sp);
  if ((g_init_mask & (1ull << dev)) && fwd_attrs_current()) return TRIATTN_OK;
  if (setup_fwd<16>() != cudaSuccess || setup_fwd<32>() != cudaSuccess || setup_bwd<16>() != cudaSuccess ||
      setup_bwd<32>() != cudaSuccess)
    return TRIATTN_ERR_CUDA;
  g_init_mask |= (1ull << dev);
  return TRIATTN_OK;
}

triattn_status check_shape(const triattn_shape* s) {
  if (s == nullptr) return TRIATTN_ERR_INVALID_ARG;
  if (s->B < 1 || s->N < 1 || s->N_o < 1 || s->H < 1 || (s->flags & ~TRIATTN_FLAG_DBIAS_FP32) != 0)
    return TRIATTN_ERR_INVALID_ARG;
  if (s->D != 16 && s->D != 32) return TRIATTN_ERR_UNSUPPORTED;
  // N outer slices, or a contiguous shard of them
  if (s->N_o > s->N) return TRIATTN_ERR_UNSUPPORTED;
  // grid limits: query / key tiles in gridDim.x, outer groups in gridDim.y,
  // B*H in gridDim.z
  if ((s->N_o + kGroupFwd - 1) / kGroupFwd > 65535 || static_cast<long long>(s->B) * s->H > 65535)
    return TRIATTN_ERR_UNSUPPORTED;
  // TMA outer dimension B*N_o*H (slices) and the [B*H, N, N] planes must fit
  // the 32-bit index arithmetic of the kernels
  if (static_cast<long long>(s->B) * (s->N_o + kGroupFwd) * s->H >= (1ll << 31)) return TRIATTN_ERR_UNSUPPORTED;
  if (static_cast<long long>(s->N) * ((s->N + 127) / 128 * 128) >= (1ll << 31)) return TRIATTN_ERR_UNSUPPORTED;
  return TRIATTN_OK;
}

// Row stride (elements) of the bias as the kernels read it: N, or N rounded up
// to a multiple of 8 for the padded copy (TMA needs 16-byte row strides).
int padded_n(int N) { return (N + 7) / 8 * 8; }

// Map over the rows of a [B, N_o, H, N, D] bf16 tensor in layout l, box =
// box_rows rows x D of one (slice, head): 3-D (D, N, B*N_o*H) when the rows
// lie inside the heads (slice = H head), 4-D (D, H, N, B*N_o) when the heads
// lie inside the rows (l.hn).
bool make_rows_map(CUtensorMap* m, const void* base, const triattn_shape* s, const RowLayout& l,
                   unsigned box_rows = 128) {
  const cuuint64_t D = static_cast<cuuint64_t>(s->D), N = static_cast<cuuint64_t>(s->N),
                   H = static_cast<cuuint64_t>(s->H), S = static_cast<cuuint64_t>(s->B) * s->N_o;
  const cuuint64_t row = static_cast<cuuint64_t>(l.row) * 2, head = static_cast<cuuint64_t>(l.head) * 2,
                   slice = static_cast<cuuint64_t>(l.slice) * 2;
  const CUtensorMapSwizzle sw = (s->D == 32) ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B;
  const cuuint32_t es[4] = {1u, 1u, 1u, 1u};
  if (!l.hn) {
    const cuuint64_t dims[3] = {D, N, S * H};
    const cuuint64_t strides[2] = {row, head};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(s->D), box_rows, 1u};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  }
  const cuuint64_t dims[4] = {D, H, N, S};
  const cuuint64_t strides[3] = {head, row, slice};
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(s->D), 1u, box_rows, 1u};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A caller's row layout: strides multiples of 8 elements (16-byte rows for
// TMA and the vector accesses), nested without overlap -- the D features of
// a row inside the smaller of the head and row strides, all rows (or heads)
// of that kind inside the larger one, a whole slice inside the slice stride
// (so the maps' dimensions are ordered by stride); with the rows inside the
// heads, the heads packed (slice = H head); the slice stride below 2^36
// elements.
bool layout_from(const triattn_layout* u, const triattn_shape* s, RowLayout* out) {
  if (u == nullptr) {
    *out = contiguous_layout(s->N, s->H, s->D);
    return true;
  }
  const long long D = s->D, N = s->N, H = s->H;
  if (u->slice <= 0 || u->head <= 0 || u->row <= 0 || ((u->slice | u->head | u->row) & 7) != 0) return false;
  if (u->slice >= (1ll << 36)) return false;
  // equal head and row strides only where one of them steps over a single
  // head or row (H = 1 or N = 1)
  if (u->head == u->row && H > 1 && N > 1) return false;
  const bool hn = u->head < u->row || (u->head == u->row && H == 1);  // heads inside a row
  // rows inside the heads: the heads of a slice packed (one map dimension for slice and head)
  if (!hn && u->slice != H * u->head) return false;
  const long long inner = hn ? u->head : u->row, outer = hn ? u->row : u->head;
  const long long n_inner = hn ? H : N, n_outer = hn ? N : H;
  if (inner < D || (n_inner - 1) * inner + D > outer || (n_outer - 1) * outer + (n_inner - 1) * inner + D > u->slice)
    return false;
  *out = RowLayout{u->slice, u->head, u->row, hn ? 1 : 0};
  return true;
}

// 3-D map over a [B*H, N, ld] bf16 matrix (the bias, its padded copy or its
// transposed copy; ld a multiple of 8), box = 128 rows x 64 columns; columns
// N .. ld-1 are outside the map (zero fill).
bool make_bias_map(CUtensorMap* m, const void* base, const triattn_shape* s, int ld) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(s->N), static_cast<cuuint64_t>(s->N),
                              static_cast<cuuint64_t>(s->B) * s->H};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld) * 2, static_cast<cuuint64_t>(ld) * s->N * 2};
  const cuuint32_t box[3] = {64u, 128u, 1u};
  const cuuint32_t es[3] = {1u, 1u, 1u};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Forward workspace: key-mask records [(B*N_o + 4) * J_K] (needed with a mask
// or when N is not a multiple of 64), then the padded bias [B*H, N, Np] (when
// N is not a multiple of 8); each part 256-byte aligned.
struct FwdWs {
  size_t rec_bytes, pad_off, pad_bytes;
  size_t total() const { return pad_off + pad_bytes; }
};
FwdWs fwd_ws(const triattn_shape* s, bool with_mask) {
  FwdWs w;
  const size_t jk = (s->N + 63) / 64;
  const bool need_rec = with_mask || s->N % 64 != 0;
  w.rec_bytes = need_rec ? round_up((static_cast<size_t>(s->B) * s->N_o + kGroupFwd) * jk * kFwdMaskRec, 256) : 0;
  w.pad_off = w.rec_bytes;
  w.pad_bytes = s->N % 8 != 0 ? round_up(static_cast<size_t>(s->B) * s->H * s->N * padded_n(s->N) * 2, 256) : 0;
  return w;
}

struct WsLayout {
  size_t rec_off, biasT_off, dq_off, db_off, total;
};

// query-row records [slices][J_Q * 128][8] BF16 (three-term splits of
// -lse sqrt(D) and -delta); transposed bias
// [B*H][N][N] BF16; dQ partials [J_K][slices][J_Q][128 x D] FP32; dbias
// partials [N_o/G][B*H][J_Q][J_K][128 x 128] FP32 (padded to whole tiles);
// each part 256-byte aligned.
WsLayout ws_layout(const triattn_shape* s, int atomic_mask = 0) {
  const size_t slices = static_cast<size_t>(s->B) * s->N_o * s->H;
  const size_t jk = (s->N + kTileK - 1) / kTileK;
  const size_t jq = (s->N + kTileQ - 1) / kTileQ;
  const size_t groups = (s->N_o + kGroupBwdFor(s->D) - 1) / kGroupBwdFor(s->D);
  WsLayout w;
  w.rec_off = 0;
  w.biasT_off = round_up(slices * jq * kTileQ * 16, 256);
  w.dq_off = w.biasT_off + round_up(static_cast<size_t>(s->B) * s->H * s->N * padded_n(s->N) * 2, 256);
  // ablation: FP32 accumulators instead of the partials (see tri_attn_bwd_atomic_ablation)
  const size_t dq_bytes =
      dq_accumulated(atomic_mask) ? slices * jq * kTileQ * s->D * 4 : jk * slices * jq * kTileQ * s->D * 4;
  const size_t db_bytes = (atomic_mask & 2) ? static_cast<size_t>(s->B) * s->H * jk * kTileK * jq * kTileQ * 4
                                            : groups * s->B * s->H * jq * jk * kTileQ * kTileK * 4;
  w.db_off = w.dq_off + round_up(dq_bytes, 256);
  w.total = w.db_off + round_up(db_bytes, 256);
  return w;
}

// ---------------------------------------------------------------- tracing
const char* const kKernelName[kKinds] = {"tri_attn_fwd",     "bwd_preprocess",  "bwd_transpose_bias",
                                         "bwd_main",         "bwd_reduce_dq",   "bwd_reduce_dbias",
                                         "bwd_main_atomic",  "bwd_finish_dq",   "bwd_finish_dbias",
                                         "dbias_combine",    "fwd_prep",        "module_ln_fwd",   "module_layout",
                                         "module_gemm",      "module_ln_bwd",   "module_colsum",
                                         "trimul_ln_in",     "trimul_proj_gemm", "trimul_gate",
                                         "trimul_contract_gemm", "trimul_ln_out", "trimul_out_gate",
                                         "trimul_colsum",   "gemm",            "trimul_proj_gate"};
struct TraceRec {
  int kind;
  cudaEvent_t a, b;
};
std::mutex g_trace_mu;
bool g_trace_on = false;
std::vector<TraceRec> g_trace;
std::vector<cudaEvent_t> g_event_pool;  // events owned by the library, reused
size_t g_event_next = 0;
std::atomic<int> g_test_starve{0};

cudaEvent_t next_event() {
  if (g_event_next == g_event_pool.size()) {
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    g_event_pool.push_back(e);
  }
  return g_event_pool[g_event_next++];
}

template <typename F>
cudaError_t traced(int kind, cudaStream_t s, F launch) {
  std::unique_lock<std::mutex> lk(g_trace_mu);
  if (!g_trace_on) {
    lk.unlock();
    return launch();
  }
  cudaEvent_t ea = next_event(), eb = next_event();
  if (ea == nullptr || eb == nullptr) return cudaErrorMemoryAllocation;
  cudaEventRecord(ea, s);
  const cudaError_t e = launch();
  cudaEventRecord(eb, s);
  g_trace.push_back({kind, ea, eb});
  return e;
}

}  // namespace

cudaError_t trace_call(int kind, cudaStream_t s, const std::function<cudaError_t()>& launch) {
  return traced(kind, s, launch);
}

WaitCtl current_wait_ctl() {
  int dev = 0;
  WaitCtl wc;
  wc.limit_ns = g_wait_limit_ns.load();
  wc.status = (init_device(&dev) == TRIATTN_OK) ? g_status_ptr[dev] : nullptr;
  return wc;
}

namespace {

WaitCtl wait_ctl(int dev) {
  WaitCtl wc;
  wc.limit_ns = g_wait_limit_ns.load();
  wc.status = g_status_ptr[dev];
  return wc;
}

}  // namespace
}  // namespace triattn

using namespace triattn;

namespace {

// The backward: atomic_mask 0 is the library's ordered path; 1, 2, 3, 4 and
// 6 are the non-deterministic ablation (FP32 atomics for dQ, dbias, or both;
// a TMA bulk reduction for dQ, alone or with atomic dbias).
triattn_status bwd_impl(const triattn_shape* shape, const void* q, const void* k, const void* v,
                        const triattn_layout* qkv_layout, const void* bias, const void* mask, const void* o,
                        const void* o_resid, const triattn_layout* o_layout, const float* lse, const void* dO,
                        const triattn_layout* do_layout, void* dq, void* dk, void* dv,
                        const triattn_layout* dqkv_layout, void* dbias, int atomic_mask, void* workspace,
                        size_t workspace_bytes, void* stream) {
  triattn_status st = check_shape(shape);
  if (st != TRIATTN_OK) return st;
  RowLayout lq, lo, ldo, lg;
  if (!layout_from(qkv_layout, shape, &lq) || !layout_from(o_layout, shape, &lo) ||
      !layout_from(do_layout, shape, &ldo) || !layout_from(dqkv_layout, shape, &lg))
    return TRIATTN_ERR_INVALID_ARG;
  const void* req[] = {q, k, v, bias, o, dO, dq, dk, dv, dbias};
  for (const void* p : req)
    if (p == nullptr || !aligned16(p)) return TRIATTN_ERR_INVALID_ARG;
  if (lse == nullptr || !aligned_to(lse, 4)) return TRIATTN_ERR_INVALID_ARG;
  if ((mask && !aligned_to(mask, 2)) || (o_resid && !aligned16(o_resid))) return TRIATTN_ERR_INVALID_ARG;
  const WsLayout w = ws_layout(shape, atomic_mask);
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || workspace_bytes < w.total)
    return TRIATTN_ERR_WORKSPACE;
  int dev = 0;
  if ((st = init_device(&dev)) != TRIATTN_OK) return st;
  BwdArgs a;
  std::memset(&a, 0, sizeof(a));
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.biasT = ws + w.biasT_off;
  if (!make_rows_map(&a.tm_q, q, shape, lq) || !make_rows_map(&a.tm_k, k, shape, lq) ||
      !make_rows_map(&a.tm_v, v, shape, lq) || !make_rows_map(&a.tm_do, dO, shape, ldo) ||
      !make_bias_map(&a.tm_biasT, a.biasT, shape, padded_n(shape->N)))
    return TRIATTN_ERR_CUDA;
  a.lq = lq;
  a.lo = lo;
  a.ldo = ldo;
  a.lg = lg;
  a.bias = bias;
  a.mask = mask;
  a.o = o;
  a.o_resid = o_resid;
  a.lse = lse;
  a.dO = dO;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.dbias = dbias;
  a.rec = reinterpret_cast<uint4*>(ws + w.rec_off);
  a.dq_part = reinterpret_cast<float*>(ws + w.dq_off);
  a.dbias_part = reinterpret_cast<float*>(ws + w.db_off);
  a.B = shape->B;
  a.N_o = shape->N_o;
  a.N = shape->N;
  a.H = shape->H;
  a.D = shape->D;
  a.dbias_fp32 = (shape->flags & TRIATTN_FLAG_DBIAS_FP32) ? 1 : 0;
  a.wc = wait_ctl(dev);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool d32 = shape->D == 32;
  cudaError_t e = cudaSuccess;
  if (dq_accumulated(atomic_mask)) e = cudaMemsetAsync(ws + w.dq_off, 0, w.db_off - w.dq_off, s);
  if (e == cudaSuccess && (atomic_mask & 2)) e = cudaMemsetAsync(ws + w.db_off, 0, w.total - w.db_off, s);
  if (e == cudaSuccess)
    e = traced(kKPre, s, [&] { return d32 ? launch_bwd_preprocess<32>(a, s) : launch_bwd_preprocess<16>(a, s); });
  if (e == cudaSuccess) e = traced(kKTrans, s, [&] { return launch_bwd_transpose_bias(a, s); });
  if (e == cudaSuccess && atomic_mask == 0)
    e = traced(kKMain, s, [&] { return d32 ? launch_bwd_main<32>(a, s) : launch_bwd_main<16>(a, s); });
  if (e == cudaSuccess && atomic_mask != 0)
    e = traced(kKMainAtomic, s, [&] {
      return d32 ? launch_bwd_main_atomic<32>(a, atomic_mask, s) : launch_bwd_main_atomic<16>(a, atomic_mask, s);
    });
  if (e == cudaSuccess && !dq_accumulated(atomic_mask))
    e = traced(kKRedDq, s, [&] { return d32 ? launch_bwd_reduce_dq<32>(a, s) : launch_bwd_reduce_dq<16>(a, s); });
  if (e == cudaSuccess && dq_accumulated(atomic_mask))
    e = traced(kKFinDq, s, [&] { return d32 ? launch_bwd_finish_dq<32>(a, s) : launch_bwd_finish_dq<16>(a, s); });
  if (e == cudaSuccess && !(atomic_mask & 2)) e = traced(kKRedDb, s, [&] { return launch_bwd_reduce_dbias(a, s); });
  if (e == cudaSuccess && (atomic_mask & 2)) e = traced(kKFinDb, s, [&] { return launch_bwd_finish_dbias(a, s); });
  return e == cudaSuccess ? TRIATTN_OK : TRIATTN_ERR_CUDA;
}

}  // namespace

extern "C" {

const char* triattn_status_string(triattn_status s) {
  switch (s) {
    case TRIATTN_OK: return "TRIATTN_OK";
    case TRIATTN_ERR_INVALID_ARG: return "TRIATTN_ERR_INVALID_ARG";
    case TRIATTN_ERR_UNSUPPORTED: return "TRIATTN_ERR_UNSUPPORTED";
    case TRIATTN_ERR_WORKSPACE: return "TRIATTN_ERR_WORKSPACE";
    case TRIATTN_ERR_CUDA: return "TRIATTN_ERR_CUDA";
    case TRIATTN_ERR_TIMEOUT: return "TRIATTN_ERR_TIMEOUT";
  }
  return "TRIATTN_ERR_UNKNOWN";
}

size_t triattn_bwd_workspace_bytes(const triattn_shape* shape) {
  if (check_shape(shape) != TRIATTN_OK) return 0;
  return ws_layout(shape).total;
}

size_t triattn_fwd_workspace_bytes(const triattn_shape* shape) {
  if (check_shape(shape) != TRIATTN_OK) return 0;
  return fwd_ws(shape, true).total();
}

}  // extern "C"

namespace {

triattn_status fwd_impl(const triattn_shape* shape, const void* q, const void* k, const void* v,
                        const triattn_layout* qkv_layout, const void* bias, const void* mask, void* o, float* lse,
                        void* o_resid, const triattn_layout* o_layout, void* workspace, size_t workspace_bytes,
                        void* stream) {
  triattn_status st = check_shape(shape);
  if (st != TRIATTN_OK) return st;
  RowLayout lq, lo;
  if (!layout_from(qkv_layout, shape, &lq) || !layout_from(o_layout, shape, &lo)) return TRIATTN_ERR_INVALID_ARG;
  const void* req[] = {q, k, v, bias, o};
  for (const void* p : req)
    if (p == nullptr || !aligned16(p)) return TRIATTN_ERR_INVALID_ARG;
  if (lse == nullptr || !aligned_to(lse, 4)) return TRIATTN_ERR_INVALID_ARG;
  if ((mask && !aligned_to(mask, 2)) || (o_resid && !aligned16(o_resid))) return TRIATTN_ERR_INVALID_ARG;
  const FwdWs fw = fwd_ws(shape, mask != nullptr);
  if (fw.total() > 0 &&
      (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || workspace_bytes < fw.total()))
    return TRIATTN_ERR_WORKSPACE;
  int dev = 0;
  if ((st = init_device(&dev)) != TRIATTN_OK) return st;
  FwdArgs a;
  std::memset(&a, 0, sizeof(a));
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.mrec = fw.rec_bytes > 0 ? ws : nullptr;
  a.bias_padded = fw.pad_bytes > 0 ? ws + fw.pad_off : nullptr;
  a.bias = bias;
  const void* bias_read = a.bias_padded != nullptr ? a.bias_padded : bias;
  a.lq = lq;
  a.lo = lo;
  if (!make_rows_map(&a.tm_q, q, shape, lq) || !make_rows_map(&a.tm_k, k, shape, lq, 64) ||
      !make_rows_map(&a.tm_v, v, shape, lq, 64) ||
      !make_bias_map(&a.tm_bias, bias_read, shape, a.bias_padded != nullptr ? padded_n(shape->N) : shape->N))
    return TRIATTN_ERR_CUDA;
  a.mask = mask;
  a.o = o;
  a.lse = lse;
  a.o_resid = o_resid;
  a.B = shape->B;
  a.N_o = shape->N_o;
  a.N = shape->N;
  a.H = shape->H;
  a.test_starve = g_test_starve.load();
  a.wc = wait_ctl(dev);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  if (a.mrec != nullptr || a.bias_padded != nullptr) e = traced(kKFwdPrep, s, [&] { return launch_fwd_prep(a, s); });
  if (e == cudaSuccess)
    e = traced(kKFwd, s, [&] { return (shape->D == 32) ? launch_fwd<32>(a, s) : launch_fwd<16>(a, s); });
  return e == cudaSuccess ? TRIATTN_OK : TRIATTN_ERR_CUDA;
}

}  // namespace

extern "C" {

triattn_status tri_attn_fwd(const triattn_shape* shape, const void* q, const void* k, const void* v,
                            const void* bias, const void* mask, void* o, float* lse, void* o_resid,
                            void* workspace, size_t workspace_bytes, void* stream) {
  return fwd_impl(shape, q, k, v, nullptr, bias, mask, o, lse, o_resid, nullptr, workspace, workspace_bytes, stream);
}

triattn_status tri_attn_fwd_strided(const triattn_shape* shape, const void* q, const void* k, const void* v,
                                    const triattn_layout* qkv_layout, const void* bias, const void* mask, void* o,
                                    float* lse, void* o_resid, const triattn_layout* o_layout, void* workspace,
                                    size_t workspace_bytes, void* stream) {
  if (qkv_layout == nullptr || o_layout == nullptr) return TRIATTN_ERR_INVALID_ARG;
  return fwd_impl(shape, q, k, v, qkv_layout, bias, mask, o, lse, o_resid, o_layout, workspace, workspace_bytes,
                  stream);
}

triattn_status tri_attn_bwd(const triattn_shape* shape, const void* q, const void* k, const void* v,
                            const void* bias, const void* mask, const void* o, const void* o_resid, const float* lse,
                            const void* dO, void* dq, void* dk, void* dv, void* dbias, void* workspace,
                            size_t workspace_bytes, void* stream) {
  return bwd_impl(shape, q, k, v, nullptr, bias, mask, o, o_resid, nullptr, lse, dO, nullptr, dq, dk, dv, nullptr,
                  dbias, 0, workspace, workspace_bytes, stream);
}

triattn_status tri_attn_bwd_strided(const triattn_shape* shape, const void* q, const void* k, const void* v,
                                    const triattn_layout* qkv_layout, const void* bias, const void* mask,
                                    const void* o, const void* o_resid, const triattn_layout* o_layout,
                                    const float* lse, const void* dO, const triattn_layout* do_layout, void* dq,
                                    void* dk, void* dv, const triattn_layout* dqkv_layout, void* dbias,
                                    void* workspace, size_t workspace_bytes, void* stream) {
  if (qkv_layout == nullptr || o_layout == nullptr || do_layout == nullptr || dqkv_layout == nullptr)
    return TRIATTN_ERR_INVALID_ARG;
  return bwd_impl(shape, q, k, v, qkv_layout, bias, mask, o, o_resid, o_layout, lse, dO, do_layout, dq, dk, dv,
                  dqkv_layout, dbias, 0, workspace, workspace_bytes, stream);
}

size_t triattn_bwd_atomic_workspace_bytes(const triattn_shape* shape, int atomic_mask) {
  if (check_shape(shape) != TRIATTN_OK || !atomic_mask_ok(atomic_mask)) return 0;
  return ws_layout(shape, atomic_mask).total;
}

triattn_status tri_attn_bwd_atomic_ablation(const triattn_shape* shape, const void* q, const void* k, const void* v,
                                            const void* bias, const void* mask, const void* o, const void* o_resid,
                                            const float* lse, const void* dO, void* dq, void* dk, void* dv,
                                            void* dbias, int atomic_mask, void* workspace, size_t workspace_bytes,
                                            void* stream) {
  if (!atomic_mask_ok(atomic_mask)) return TRIATTN_ERR_INVALID_ARG;
  if (shape != nullptr && shape->flags != 0) return TRIATTN_ERR_INVALID_ARG;
  return bwd_impl(shape, q, k, v, nullptr, bias, mask, o, o_resid, nullptr, lse, dO, nullptr, dq, dk, dv, nullptr,
                  dbias, atomic_mask, workspace, workspace_bytes, stream);
}

triattn_status tri_attn_dbias_combine(const triattn_shape* shape, const float* parts, int R, void* dbias,
                                      void* stream) {
  if (shape == nullptr || R < 1 || parts == nullptr || dbias == nullptr || !aligned16(parts) || !aligned16(dbias))
    return TRIATTN_ERR_INVALID_ARG;
  if (shape->B < 1 || shape->H < 1 || shape->N < 1) return TRIATTN_ERR_INVALID_ARG;
  int dev = 0;
  triattn_status st = init_device(&dev);
  if (st != TRIATTN_OK) return st;
  const size_t elems = static_cast<size_t>(shape->B) * shape->H * shape->N * shape->N;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const cudaError_t e = traced(kKCombine, s, [&] { return launch_dbias_combine(parts, R, elems, dbias, s); });
  return e == cudaSuccess ? TRIATTN_OK : TRIATTN_ERR_CUDA;
}

triattn_status triattn_device_status(void* stream) {
  int dev = 0;
  triattn_status st = init_device(&dev);
  if (st != TRIATTN_OK) return st;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return TRIATTN_ERR_CUDA;
  uint32_t word = 0;
  if (cudaMemcpy(&word, g_status_ptr[dev], sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
    return TRIATTN_ERR_CUDA;
  if (word == 0) return TRIATTN_OK;
  const uint32_t zero = 0;
  if (cudaMemcpy(g_status_ptr[dev], &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
    return TRIATTN_ERR_CUDA;
  return (word & kDevTimeout) ? TRIATTN_ERR_TIMEOUT : TRIATTN_ERR_CUDA;
}

void triattn_set_wait_limit_ns(unsigned long long cap_ns) {
  g_wait_limit_ns.store(cap_ns > 0 ? cap_ns : kDefaultWaitNs);
}

void triattn_trace_enable(int on) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  if (on) {
    g_trace.clear();
    g_event_next = 0;
  }
  g_trace_on = on != 0;
}

int triattn_trace_read(triattn_trace_entry* out, int max_entries) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  triattn_trace_entry acc[kKinds];
  for (int k = 0; k < kKinds; ++k) acc[k] = {kKernelName[k], 0, 0.0, 1e30, 0.0};
  for (const TraceRec& r : g_trace) {
    float ms = 0.f;
    if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess) return -1;
    triattn_trace_entry& e = acc[r.kind];
    e.launches += 1;
    e.total_ms += ms;
    if (ms < e.min_ms) e.min_ms = ms;
    if (ms > e.max_ms) e.max_ms = ms;
  }
  int n = 0;
  for (int k = 0; k < kKinds && n < max_entries; ++k)
    if (acc[k].launches > 0 && out != nullptr) out[n++] = acc[k];
  return n;
}

void triattn_test_set_starve(int on) { g_test_starve.store(on != 0 ? 1 : 0); }

size_t triattn_gemm_workspace_bytes(int M, int N, int K, int batch) {
  if (M < 1 || N < 1 || K < 1 || batch < 1) return 0;
  return gemm_splitk_bytes(M, N, K, batch);
}

triattn_status triattn_gemm(int ta, int tb, int M, int N, int K, const void* A, long long lda, const void* B,
                            long long ldb, void* C, long long ldc, int c_f32, int batch, long long sA, long long sB,
                            long long sC, void* workspace, size_t workspace_bytes, void* stream) {
  if (M < 1 || N < 1 || K < 1 || batch < 1 || A == nullptr || B == nullptr || C == nullptr)
    return TRIATTN_ERR_INVALID_ARG;
  if (lda < (ta ? M : K) || ldb < (tb ? K : N) || ldc < N) return TRIATTN_ERR_INVALID_ARG;
  int dev = 0;
  triattn_status st = init_device(&dev);
  if (st != TRIATTN_OK) return st;
  const WaitCtl wc = wait_ctl(dev);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const cudaError_t e = traced(kKGemm, s, [&] {
    return launch_gemm(ta != 0, tb != 0, M, N, K, A, lda, B, ldb, C, ldc, c_f32 != 0, batch, sA, sB, sC, workspace,
                       workspace_bytes, wc, s);
  });
  if (e == cudaErrorInvalidValue) return TRIATTN_ERR_INVALID_ARG;
  return e == cudaSuccess ? TRIATTN_OK : TRIATTN_ERR_CUDA;
}

}  // extern "C"
