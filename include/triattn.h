/*
 * libtriattn — triangular (pair-biased, slice-batched) attention, forward and
 * backward, on one NVIDIA GB300 (sm_103a).
 *
 * The operation ("TurboPairFormer: Fast and Stable Protein Folding Model
 * Training with an Optimized Triangle Attention Kernel", Abstract, Figure 1(a),
 * Table 1 and Figure 6): for every example b, outer slice o, head h,
 *
 *   S[q,k]  = Q[b,o,h,q,:] . K[b,o,h,k,:] / sqrt(D) + bias[b,h,q,k] + mask[b,o,k]
 *   O[b,o,h,q,:] = sum_k softmax_k(S)[q,k] V[b,o,h,k,:]
 *
 * with ONE pair bias shared by all N_o slices.  The backward returns dQ, dK,
 * dV and dbias, where dbias[b,h] is the sum over slices o of dS_o
 * (Figure 1(a): the third reduction axis).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All tensor pointers are DEVICE pointers to contiguous row-major arrays,
 *    16-byte aligned, except the key mask (2-byte aligned) and lse (4-byte
 *    aligned), so that a shard of the outer axis may start at any slice.
 *    "bf16" means IEEE bfloat16 stored as uint16.
 *  - Layouts (the strided entry points below take q, k, v, o, o_resid, dO,
 *    dq, dk, dv in other row layouts):
 *             q, k, v, o, o_resid, dO, dq, dk, dv  [B, N_o, H, N, D] bf16
 *             bias, dbias                         [B, H, N, N]      bf16
 *             mask (optional, additive)           [B, N_o, N]       bf16
 *             lse                                 [B, N_o, H, N]    fp32 (natural log)
 *  - The method has N_o = N outer slices (Table 1); a call may also take a
 *    contiguous shard of them (one GPU's part when the outer axis is split
 *    across GPUs): 1 <= N_o <= N.  D must be 16 or 32; any N >= 1 works,
 *    ragged or not relative to the tiles, up to the grid and 32-bit index
 *    limits (ceil(N_o / 4) <= 65535, B*H <= 65535, B*(N_o + 4)*H < 2^31,
 *    N * ceil(N / 128) * 128 < 2^31; beyond them TRIATTN_ERR_UNSUPPORTED).
 *    When N is not a multiple of 8, the forward reads the bias from a copy
 *    with rows padded to 16 bytes in its workspace, and the backward's
 *    transposed copy is padded the same way.  The backward's FP32 partials
 *    grow as N_o * N^2 (triattn_bwd_workspace_bytes); for long crops run the
 *    outer axis in chunks with TRIATTN_FLAG_DBIAS_FP32 and combine them with
 *    tri_attn_dbias_combine.
 *  - A row whose keys are all masked (every score -inf) yields O = 0,
 *    residual 0, lse = -inf and zero gradient contributions.
 *  - The caller owns every buffer, the workspace and the stream.  The library
 *    allocates no device memory; it keeps only host-side state (TMA
 *    descriptors are built per call; kernel attributes are set on a device's
 *    first call, and set again if a device reset has cleared them).
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *    default stream).  Argument errors are returned synchronously and nothing
 *    is launched.  A launch failure returns TRIATTN_ERR_CUDA.  A device-side
 *    wait that exceeds its time limit (about 2 s) is recorded in a device
 *    status word that triattn_device_status() reads back.
 *  - Results are bitwise reproducible across calls with the same inputs and
 *    shape: no floating-point atomics are used, every reduction has a fixed
 *    order, and the kernel configuration depends only on (D, N).
 */
#ifndef TRIATTN_H_
#define TRIATTN_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  int B;          /* examples */
  int N_o;        /* outer slices: N, or a contiguous shard of them (1 <= N_o <= N) */
  int N;          /* tokens per crop (queries = keys = N) */
  int H;          /* heads */
  int D;          /* features per head: 16 or 32 */
  unsigned flags; /* 0, or TRIATTN_FLAG_DBIAS_FP32 (backward only) */
} triattn_shape;

/*
 * Backward flag: write dbias as FP32 [B, H, N, N] (the FP32 sum over this
 * call's outer slices, not rounded) instead of BF16.  Used when the outer
 * axis is split across GPUs: every GPU's FP32 dbias is gathered and
 * tri_attn_dbias_combine() adds them in rank order and rounds once.  Other
 * flag bits are rejected with TRIATTN_ERR_INVALID_ARG; the forward accepts
 * and ignores this one.
 */
#define TRIATTN_FLAG_DBIAS_FP32 1u

typedef enum {
  TRIATTN_OK = 0,
  TRIATTN_ERR_INVALID_ARG = 1,  /* null / misaligned pointer, bad shape field */
  TRIATTN_ERR_UNSUPPORTED = 2,  /* D not in {16, 32}, a shape outside the supported set, size overflow */
  TRIATTN_ERR_WORKSPACE = 3,    /* workspace missing or smaller than required */
  TRIATTN_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed */
  TRIATTN_ERR_TIMEOUT = 5       /* a device wait exceeded its limit */
} triattn_status;

/* Human-readable name of a status code (static string, never NULL). */
const char* triattn_status_string(triattn_status s);

/*
 * Workspace bytes tri_attn_fwd may need for `shape` (0 on an invalid shape,
 * and 0 when no call of that shape needs one): the key-mask records, one of
 * 144 bytes per (slice, 64-key tile) plus four padding slices, and, when N
 * is not a multiple of 8, the bias copied with 16-byte aligned rows.
 */
size_t triattn_fwd_workspace_bytes(const triattn_shape* shape);

/*
 * Forward.  "TurboPairFormer", Abstract and Figure 1(a) (the operation),
 * Figure 7(b) and Figure 9 (the saved output residual).
 *
 *   o       [B,N_o,H,N,D] bf16  out: O rounded once (round-to-nearest) from FP32.
 *   lse     [B,N_o,H,N]   fp32  out: log sum_k exp(S[q,k]) (natural log).
 *   o_resid [B,N_o,H,N,D] bf16  out, optional (NULL = not written): the
 *           output-rounding residual E = bf16(O_fp32 - float(o)), the BF16
 *           approximation of what rounding O to BF16 lost.  The backward uses
 *           o + o_resid for its softmax correction.
 *   mask    optional (NULL = no mask).
 *   workspace  device scratch of triattn_fwd_workspace_bytes(shape) bytes,
 *           256-byte aligned, contents ignored.  It may be NULL (with 0
 *           bytes) when mask is NULL and N is a multiple of 64: the forward
 *           then needs none.
 * Launches the forward kernel, preceded (when the workspace is used) by one
 * small kernel that writes the key-mask records and the padded bias.
 */
triattn_status tri_attn_fwd(const triattn_shape* shape,
                            const void* q, const void* k, const void* v,
                            const void* bias, const void* mask,
                            void* o, float* lse, void* o_resid,
                            void* workspace, size_t workspace_bytes,
                            void* stream);

/*
 * Workspace bytes tri_attn_bwd needs for `shape` (0 on an invalid shape).
 * The workspace holds, per query row, a 16-byte record of -lse*sqrt(D) and
 * -delta (each split into three BF16 terms); a transposed copy of the bias; the
 * single-writer FP32 dQ partials (one per key tile) and the single-writer
 * FP32 dbias partials (one per outer group of 4 slices at D = 32, 8 at
 * D = 16) ("TurboPairFormer",
 * Figure 2(b), Figure 7, Table 11).
 */
size_t triattn_bwd_workspace_bytes(const triattn_shape* shape);

/*
 * Backward.  "TurboPairFormer", Abstract, Figure 2, Figure 7(b)-(d),
 * Figure 11(a) and Table 11 (key-tile-parallel partition):
 *   1. preprocess: delta[q] = sum_d dO[q,d] * (o[q,d] + o_resid[q,d]) in FP32
 *      (o_resid NULL: compensation off, delta = sum_d dO*o); per query row a
 *      16-byte record holds -lse[q]*sqrt(D) and -delta[q], each split into
 *      three BF16 terms;
 *   2. a small kernel writes the bias transposed (key-major) into the
 *      workspace;
 *   3. main: one CTA per (b, h, key tile, outer group of slices) recomputes
 *      S, P, dP and dS once per query tile, keeps dK and dV on chip and
 *      writes one FP32 dQ partial per key tile and one FP32 dbias partial per
 *      outer group, each with a single writer;
 *   4. a reduction kernel adds the dQ partials in ascending key-tile order;
 *   5. a reduction kernel adds the dbias partials in ascending group order.
 *
 *   q,k,v,bias,mask  the forward's inputs (mask may be NULL).
 *   o, lse           the forward's outputs; o_resid optional (see above).
 *   dO               [B,N_o,H,N,D] bf16 incoming gradient.
 *   dq, dk, dv       [B,N_o,H,N,D] bf16 out.
 *   dbias            [B,H,N,N] bf16 out.
 *   workspace        device scratch of at least
 *                    triattn_bwd_workspace_bytes(shape) bytes, 256-byte
 *                    aligned; contents on entry are ignored.
 * Launches five kernels in stream order.
 */
triattn_status tri_attn_bwd(const triattn_shape* shape,
                            const void* q, const void* k, const void* v,
                            const void* bias, const void* mask,
                            const void* o, const void* o_resid, const float* lse,
                            const void* dO,
                            void* dq, void* dk, void* dv, void* dbias,
                            void* workspace, size_t workspace_bytes,
                            void* stream);

/*
 * The same forward and backward on tensors in other row layouts, e.g. the
 * heads of a projection's pair rows read and written where they lie (the
 * module below), with results bitwise equal to the contiguous calls on the
 * same values.
 *
 * A layout places row (b, o, h, n) of a [B, N_o, H, N, D] tensor, its D
 * features contiguous, at element  slice * (b N_o + o) + head * h + row * n
 * from the tensor's base pointer.  The contiguous layout of the calls above
 * is {H N D, N D, D}; H heads side by side at column c of the pair rows of a
 * row-major [B, N, N, ld] matrix are {N ld, D, ld} from base + c.
 * Requirements (else TRIATTN_ERR_INVALID_ARG): every stride a positive
 * multiple of 8 elements and the rows of one tensor disjoint, nested by
 * stride -- with a = min(head, row), b = max(head, row) and n_a, n_b the
 * counts of heads or rows they step over (H or N): (n_a - 1) a + D <= b and
 * (n_b - 1) b + (n_a - 1) a + D <= slice < 2^36, head and row different
 * unless H or N is 1, and slice = H head when head > row (both layouts above
 * qualify).  The caller keeps the rows of one tensor from overlapping those
 * of another that a call writes.
 *   qkv_layout   q, k, v (forward and backward)
 *   o_layout     o and o_resid (forward and backward)
 *   do_layout    dO (backward)
 *   dqkv_layout  dq, dk, dv (backward)
 * (all four required on the backward).
 * lse, bias, mask, dbias, the workspaces and every other rule are those of
 * tri_attn_fwd / tri_attn_bwd.  The ablation entry points take the
 * contiguous layout only.
 */
typedef struct {
  long long slice; /* elements between consecutive (b, o) slices, index b N_o + o */
  long long head;  /* elements between consecutive heads */
  long long row;   /* elements between consecutive tokens n */
} triattn_layout;

triattn_status tri_attn_fwd_strided(const triattn_shape* shape,
                                    const void* q, const void* k, const void* v,
                                    const triattn_layout* qkv_layout,
                                    const void* bias, const void* mask,
                                    void* o, float* lse, void* o_resid,
                                    const triattn_layout* o_layout,
                                    void* workspace, size_t workspace_bytes,
                                    void* stream);
triattn_status tri_attn_bwd_strided(const triattn_shape* shape,
                                    const void* q, const void* k, const void* v,
                                    const triattn_layout* qkv_layout,
                                    const void* bias, const void* mask,
                                    const void* o, const void* o_resid,
                                    const triattn_layout* o_layout,
                                    const float* lse,
                                    const void* dO, const triattn_layout* do_layout,
                                    void* dq, void* dk, void* dv,
                                    const triattn_layout* dqkv_layout,
                                    void* dbias,
                                    void* workspace, size_t workspace_bytes,
                                    void* stream);

/*
 * Allocation-free backward.  The paper has no counterpart to this entry
 * point; it is a deployment convenience of this library.
 *
 * Some callers cannot allocate device memory: a plugin inside a host
 * framework that owns all device memory and does not let extensions call
 * cudaMalloc, or a latency-critical loop that cannot pay for cudaMalloc's
 * implicit device synchronisation.  This entry point runs the same five
 * backward kernels as tri_attn_bwd but takes no workspace: its scratch
 * (the row records, the transposed bias and the FP32 partials) lives in a
 * file-scope device array of
 * TRIATTN_NOALLOC_SCRATCH_BYTES (64 MiB) inside the library, which every GPU
 * that loads the library holds until the process exits.
 *   - A shape whose triattn_bwd_workspace_bytes() exceeds
 *     TRIATTN_NOALLOC_SCRATCH_BYTES is rejected with TRIATTN_ERR_WORKSPACE
 *     before anything is launched (B=1, N=48, H=2, D=16 needs 1.6 MiB;
 *     a 384-token crop with H=4, D=32 needs 438 MiB and is rejected).
 *   - Every call looks up the array's device address on the current device
 *     with cudaGetSymbolAddress (no allocation; a device reset gives the
 *     array a new address).  The first call on a device may also load the
 *     library's device code there: make that first call before any stream
 *     capture.
 *   - It calls no cudaMalloc, no cudaFree and no allocating library routine.
 *   - Every call uses the same array, which keeps the previous call's
 *     contents.  Nothing needs clearing: the kernels write every scratch word
 *     before they read it.  Calls that overlap on the GPU (other streams, or
 *     other host threads without ordering) race on the array; the caller
 *     must serialise them.
 * Arguments, layouts and the other error codes are those of tri_attn_bwd.
 */
#define TRIATTN_NOALLOC_SCRATCH_BYTES (64ull << 20)
triattn_status tri_attn_bwd_noalloc(const triattn_shape* shape,
                                    const void* q, const void* k, const void* v,
                                    const void* bias, const void* mask,
                                    const void* o, const void* o_resid, const float* lse,
                                    const void* dO,
                                    void* dq, void* dk, void* dv, void* dbias,
                                    void* stream);

/*
 * ABLATION ONLY, not the library's backward: the same computation with the
 * single-writer FP32 partials of dQ (atomic_mask = 1), of dbias (2) or of
 * both (3) replaced by FP32 atomic adds into zero-initialised FP32
 * accumulators, or the dQ partials replaced by TMA bulk reductions
 * (cp.reduce.async.bulk ... add.f32, one per 128-row dQ tile, this GPU's
 * memory only) into such an accumulator (4), alone or with atomic dbias (6);
 * small kernels then round the accumulators to BF16 (the non-deterministic
 * variants of "TurboPairFormer", Section "Deterministic reductions",
 * Table 12).  It exists to measure what the ordered partials
 * cost; the atomically added gradients are NOT bitwise reproducible between
 * calls (FP32 addition order varies), dK, dV and the ordered one are.
 * Arguments are those of tri_attn_bwd; the workspace must hold
 * triattn_bwd_atomic_workspace_bytes(shape, atomic_mask) bytes (the row
 * records, the transposed bias, then the FP32 accumulators
 * [B*N_o*H][J_Q*128][D] for dQ and [B*H][J_K*128][J_Q*128] for dbias, or
 * the partials of the operand that stays ordered).  atomic_mask other than
 * 1, 2, 3, 4 or 6 returns TRIATTN_ERR_INVALID_ARG (and 0 bytes).
 */
size_t triattn_bwd_atomic_workspace_bytes(const triattn_shape* shape, int atomic_mask);
triattn_status tri_attn_bwd_atomic_ablation(const triattn_shape* shape,
                                            const void* q, const void* k, const void* v,
                                            const void* bias, const void* mask,
                                            const void* o, const void* o_resid, const float* lse,
                                            const void* dO,
                                            void* dq, void* dk, void* dv, void* dbias,
                                            int atomic_mask,
                                            void* workspace, size_t workspace_bytes,
                                            void* stream);

/*
 * dbias of an outer axis split across R GPUs: dbias = bf16(sum over r of
 * parts[r]), the FP32 additions in ascending r (so the result is bitwise
 * reproducible and independent of how the parts were gathered).  `parts` is
 * [R][B, H, N, N] FP32 (each part written by tri_attn_bwd with
 * TRIATTN_FLAG_DBIAS_FP32 on its shard), `dbias` [B, H, N, N] BF16; the
 * shape's N_o and flags are not used.  R < 1 returns TRIATTN_ERR_INVALID_ARG.
 */
triattn_status tri_attn_dbias_combine(const triattn_shape* shape, const float* parts, int R, void* dbias,
                                      void* stream);

/*
 * The triangle-attention module around the core ("TurboPairFormer",
 * Figure 6 and its worked example; shapes from Table 1): with M = B*N*N
 * pairs of C features each,
 *
 *   x    = LayerNorm(z; ln_w, ln_b)  over the C features of each pair, eps 1e-5
 *   P    = x W_in                    W_in [C, 3HD + H]
 *   q, k, v [b, i, h, j, :] = P[(b, i, j), {0, HD, 2HD} + h D + (0 .. D-1)]
 *   bias [b, h, i, j]       = P[(b, i, j), 3HD + h]
 *   o    = tri_attn_fwd(q, k, v, bias, mask)     (N_o = N)
 *   out  = o_flat W_o                W_o [HD, C], o_flat[(b, i, j), h D + d] = o[b, i, h, j, d]
 *
 * No projection biases and no gate; the residual update z + out is left to
 * the caller.  The projections are the library's tensor-core GEMM
 * (triattn_gemm: BF16 operands, FP32 accumulation); the core is
 * tri_attn_fwd_strided / tri_attn_bwd_strided, reading q, k, v from P's pair
 * rows and writing o into o_flat, dq, dk, dv into dP's pair rows where they
 * lie; the LayerNorm, the bias planes and the LayerNorm's parameter-gradient
 * sums are the library's kernels.
 *
 * Shape: B >= 1, N as for the core (multiple of 8, 8..4096), B*N*N < 2^31,
 * C a multiple of 32 up to 256, H up to 64, D 16 or 32, flags 0.  Otherwise
 * TRIATTN_ERR_INVALID_ARG (non-positive field, flags) or
 * TRIATTN_ERR_UNSUPPORTED; the size queries return 0.
 *
 * Layouts (device pointers, contiguous row-major, 16-byte aligned):
 *   z, dz    [B, N, N, C] bf16        out, d_out [B, N, N, C] bf16
 *   ln_w, ln_b, d_ln_w, d_ln_b  [C] fp32
 *   w_in [C, 3HD + H] bf16, w_o [HD, C] bf16
 *   d_w_in [C, 3HD + H] fp32, d_w_o [HD, C] fp32   (overwritten, not accumulated)
 *   mask  optional [B, N, N] bf16 additive key mask of each slice (the core's)
 *   ctx   triattn_module_ctx_bytes(shape) bytes, 256-byte aligned: written by
 *         the forward (x, the LayerNorm statistics, P, the bias planes, lse,
 *         the output residual, o_flat), read by the backward of the same
 *         inputs.
 *   workspace  triattn_module_workspace_bytes(shape) bytes, 256-byte
 *         aligned, contents ignored; either call may use it (it also serves
 *         for the GEMMs' split-K partials and the core's workspaces).
 *
 * Results are bitwise reproducible for a fixed shape and device: every
 * reduction, the GEMMs' split-K sums included, has a fixed order.  Argument
 * errors return before anything is launched; a failed launch returns
 * TRIATTN_ERR_CUDA.
 */
typedef struct {
  int B;          /* examples */
  int N;          /* tokens per crop */
  int C;          /* pair features */
  int H;          /* heads */
  int D;          /* features per head: 16 or 32 */
  unsigned flags; /* 0 */
} triattn_module_shape;

size_t triattn_module_ctx_bytes(const triattn_module_shape* shape);
size_t triattn_module_workspace_bytes(const triattn_module_shape* shape);

/* Forward: writes out and ctx. */
triattn_status tri_attn_module_fwd(const triattn_module_shape* shape, const void* z, const void* mask,
                                   const float* ln_w, const float* ln_b, const void* w_in, const void* w_o,
                                   void* out, void* ctx, void* workspace, size_t workspace_bytes, void* stream);

/* Backward of <out, d_out>: dz (bf16), d_ln_w, d_ln_b, d_w_in, d_w_o (fp32).
 * z, mask, ln_w, w_in, w_o and ctx must be those of the forward call. */
triattn_status tri_attn_module_bwd(const triattn_module_shape* shape, const void* z, const void* mask,
                                   const float* ln_w, const void* w_in, const void* w_o, const void* ctx,
                                   const void* d_out, void* dz, float* d_ln_w, float* d_ln_b, float* d_w_in,
                                   float* d_w_o, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Triangle multiplicative update, outgoing or incoming ("TurboPairFormer",
 * Figure 12; shapes from Table 10).  With M = B*N*N pairs:
 *
 *   x   = LayerNorm(z; ln_in_w, ln_in_b)            over C_z, eps 1e-5
 *   p   = x W_p                                     W_p [C_z, 4 C_h + C_z], columns
 *                                                   a_v | a_g | b_v | b_g | g
 *   a   = m * sigmoid(a_g) * a_v,  b = m * sigmoid(b_g) * b_v   (m: pair mask)
 *   outgoing: X[b,i,j,c] = sum_k a[b,i,k,c] * b[b,j,k,c]
 *   incoming: X[b,i,j,c] = sum_k a[b,k,i,c] * b[b,k,j,c]
 *   out = sigmoid(g) * (LayerNorm(X; ln_out_w, ln_out_b) W_o)   W_o [C_h, C_z]
 *
 * No projection biases; the residual update z + out is left to the caller.
 * The projections and the per-channel contraction are the library's
 * tensor-core GEMM (triattn_gemm: BF16 operands, FP32 accumulation; the
 * contraction one batched GEMM over the B*C_h channel matrices).  The input
 * projection applies the gating and masking in its epilogue, from the FP32
 * accumulators, and writes a, b channel-major and g: p itself is never
 * stored, and the backward recomputes its branch columns.  The LayerNorms,
 * the output gate and the parameter-gradient sums are the library's kernels.
 *
 * Shape: B >= 1; N a multiple of 8, 8..4096, B*N*N < 2^31; C_z a multiple of
 * 32 up to 256; C_h 32, 64, 96 or 128; direction TRIATTN_TRIMUL_OUTGOING or
 * TRIATTN_TRIMUL_INCOMING; flags 0.  Otherwise TRIATTN_ERR_INVALID_ARG
 * (non-positive field, direction, flags) or TRIATTN_ERR_UNSUPPORTED; the size
 * queries return 0.
 *
 * Layouts (device pointers, contiguous row-major, 16-byte aligned):
 *   z, dz, out, d_out  [B, N, N, C_z] bf16
 *   mask               optional [B, N, N] bf16, multiplicative (1 keeps a pair, 0 drops it)
 *   ln_in_w, ln_in_b, d_ln_in_w, d_ln_in_b    [C_z] fp32
 *   ln_out_w, ln_out_b, d_ln_out_w, d_ln_out_b [C_h] fp32
 *   w_p [C_z, 4 C_h + C_z] bf16, w_o [C_h, C_z] bf16
 *   d_w_p, d_w_o       same shapes, fp32 (overwritten, not accumulated)
 *   ctx   triattn_trimul_ctx_bytes(shape) bytes, 256-byte aligned: written
 *         by the forward (x and its statistics, g, the channel-major a, b
 *         and X, the output LayerNorm statistics, its output y, and
 *         u = y W_o), read by the backward of the same inputs.
 *   workspace  triattn_trimul_workspace_bytes(shape) bytes, 256-byte
 *         aligned, contents ignored (also the GEMMs' split-K partials).
 *
 * Bitwise reproducible for a fixed shape and device.  Argument errors
 * return before anything is launched; a failed launch returns
 * TRIATTN_ERR_CUDA.
 */
#define TRIATTN_TRIMUL_OUTGOING 0
#define TRIATTN_TRIMUL_INCOMING 1

typedef struct {
  int B;          /* examples */
  int N;          /* tokens per crop */
  int C_z;        /* pair features */
  int C_h;        /* hidden channels of the contraction */
  int direction;  /* TRIATTN_TRIMUL_OUTGOING or TRIATTN_TRIMUL_INCOMING */
  unsigned flags; /* 0 */
} triattn_trimul_shape;

size_t triattn_trimul_ctx_bytes(const triattn_trimul_shape* shape);
size_t triattn_trimul_workspace_bytes(const triattn_trimul_shape* shape);

/* Forward: writes out and ctx. */
triattn_status triattn_trimul_fwd(const triattn_trimul_shape* shape, const void* z, const void* mask,
                                  const float* ln_in_w, const float* ln_in_b, const void* w_p,
                                  const float* ln_out_w, const float* ln_out_b, const void* w_o, void* out,
                                  void* ctx, void* workspace, size_t workspace_bytes, void* stream);

/* Backward of <out, d_out>: dz (bf16) and the fp32 parameter gradients.
 * z, mask, the parameters and ctx must be those of the forward call. */
triattn_status triattn_trimul_bwd(const triattn_trimul_shape* shape, const void* z, const void* mask,
                                  const float* ln_in_w, const void* w_p, const float* ln_out_w, const void* w_o,
                                  const void* ctx, const void* d_out, void* dz, float* d_ln_in_w, float* d_ln_in_b,
                                  float* d_w_p, float* d_ln_out_w, float* d_ln_out_b, float* d_w_o,
                                  void* workspace, size_t workspace_bytes, void* stream);

/*
 * The library's tensor-core GEMM, as used by the multiplicative update and
 * the module (exported so that it can be tested and reused; not one of the
 * method's operations).  Row-major C[M, N] = op(A) op(B): A is [M, K] with
 * row stride lda, or [K, M] when ta != 0; B is [K, N] with row stride ldb,
 * or [N, K] when tb != 0; BF16 operands, FP32 accumulation; C is BF16, or
 * FP32 when c_f32 != 0, with row stride ldc.  `batch` matrices are sA, sB,
 * sC elements apart.  Strides are in elements: lda, ldb (and sA, sB when
 * batch > 1) multiples of 8, A and B 16-byte aligned; C 16-byte aligned
 * with ldc a multiple of 8 (BF16) or 4 (FP32).  When the output tiles
 * cannot fill the GPU, K is split into FP32 partials in `workspace` (at
 * least triattn_gemm_workspace_bytes() bytes, 16-byte aligned; NULL runs
 * unsplit) that a second kernel adds in fixed order: bitwise reproducible.
 * Invalid arguments return TRIATTN_ERR_INVALID_ARG before any launch.
 */
size_t triattn_gemm_workspace_bytes(int M, int N, int K, int batch);
triattn_status triattn_gemm(int ta, int tb, int M, int N, int K, const void* A, long long lda, const void* B,
                            long long ldb, void* C, long long ldc, int c_f32, int batch, long long sA, long long sB,
                            long long sC, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Synchronises `stream`, then reads and clears the device status word that
 * kernels set when a bounded wait gives up.  Returns TRIATTN_OK,
 * TRIATTN_ERR_TIMEOUT, or TRIATTN_ERR_CUDA if the synchronisation failed.
 */
triattn_status triattn_device_status(void* stream);

/*
 * Test hook, off by default: when `cap_ns` > 0 every bounded device wait of
 * later launches gives up after `cap_ns` nanoseconds instead of the default
 * limit (about 2 s).  0 restores the default.
 */
void triattn_set_wait_limit_ns(unsigned long long cap_ns);

/*
 * Kernel tracing.  triattn_trace_enable(1) clears earlier records and makes
 * every later kernel launch of the library record a pair of CUDA events on
 * its launch stream (on = 0 stops recording; records are kept).
 * triattn_trace_read() synchronises the recorded events and writes one entry
 * per kernel kind that launched (at most `max_entries`), returning the
 * number written, or -1 if an event query failed.  Kernel names are static
 * strings.  Recording costs one cudaEventRecord before and after each launch.
 */
typedef struct {
  const char* kernel;
  int launches;
  double total_ms;
  double min_ms;
  double max_ms;
} triattn_trace_entry;

void triattn_trace_enable(int on);
int triattn_trace_read(triattn_trace_entry* out, int max_entries);

/*
 * Test hook, off by default.  While `on` is nonzero, the forward kernel's
 * producer warp skips its first K-tile load, so nothing ever completes the
 * barrier the MMA warp waits on: the bounded wait runs out, the kernel
 * records TRIATTN_ERR_TIMEOUT in the device status word and every CTA
 * returns.  Used only to test timeout reporting (with a short limit set by
 * triattn_set_wait_limit_ns); outputs of such a call are undefined.
 */
void triattn_test_set_starve(int on);

#ifdef __cplusplus
}
#endif

#endif /* TRIATTN_H_ */
