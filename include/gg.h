/*
 * gg.h -- C ABI of the GB300 (sm_103a) Mixture-of-Experts grouped GEMM library.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - T = num_tokens, topk = experts per token, R = T * topk routed rows,
 *    E = experts.  A "flat slot" f = t * topk + j names slot j of token t.
 *    An "expert-order row" i lies in [offsets[e], offsets[e+1]) for its expert.
 *  - bf16 tensors are passed as `gg_bf16*` (raw IEEE bfloat16 bits), row-major,
 *    rows contiguous.  Weights W are (E, N, K) with K contiguous.
 *  - Every pointer argument is a DEVICE pointer owned by the caller, unless it
 *    is documented otherwise.  The library allocates no device memory.
 *  - Calls are asynchronous on `stream` (a cudaStream_t passed as void*; NULL
 *    = the legacy default stream).  Inputs must stay valid until the stream
 *    reaches the call.
 *  - Return value: GG_OK (0), or a negative GG_ERR_* code for an error found
 *    synchronously on the host (bad arguments, unsupported shape, launch
 *    failure).  Nothing is launched when an error is returned.
 *  - `status` (optional, may be NULL): a device int32 the kernels set, with an
 *    atomic compare-and-swap from 0, to a GG_DEV_* code when they find bad
 *    input data (an expert id out of range, a row index out of range) or a
 *    bounded wait ran out.  The offending access is skipped, never performed.
 *    The caller zeroes it and reads it after synchronising, or lets
 *    gg_read_status do both (it maps the word to GG_ERR_DEVICE_CHECK or
 *    GG_ERR_TIMEOUT).
 *  - `workspace` (the entry points that take one): caller-owned device
 *    scratch of at least gg_workspace_size() bytes for that call, 16-byte
 *    aligned; no initialisation needed, contents garbage afterwards.  Too
 *    small -> GG_ERR_WORKSPACE with nothing launched.
 *  - Size rules (else GG_ERR_UNSUPPORTED): row widths K and N multiples of 8
 *    (16-byte rows), every tensor pointer 16-byte aligned, E <= GG_MAX_EXPERTS,
 *    topk <= GG_MAX_TOPK, R < 2^31.
 *  - An empty problem (no rows or no output columns) returns GG_OK without a
 *    launch; an empty reduction writes zeros, and then the inputs that have
 *    no elements (the reduced-over operands) may be NULL.
 *
 * Sources cited below (page title, then section):
 *  [U] unslothai--unsloth unsloth/kernels/moe/grouped_gemm/interface.py
 *  [V] vllm third_party/triton_kernels/matmul_ogs.py
 *  [W] VLA/wall_x/fusions/backend.py
 */
#ifndef GG_H
#define GG_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t gg_bf16;

/* host-side return codes */
#define GG_OK 0
#define GG_ERR_INVALID_ARG (-1)
#define GG_ERR_UNSUPPORTED (-2)
#define GG_ERR_CUDA (-3)
#define GG_ERR_DEVICE_CHECK (-4) /* from gg_read_status: a kernel found bad input data */
#define GG_ERR_TIMEOUT (-5)      /* from gg_read_status: a bounded wait in a kernel ran out */
#define GG_ERR_WORKSPACE (-6)

/* device status word codes */
#define GG_DEV_OK 0
#define GG_DEV_BAD_EXPERT_ID 1
#define GG_DEV_BAD_ROW_INDEX 2
#define GG_DEV_SIZES_MISMATCH 3
#define GG_DEV_TIMEOUT 4

#define GG_MAX_EXPERTS 2048
#define GG_MAX_TOPK 64
#define GG_ROUTE_NOALLOC_SCRATCH_BYTES (1u << 20)
/* gg_forward_combine without a workspace (bf16 accumulation) takes topk up to this */
#define GG_COMBINE_BF16_MAX_TOPK 16

/* operations for gg_workspace_size */
#define GG_OP_ROUTE 1            /* gg_route_hist_offsets */
#define GG_OP_BACKWARD_DW 2      /* gg_backward_dW with a gathered operand */
#define GG_OP_FORWARD_COMBINE 3  /* gg_forward_combine, fp32 accumulation */
/* flags for gg_workspace_size */
#define GG_PERMUTE_X 1
#define GG_PERMUTE_Y 2

/* Human-readable text for a GG_* return code (static storage). */
const char* gg_status_string(int code);
/* Human-readable text for a GG_DEV_* device status code (static storage). */
const char* gg_device_status_string(int code);
/* Text of the last CUDA error seen by a host call on this thread. */
const char* gg_last_cuda_error(void);

/* Bytes of workspace an entry point needs for this problem (0: it takes none,
 * or needs none for these flags).  Same size arguments as the call (for a
 * call without N or K pass 0); flags: GG_PERMUTE_X | GG_PERMUTE_Y as the
 * call's permute flags.  No counterpart on the pages: the library allocates
 * nothing, so every scratch buffer comes from the caller through this size. */
size_t gg_workspace_size(int op, int64_t T, int topk, int E, int64_t N, int64_t K, int flags);

/* Synchronises `stream`, reads the device status word `status` (device int32)
 * and returns GG_OK when it is GG_DEV_OK, GG_ERR_TIMEOUT for GG_DEV_TIMEOUT,
 * GG_ERR_DEVICE_CHECK for any other device code, GG_ERR_CUDA if the read
 * fails.  *code (host int32, may be NULL) receives the GG_DEV_* code.  The
 * word is left as it is.  No counterpart on the pages. */
int gg_read_status(const int32_t* status, int32_t* code, void* stream);

/* Tile schedule of the grouped-GEMM launches (process-wide; returns the
 * previous mode, or GG_ERR_INVALID_ARG for an unknown one).
 *   GG_SCHEDULE_AUTO (default): 2-CTA launches over experts whose tiles are
 *     long (at least 48 reduction blocks of 64 a tile; dW: a mean expert of
 *     at least 32 blocks) hand tiles out dynamically, from a device counter
 *     in tile order, so the pairs that read one operand tile read it at about
 *     the same time and DRAM sees it once; shorter tiles keep the static
 *     round-robin (pair p takes tiles p, p + P, ...).
 *   GG_SCHEDULE_STATIC, GG_SCHEDULE_DYNAMIC: always that schedule (dynamic
 *     only where the launch supports it; the dual GEMM is always static).
 * Results are identical bit for bit under either schedule: a tile's sums
 * do not depend on which pair computes it.  The dynamic schedule uses one of
 * 1024 device counter pairs per launch, in turn, reset by the launch itself
 * as it ends: more than 1023 dynamic launches in flight at once on one
 * device (streams that run concurrently, or replays of one captured graph
 * running concurrently with themselves) is not supported.  Launches of more
 * than 2^30 tiles keep the static schedule.  No counterpart on the pages. */
#define GG_SCHEDULE_AUTO 0
#define GG_SCHEDULE_STATIC 1
#define GG_SCHEDULE_DYNAMIC 2
int gg_set_gemm_schedule(int mode);

/* Diagnostic: runs, in one CTA, the bounded mbarrier wait that every
 * pipelined kernel of this library uses, on a barrier phase nothing ever
 * completes, with a limit of limit_ns (0 < limit_ns <= 2 s).  The wait gives
 * up, sets *status to GG_DEV_TIMEOUT (if it was 0) and writes *result = 0
 * (1 would mean the phase completed).  status and result are device int32s.
 * Lets a caller check that a stuck wait ends with an error status instead of
 * a hang, leaving the context usable.  No counterpart on the pages. */
int gg_selftest_bounded_wait(int32_t* status, int32_t* result, uint64_t limit_ns, void* stream);

/* ------------------------------------------------------------------ route --
 * Routing metadata from the router's choices ([U] grouped_gemm_forward
 * docstring: m_sizes = tokens per expert, gather_indices sliced by
 * cumsum(m_sizes) gives each expert's token slots; [V] RoutingData.expt_hist,
 * GatherIndx / ScatterIndx; [V] ragged-dw comment for the padded layout;
 * [W] permute).
 *
 *  topk_ids       [T, topk] int32 expert id of each slot (must be in [0, E)).
 *  pad_block      > 0: also write padded_offsets; <= 0: padded_offsets unused.
 *  m_sizes        [E]   out: rows per expert.
 *  offsets        [E+1] out: exclusive prefix of m_sizes, offsets[E] = R.
 *  padded_offsets [E+1] out (or NULL): prefix of ceil(m_e/pad_block)*pad_block.
 *  gather_idx     [R]   out: flat slot f held by expert-order row i; within an
 *                       expert, slots ascend (stable order).
 *  row_id_map     [R]   out (or NULL): inverse, row_id_map[gather_idx[i]] = i.
 *  workspace      device scratch of at least gg_route_workspace_size() bytes,
 *                 owned by the caller; contents need no initialisation and are
 *                 garbage afterwards.  Too small -> GG_ERR_WORKSPACE.
 * An id outside [0, E) sets GG_DEV_BAD_EXPERT_ID; that slot is not counted and
 * gets no row (the outputs are then incomplete). */
size_t gg_route_workspace_size(int64_t T, int topk, int E);
int gg_route_hist_offsets(const int32_t* topk_ids, int64_t T, int topk, int E, int pad_block,
                          int32_t* m_sizes, int32_t* offsets, int32_t* padded_offsets,
                          int32_t* gather_idx, int32_t* row_id_map, void* workspace,
                          size_t workspace_bytes, int32_t* status, void* stream);

/* ------------------------------------------------ route, allocation-free --
 * No counterpart on the pages.  Same outputs as gg_route_hist_offsets, for
 * callers that cannot allocate device memory or pass a workspace: a runtime
 * that owns all device memory in its own arena and hands this code only its
 * input and output buffers, or a latency-critical path that must not pay for
 * an allocation.  There is no workspace argument: the counting sort's scratch
 * is a static device array of GG_ROUTE_NOALLOC_SCRATCH_BYTES (1 MiB) that
 * every GPU loading the library holds until the process exits.
 *  - The first call on each device looks up that array's device address
 *    (once per device, with that device current); make that first call
 *    before any stream capture.
 *  - Each device holds its own copy of the array, shared by every call on
 *    that device: calls that overlap on the same device (concurrent streams)
 *    race on it, so the caller must serialise them; calls on different
 *    devices do not interfere.  No state carries over between calls.
 *  - A problem whose scratch, ceil(T*topk/256) * E * 4 bytes, exceeds the
 *    array returns GG_ERR_WORKSPACE without launching.  A device numbered 64
 *    or higher returns GG_ERR_UNSUPPORTED.
 * Allocates nothing. */
int gg_route_hist_offsets_noalloc(const int32_t* topk_ids, int64_t T, int topk, int E,
                                  int pad_block, int32_t* m_sizes, int32_t* offsets,
                                  int32_t* padded_offsets, int32_t* gather_idx,
                                  int32_t* row_id_map, int32_t* status, void* stream);

/* ---------------------------------------------------------------- permute --
 * Token rows into expert order ([W] permute; [U] permute_x): for every slot f
 * of token t, Xp[row_id_map[f], :] = X[t, :].  Equivalently
 * Xp[i, :] = X[gather_idx[i] / topk, :].  Bit-exact copy.
 *  X [T, K] bf16, row_id_map [R] int32 (from gg_route_hist_offsets),
 *  Xp [R, K] bf16 out.  A map entry outside [0, R) sets GG_DEV_BAD_ROW_INDEX. */
int gg_permute(const gg_bf16* X, const int32_t* row_id_map, int64_t T, int topk, int64_t K,
               gg_bf16* Xp, int32_t* status, void* stream);

/* ------------------------------------------------------ unpermute-combine --
 * Expert outputs back to token order, weighted combine over a token's slots
 * ([W] unpermute: combine with routing probabilities; [V] matmul_ogs_torch:
 * accumulate every slot of a token in fp32):
 *   out[t, :] = bf16( sum_{j<topk} w[t*topk+j] * Y[row(t*topk+j), :] )
 * summed in fp32 in j order.
 *  Y [R, N] bf16; row_id_map [R] int32, or NULL when Y is already in
 *  token-slot order (row(f) = f, e.g. after a forward with permute_y);
 *  topk_w [T, topk] fp32, or NULL for unit weights; out [T, N] bf16.
 * With row_id_map = NULL and topk_w = NULL this is the top-k sum of a
 * token-slot-ordered tensor ([U] GroupedGemm.backward, the sum over topk). */
int gg_unpermute_combine(const gg_bf16* Y, const int32_t* row_id_map, const float* topk_w,
                         int64_t T, int topk, int64_t N, gg_bf16* out, int32_t* status,
                         void* stream);

/* ----------------------------------------------- unpermute-combine, bwd --
 * Gradient of gg_unpermute_combine ([W] unpermute_bwd: gradients of the
 * unpermute forward, taking the forward's input for the probabilities'
 * gradient; no probabilities means unit weights).  With G = dL/d out:
 *   dY[row(f), :] = bf16( w[f] * G[t, :] )            for every slot f = t*topk + j
 *   dw[f]         = sum_n G[t, n] * Y[row(f), n]      (fp32)
 *  G [T, N] bf16; Y [R, N] bf16, the forward's input (needed only for dw);
 *  row_id_map [R] int32 or NULL (identity); topk_w [T, topk] fp32 or NULL (1);
 *  dY [R, N] bf16 out (every row written once); dw [T, topk] fp32 out or NULL.
 *  dw without Y -> GG_ERR_INVALID_ARG.  Deterministic (fixed reduction order).
 *  A map entry outside [0, R) sets GG_DEV_BAD_ROW_INDEX; that slot gets dw 0. */
int gg_unpermute_combine_bwd(const gg_bf16* G, const gg_bf16* Y, const int32_t* row_id_map,
                             const float* topk_w, int64_t T, int topk, int64_t N, gg_bf16* dY,
                             float* dw, int32_t* status, void* stream);

/* ---------------------------------------------------------------- forward --
 * Grouped GEMM forward ([U] grouped_gemm_forward; [V] matmul_ogs docstring:
 * Y[idx_y(e)] = X[idx_x(e)] @ W[e]^T):
 *   for every expert-order row i of expert e:
 *     a   = X[gather_idx[i] / topk]  if permute_x  (X is [T, K])
 *           X[i]                      otherwise    (X is [R, K], expert order)
 *     y   = a @ W[e]^T                (fp32 accumulate)
 *     y  *= topk_w[gather_idx[i]]     if fuse_mul_post (needs permute_y)
 *     Y[gather_idx[i]] = bf16(y)      if permute_y (token-slot order)
 *     Y[i]             = bf16(y)      otherwise
 *  W [E, N, K] bf16; m_sizes [E] int32 with sum R; gather_idx [R] (needed when
 *  a permute flag is set); topk_w [T, topk] fp32 (needed for fuse_mul_post);
 *  Y [R, N] bf16 out.  permute_x and permute_y may be combined (gather on
 *  load and scatter on store in one pass). */
int gg_forward(const gg_bf16* X, const gg_bf16* W, const int32_t* m_sizes,
               const int32_t* gather_idx, const float* topk_w, int64_t T, int topk, int E,
               int64_t N, int64_t K, int permute_x, int permute_y, int fuse_mul_post,
               gg_bf16* Y, int32_t* status, void* stream);

/* ---------------------------------------------- forward + fused combine --
 * The forward grouped GEMM with the weighted top-k combine of
 * gg_unpermute_combine fused into its epilogue as atomic adds ([V] the
 * scatter path: with several active experts per token each token row is a
 * sum over its slots; the output starts zeroed):
 *   out[t] = sum over the slots f = t*topk + j of  w[f] * (a_f @ W[e(f)]^T)
 *   a_f, W[e] as gg_forward (permute_x selects X [T, K] with the gather, else
 *   X [R, K] in expert order); w = topk_w [T, topk] fp32, or 1 when NULL.
 *  out [T, N] bf16 out.  Two accumulations:
 *   - with a workspace of gg_workspace_size(GG_OP_FORWARD_COMBINE, T, topk,
 *     E, N, K, 0) bytes (T*N fp32): the call zeroes it, every slot's scaled
 *     fp32 row is added there with fp32 atomic adds, and one pass rounds the
 *     sums to bf16 into out (any topk);
 *   - workspace NULL: out is zeroed and every slot's row, rounded to bf16, is
 *     added with bf16 atomic adds (each add rounds); topk above
 *     GG_COMBINE_BF16_MAX_TOPK returns GG_ERR_WORKSPACE, since the summed
 *     roundings of more slots approach the 1e-2 relative error bound.
 *  NOT deterministic: the order of a token's topk adds depends on scheduling,
 *  so the last bits can differ from run to run; gg_forward with permute_y and
 *  gg_unpermute_combine give the deterministic result (one fp32 sum, rounded
 *  once).  The per-slot rows are not stored, so training that needs them
 *  (the routing-weight gradient of gg_unpermute_combine_bwd) uses that path. */
int gg_forward_combine(const gg_bf16* X, const gg_bf16* W, const int32_t* m_sizes,
                       const int32_t* gather_idx, const float* topk_w, int64_t T, int topk, int E,
                       int64_t N, int64_t K, int permute_x, gg_bf16* out, void* workspace,
                       size_t workspace_bytes, int32_t* status, void* stream);

/* ------------------------------------------------------ forward + SwiGLU --
 * The forward grouped GEMM with the gated activation fused into its epilogue
 * ([V] FusedActivation with reduction_n = 2: each pair of adjacent output
 * columns reduces to one).  Output columns are interleaved gate/up:
 *   y   = as gg_forward (no scatter, no scale)          [R, N]
 *   A[i, c] = bf16( silu(y[2c]) * y[2c+1] )             [R, N/2], from the fp32 y
 *   silu(g) = g / (1 + exp(-g))
 *  Y [R, N] bf16 out, or NULL to store only the activation (inference);
 *  training keeps Y for gg_swiglu_bwd.  N must be a multiple of 16. */
int gg_forward_swiglu(const gg_bf16* X, const gg_bf16* W, const int32_t* m_sizes,
                      const int32_t* gather_idx, int64_t T, int topk, int E, int64_t N, int64_t K,
                      int permute_x, gg_bf16* Y, gg_bf16* A, int32_t* status, void* stream);

/* Gradient of that activation: from the stored H = y [rows, 2I] and
 * dA = dL/dA [rows, I] (bf16), with s = 1 / (1 + exp(-g)):
 *   dH[r, 2c]   = dA * u * s * (1 + g * (1 - s))      (gate)
 *   dH[r, 2c+1] = dA * g * s                            (up)
 * dH [rows, 2I] bf16 out.  I must be a multiple of 8. */
int gg_swiglu_bwd(const gg_bf16* H, const gg_bf16* dA, int64_t rows, int64_t I, gg_bf16* dH,
                  void* stream);

/* ------------------------------------------------------------ backward dX --
 * Gradient of the forward's input ([U] grouped_gemm_dX; GroupedGemm.backward):
 *   for every expert-order row i of expert e:
 *     g  = dY[gather_idx[i]] if permute_y else dY[i]     (dY is [R, N])
 *     dx = g @ W[e]                                      (reduce over N)
 *     dX[gather_idx[i]] = bf16(dx) if permute_x (token-slot order) else dX[i]
 *  dX [R, K] bf16 out.  dX_tok [T, K] bf16 out or NULL: with permute_x, the
 *  per-token sum over its topk slots of the stored bf16 dX rows (fp32 sum in
 *  slot order).  dX_tok without permute_x -> GG_ERR_INVALID_ARG.  The flags
 *  are those of the forward call being differentiated. */
int gg_backward_dX(const gg_bf16* dY, const gg_bf16* W, const int32_t* m_sizes,
                   const int32_t* gather_idx, int64_t T, int topk, int E, int64_t N, int64_t K,
                   int permute_x, int permute_y, gg_bf16* dX, gg_bf16* dX_tok, int32_t* status,
                   void* stream);

/* ---------------------------------------------- backward dX + SwiGLU bwd --
 * The backward dX of a grouped GEMM whose input was the SwiGLU activation of
 * gg_forward_swiglu, with the activation's backward fused into the epilogue
 * (the two steps of gg_backward_dX and gg_swiglu_bwd in one pass; the
 * activation gradient never goes to memory and is not rounded to bf16):
 *   for every expert-order row i of expert e:
 *     da = dY[i] @ W[e]                                  (fp32, [K])
 *     g = H[i, 2c], u = H[i, 2c+1], s = 1 / (1 + exp(-g))
 *     dH[i, 2c]   = bf16( da[c] * u * s * (1 + g * (1 - s)) )
 *     dH[i, 2c+1] = bf16( da[c] * g * s )
 *  dY [R, N] bf16 in expert order (gg_permute a token-slot-order gradient
 *  first); W [E, N, K]; H [R, 2K] bf16, the stored forward output of
 *  gg_forward_swiglu (expert order); dH [R, 2K] bf16 out. */
int gg_backward_dX_swiglu(const gg_bf16* dY, const gg_bf16* W, const int32_t* m_sizes, int64_t T,
                          int topk, int E, int64_t N, int64_t K, const gg_bf16* H, gg_bf16* dH,
                          int32_t* status, void* stream);

/* ------------------------------------------------------------ backward dW --
 * Gradient of the expert weights ([U] grouped_gemm_dW; [V] ragged-dw comment:
 * the reduction dimension is each expert's own rows):
 *   dW[e] = sum over expert-order rows i of e of  outer(g_i, a_i)   -> (N, K)
 *     a_i = X[gather_idx[i] / topk] if permute_x else X[i]
 *     g_i = dY[gather_idx[i]]       if permute_y else dY[i]
 *  fp32 accumulate, bf16 out; an expert with no rows gets dW[e] = 0.
 *  X [T, K] if permute_x else [R, K]; dY [R, N]; dW [E, N, K] bf16 out.
 *  workspace (may be NULL): with a permute flag and at least
 *  gg_workspace_size(GG_OP_BACKWARD_DW, T, topk, E, N, K, flags) bytes, the
 *  gathered operands are first copied into expert order there (X rows
 *  R*K*2 bytes, dY rows R*N*2 bytes) and the reduction reads dense tiles;
 *  with NULL the row gathers are fused into the reduction's operand loads,
 *  which is 2.5-4x slower on sm_103a (each reduction block needs 64 newly
 *  gathered rows, fetched in 16-byte pieces).  Both give the same products. */
int gg_backward_dW(const gg_bf16* X, const gg_bf16* dY, const int32_t* m_sizes,
                   const int32_t* gather_idx, int64_t T, int topk, int E, int64_t N, int64_t K,
                   int permute_x, int permute_y, gg_bf16* dW, void* workspace,
                   size_t workspace_bytes, int32_t* status, void* stream);

/* --------------------------------------------------------- dual asymmetric --
 * Two experts' GEMMs with different row counts and output widths in one
 * launch ([W] asym_dual_gmm_separated):  Y0 = op(X0) @ op(W0),
 * Y1 = op(X1) @ op(W1), shared reduction length k.
 *  trans_a = 0: X0 [m0, k], X1 [m1, k];  trans_a = 1: X0 [k, m0], X1 [k, m1].
 *  trans_b = 0: W0 [k, n0], W1 [k, n1];  trans_b = 1: W0 [n0, k], W1 [n1, k].
 *  Y0 [m0, n0], Y1 [m1, n1] bf16 out, fp32 accumulate.
 *  m0, m1, n0, n1 and k must be multiples of 8 (16-byte rows either way). */
int gg_dual_asym(const gg_bf16* X0, const gg_bf16* X1, const gg_bf16* W0, const gg_bf16* W1,
                 gg_bf16* Y0, gg_bf16* Y1, int64_t m0, int64_t m1, int64_t k, int64_t n0,
                 int64_t n1, int trans_a, int trans_b, int32_t* status, void* stream);

/* ------------------------------------------------------- expert parallel --
 * Rows routed to experts held by other ranks ([V] FusedComm and
 * post_matmul_comm_torch: routed rows exchanged between the ranks that hold
 * different experts).  G ranks; rank r holds experts [r*E_loc, (r+1)*E_loc),
 * E = G * E_loc <= GG_MAX_EXPERTS.  After gg_route_hist_offsets and
 * gg_permute over all E experts, rank r's rows for rank d's experts are the
 * contiguous block d of its expert-order rows.  The caller exchanges, with
 * its own collectives (e.g. NCCL all-to-all), first the counts
 * (recv_m[s][e] = rank s's m_sizes[r*E_loc + e]), then the rows: rank r
 * receives from each source s, in source order, s's rows for r's experts,
 * expert after expert.  The local GEMMs want expert-contiguous rows:
 *   received row j of block (s, e), q-th in it, becomes local row
 *   row_map[j] = local_off[e] + sum_{s'<s} recv_m[s'][e] + q,
 * local_off = exclusive prefix of local_m_sizes[e] = sum_s recv_m[s][e]; so
 * gg_permute(X_recv, row_map, topk = 1) gives them, and after the local
 * GEMMs gg_unpermute_combine(Y_loc, row_map, NULL, R_loc, 1) puts the results
 * back in received order for the return exchange.  Within an expert, rows
 * stay in (source rank, source row) order: the order of one routing of every
 * rank's tokens numbered rank after rank. */

/* Host-side plan (no GPU work; all arrays host memory).  m_sizes [G*E_loc]:
 * this rank's histogram over all experts; recv_m [G][E_loc]: received counts.
 * Out: send_counts [G] rows for each rank, recv_counts [G] rows from each
 * rank, local_m_sizes [E_loc]; row_map [R_loc] (or NULL) as above, row_map_len
 * must be R_loc = sum of recv_m.  Negative counts -> GG_ERR_INVALID_ARG. */
int gg_ep_plan(const int32_t* m_sizes, const int32_t* recv_m, int G, int E_loc, int64_t* send_counts,
               int64_t* recv_counts, int32_t* local_m_sizes, int32_t* row_map, int64_t row_map_len);

/* The same row_map computed on the device from the device copy of recv_m
 * [G][E_loc] (int32), for R_loc received rows; row_map [R_loc] int32 out.
 * R_loc not equal to the sum of recv_m (or a negative count) sets
 * GG_DEV_SIZES_MISMATCH; rows past the counted ones get -1. */
int gg_ep_recv_map(const int32_t* recv_m, int G, int E_loc, int64_t R_loc, int32_t* row_map,
                   int32_t* status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GG_H */
