/*
 * moe.h -- C ABI of the dropless Mixture-of-Experts layer hot path (GB300, sm_103a).
 *
 * The layer (per token t of x [T, d]):
 *   router   s_t    = x_t W_r (+ b)                           fp32 scores over E experts
 *   route    S_t    = the k largest s_t, descending, ties -> lower expert index
 *            w_t,j  = exp(s_t,e_j) / sum_{i in S_t} exp(s_t,e_i)   (softmax renormalised on the top-k)
 *   permute  every copy q = t*k + j goes to row dest[q] of an expert-contiguous buffer,
 *            experts in ascending order, copies of one expert in ascending q (stable)
 *   experts  Y_q    = (silu(x_t W1_e^T) * (x_t W3_e^T)) W2_e^T   SwiGLU, one grouped GEMM
 *   combine  y_t    = sum_j w_t,j Y_dest[t*k+j] + sum_s SwiGLU_s(x_t)   (shared experts, weight 1)
 *   backward dX chain and dW products computed by separate calls.
 * Sources: routing as fused softmax -> top-k -> mask and an FP32 router ("MoE operator
 * optimisation: routing hardware acceleration and zero-copy communication", sections 2.1
 * and 4.2); dropless routing (Pangu Ultra MoE tech-report article, dropless vs
 * drop-and-pad); rearrange / un-rearrange of token copies (Huawei MoE training-operator
 * article, "VectorSort", Fig. 3) with dispatch preprocessing that never waits on the device
 * (same article, sync elimination, Fig. 4); grouped matmul over experts (MindSpore
 * DeepSeek-V3 page, section 02.1); shared + routed weighted sum (Pangu Ultra MoE article,
 * contribution analysis); expert dW and dX computed separately (Pangu Ultra MoE article,
 * adaptive pipe overlap; MindSpore page, section 01.2).
 *
 * Conventions of every call:
 *  - Tensor pointers are DEVICE pointers owned by the caller, row-major, 16-byte aligned.
 *    The library allocates and frees nothing.
 *  - Calls are asynchronous on `stream` and never synchronise (except moe_get_device_error).
 *  - Calls run on the calling thread's current CUDA device. Several host threads may call the
 *    library at once (each with its own device, or its own stream and workspace): the one-time
 *    per-device setup (kernel attributes, device properties) is made under a lock.
 *  - Activations and expert weights are fp32 (MOE_F32) or bf16 (MOE_BF16) as dims->dtype says;
 *    router weights, scores, gates, dgate and score gradients are always fp32; indices int32.
 *  - Expert weights are K-major: W13 [E][2f][d] (gate rows 0..f-1, up rows f..2f-1),
 *    W2 [E][d][f]; shared experts Ws13 [S][2f_s][d], Ws2 [S][d][f_s]. Gradients share layouts.
 *  - Buffers with "routed rows" have T*k rows in the permuted (expert-contiguous) order;
 *    "shared rows" have S*T rows, shared expert s owning rows s*T .. s*T+T-1.
 *  - Return value: MOE_OK, or a negative status for an argument error detected on the host
 *    (nothing is launched then), or MOE_ERR_LAUNCH / MOE_ERR_CUDA for a CUDA error.
 *  - Errors found on the device (an expert id out of range, a bounded wait that ran out) are
 *    recorded in an error word inside the workspace; moe_get_device_error reads and clears it.
 *  - T == 0 is a valid no-op (except in the calls that return balance statistics, whose
 *    means over the tokens need T >= 1: they reject T == 0 with MOE_ERR_BAD_DIMS).
 *  - bf16 needs d, f, f_s multiples of 64; fp32 needs multiples of 8. E <= 1024, 1 <= k <= min(E, 32).
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t; /* a cudaStream_t; NULL = legacy default stream */

enum moe_status {
  MOE_OK = 0,
  MOE_ERR_NULL_POINTER = -1,        /* a required pointer is NULL */
  MOE_ERR_MISALIGNED = -2,          /* a pointer is not 16-byte aligned (workspace: 256) */
  MOE_ERR_BAD_DIMS = -3,            /* T < 0, d/f/f_s not a multiple of the dtype's unit, E out of range */
  MOE_ERR_BAD_TOPK = -4,            /* k < 1, k > E or k > 32 */
  MOE_ERR_UNSUPPORTED_DTYPE = -5,   /* dtype is neither MOE_F32 nor MOE_BF16 */
  MOE_ERR_WORKSPACE_TOO_SMALL = -6, /* ws_bytes < moe_workspace_bytes(dims) */
  MOE_ERR_LAUNCH = -7,              /* a kernel launch failed */
  MOE_ERR_CUDA = -8,                /* another CUDA runtime/driver call failed */
  MOE_ERR_UNSUPPORTED_DEVICE = -9,  /* bf16 grouped GEMM needs an sm_103 (GB300) device */
  MOE_ERR_DEVICE_EXPERT_ID = -100,  /* device: expert id outside [0, E) or repeated in a row */
  MOE_ERR_DEVICE_TIMEOUT = -101     /* device: a bounded wait ran out */
};

enum moe_dtype { MOE_F32 = 0, MOE_BF16 = 1 };

typedef struct moe_dims {
  int64_t T;     /* tokens */
  int32_t d;     /* hidden size */
  int32_t E;     /* routed experts */
  int32_t k;     /* experts per token */
  int32_t f;     /* routed expert FFN width */
  int32_t S;     /* shared experts (0 allowed) */
  int32_t f_s;   /* shared expert FFN width */
  int32_t dtype; /* enum moe_dtype */
  /* 0: dropless (every token copy is computed). C > 0: the drop-and-pad variant the pages
   * compare dropless training with (Pangu Ultra MoE tech-report article, dropless vs
   * drop-and-pad; CANN MoE page, section 4.3): every expert gets exactly C rows; the first C
   * copies of an expert in token order are kept, later ones are dropped (dest = -1, they
   * add nothing to y and pass no gradient back through the expert); unused rows are
   * zero padding. The permuted buffers (x_perm, row_src, w_perm, z, h, y_perm, dy_perm,
   * dz, dx_perm) then have R = E*C rows instead of R = T*k, and offsets[e] = e*C. */
  int32_t capacity;
  /* enum moe_rearrange (flags): how the bf16 dropless layer moves token rows between token
   * order and expert order around the expert GEMMs. MOE_REARRANGE_COPY (0, default):
   * rearranged copies in memory (x_perm, dy_perm) and an un-rearranging combine that
   * gathers each token's k expert rows from y_perm by dest. MOE_REARRANGE_GATHER (1): the
   * rearrangement is fused into the GEMMs' operand loads (row gathers from x and dy by
   * row_src). MOE_REARRANGE_SCATTER (2): moe_layer_fwd's second expert GEMM writes each
   * output row at its token-major slot t*k + j instead of its expert-order row, so the
   * combine reads every token's k rows as one contiguous block. Both together: 3. The
   * results are identical in every form. fp32 layers and the drop-and-pad variant always use
   * the copies. */
  int32_t rearrange;
} moe_dims;

enum moe_rearrange { MOE_REARRANGE_COPY = 0, MOE_REARRANGE_GATHER = 1, MOE_REARRANGE_SCATTER = 2 };

/* Human-readable text of a status code (static string). */
const char* moe_status_string(int status);

/* Bytes of device workspace every call below may use for dims (>= 256). The workspace holds
 * the device error word, small scratch (per-chunk expert histograms, gate partials) and, for
 * moe_layer_fwd/bwd, the transient intermediates of the layer. */
size_t moe_workspace_bytes(const moe_dims* dims);

/* Zero the error word and scratch headers of a fresh workspace (async). Call once after
 * allocating it. ws: device, >= moe_workspace_bytes(dims) bytes, 256-byte aligned. */
int moe_workspace_init(void* ws, size_t ws_bytes, const moe_dims* dims, moe_stream_t stream);

/* Synchronise `stream`, copy the workspace error word to *out (MOE_OK if none) and clear it. */
int moe_get_device_error(void* ws, moe_stream_t stream, int* out);

/* a0. Router scores L = x W_r, fp32 FMA accumulation (no TF32), the router kept in FP32
 * ("MoE operator optimisation ...", section 4.2).
 * x [T, d] (dims->dtype), w_r [d][E] fp32 -> logits [T][E] fp32 (written fully). */
int moe_router_logits(const void* x, const float* w_r, const moe_dims* dims, float* logits,
                      void* ws, size_t ws_bytes, moe_stream_t stream);

/* a1. Fused softmax -> top-k -> renormalised gates -> per-expert counts ("MoE operator
 * optimisation ...", section 2.1). One warp per token.
 * logits [T][E] fp32; bias [E] fp32 or NULL (added in fp32 before selection and gating);
 * -> topk_idx [T][k] int32 (descending score, ties to the lower index), topk_w [T][k] fp32,
 *    counts [E] int32 (zeroed and filled by this call). Scores must be finite. */
int moe_route_topk(const float* logits, const float* bias, int64_t T, int32_t E, int32_t k,
                   int32_t* topk_idx, float* topk_w, int32_t* counts,
                   void* ws, size_t ws_bytes, moe_stream_t stream);

/* a2. VectorSort rearrange (Huawei MoE training-operator article, "VectorSort", Fig. 3):
 * per-chunk expert histograms -> scan -> stable scatter, all on the device (no host wait,
 * same article, Fig. 4), with each row moved once in 16-byte vectors.
 * x [T, d]; topk_idx [T][k]; topk_w [T][k] fp32 or NULL ->
 *   x_perm [T*k, d] (row dest[q] = x[q / k]), dest [T*k] int32, row_src [T*k] int32,
 *   offsets [E+1] int32 (exclusive scan of the per-expert counts),
 *   w_perm [T*k] fp32 or NULL (w_perm[dest[q]] = topk_w[q]).
 * An id outside [0, E) or repeated within a row records MOE_ERR_DEVICE_EXPERT_ID; such copies
 * get dest = -1 and are not moved (nothing is written out of bounds).
 * With dims->capacity = C > 0 (drop-and-pad): x_perm, row_src and w_perm have E*C rows,
 * offsets[e] = e*C, dest = -1 for a dropped copy, and the padding rows hold zeros
 * (row_src = -1, w_perm = 0). */
int moe_permute(const void* x, const int32_t* topk_idx, const float* topk_w, const moe_dims* dims,
                void* x_perm, int32_t* dest, int32_t* row_src, int32_t* offsets, float* w_perm,
                void* ws, size_t ws_bytes, moe_stream_t stream);

/* a2 without a workspace, for callers that cannot allocate device memory (an allocator-free
 * runtime, a memory pool that must not grow, a process limited to the buffers it was given).
 * The pages have no counterpart of this call. Same outputs and results as moe_permute for the
 * dropless permutation (dims->capacity must be 0; f, S and f_s are not read), with the same
 * row-width rule (d a multiple of 64 for bf16, of 8 for fp32); the permutation's scratch lives
 * in one static device array of the library (about 1.5 MB, held by every GPU that loads the
 * library until the process exits) instead of a workspace.
 * Limits: T*k <= 262144 and E * ceil(T/64) <= 65536, else MOE_ERR_WORKSPACE_TOO_SMALL (nothing
 * launched). dev_err: optional 4-byte-aligned device int (else MOE_ERR_MISALIGNED) that
 * receives MOE_ERR_DEVICE_EXPERT_ID for invalid ids (first error wins; the caller zeroes it),
 * or NULL. The first call on a device looks up the
 * array's address for that device; make it before any stream capture. Every call shares the
 * array: calls that overlap on the GPU race, so order them on one stream. */
int moe_permute_noalloc(const void* x, const int32_t* topk_idx, const float* topk_w,
                        const moe_dims* dims, void* x_perm, int32_t* dest, int32_t* row_src,
                        int32_t* offsets, float* w_perm, int* dev_err, moe_stream_t stream);

/* a2 (gather-only mode, used for dY in the backward): x_perm[dest[q]] = x[q / k] for a dest
 * from moe_permute. x [T, d] -> x_perm [T*k, d]. Copies with dest < 0 are skipped. */
int moe_permute_rows(const void* x, const int32_t* dest, const moe_dims* dims, void* x_perm,
                     moe_stream_t stream);

/* a3. Grouped SwiGLU forward over the ragged expert segments (one persistent tcgen05/TMEM
 * grouped GEMM launch per matmul for bf16; a SIMT fp32-FMA kernel for fp32); tile schedules
 * are built on the device from `offsets`.
 * x_perm [T*k, d], x [T, d] (shared experts' input), w13, w2, ws13, ws2 (NULL if S == 0),
 * offsets [E+1] ->
 *   z [T*k, 2f], h [T*k, f] (routed rows), z_sh [S*T, 2f_s], h_sh [S*T, f_s] (shared rows),
 *   y_perm [T*k, d] (routed expert outputs, ungated), y_sh [T, d] (sum of the shared experts).
 * Outputs are rounded once to dims->dtype; accumulation is fp32. */
int moe_grouped_swiglu_fwd(const void* x_perm, const void* x, const void* w13, const void* w2,
                           const void* ws13, const void* ws2, const int32_t* offsets,
                           const moe_dims* dims, void* z, void* h, void* z_sh, void* h_sh,
                           void* y_perm, void* y_sh, void* ws, size_t ws_bytes, moe_stream_t stream);

/* a4. VectorSort un-rearrange fused with the gate weighting and the shared-expert add
 * (Huawei MoE training-operator article, Fig. 3; Pangu Ultra MoE article, weighted sum):
 *   y_t = sum_{j=0..k-1} topk_w[t,j] * y_perm[dest[t*k+j]] + y_sh[t]
 * summed in fp32 in that order and rounded once. topk_w NULL = weight 1; y_sh may be NULL.
 * y_perm [T*k, d], dest [T*k] -> y [T, d]. dest NULL: y_perm is already in token-major
 * order (row t*k + j holds copy j of token t, as moe_layer_fwd's second expert GEMM writes
 * it under MOE_REARRANGE_SCATTER); a dropped copy (drop-and-pad) needs dest. */
int moe_unpermute_combine(const void* y_perm, const int32_t* dest, const float* topk_w,
                          const void* y_sh, const moe_dims* dims, void* y, moe_stream_t stream);

/* a5 (expert dX chain; Pangu Ultra MoE article: dW and dX computed separately).
 *   D = dY_perm W2_e;  dgate_q = sum_f D*h (h recomputed from z);
 *   dz = [w*D*b*silu'(a) | w*D*silu(a)];  hw = w*h;  dx_perm = dz W13_e.
 * Shared experts: the same with w = 1 over all T rows, their dX summed into dx_sh.
 * dy_perm [T*k, d] (moe_permute_rows of dY), dy [T, d], z [T*k, 2f], z_sh [S*T, 2f_s],
 * w13, w2, ws13, ws2, w_perm [T*k], offsets [E+1], dest [T*k] ->
 *   dz [T*k, 2f], dz_sh [S*T, 2f_s], hw [T*k, f], hw_sh [S*T, f_s], dx_perm [T*k, d],
 *   dx_sh [T, d], dgate [T][k] fp32 (token order). */
int moe_grouped_bwd_dx(const void* dy_perm, const void* dy, const void* z, const void* z_sh,
                       const void* w13, const void* w2, const void* ws13, const void* ws2,
                       const float* w_perm, const int32_t* offsets, const int32_t* dest,
                       const moe_dims* dims, void* dz, void* dz_sh, void* hw, void* hw_sh,
                       void* dx_perm, void* dx_sh, float* dgate,
                       void* ws, size_t ws_bytes, moe_stream_t stream);

/* a6 (expert dW products, separate from the dX chain):
 *   dW2_e = dY_perm_e^T hw_e  ([d][f]),  dW13_e = dz_e^T x_perm_e  ([2f][d]),
 * reduction over the ragged segment rows; an expert with no rows gets zeros.
 * Shared: dWs2_s = dY^T hw_sh_s, dWs13_s = dz_sh_s^T x. */
int moe_grouped_bwd_dw(const void* x_perm, const void* x, const void* hw, const void* hw_sh,
                       const void* dz, const void* dz_sh, const void* dy_perm, const void* dy,
                       const int32_t* offsets, const moe_dims* dims,
                       void* dw13, void* dw2, void* dws13, void* dws2,
                       void* ws, size_t ws_bytes, moe_stream_t stream);

/* Router backward of the renormalised softmax on the top-k:
 *   dlogits[t, e_j] = w_j (dgate_j - sum_i w_i dgate_i), 0 for experts outside the top-k.
 * topk_idx, topk_w, dgate [T][k] -> dlogits [T][E] fp32 (written fully). */
int moe_route_topk_bwd(const int32_t* topk_idx, const float* topk_w, const float* dgate,
                       int64_t T, int32_t E, int32_t k, float* dlogits, moe_stream_t stream);

/* Load-balance statistics (Pangu Ultra MoE tech-report article, load-balancing section:
 * sequence-level, global-batch and EP-group balance losses; MoE operator optimisation page,
 * section 4.3: a load term added to the loss). The pages give no formula; the reading taken is
 * the usual auxiliary loss over one micro-batch (a sequence of T tokens):
 *   P_e = (1/T) sum_t softmax(s_t)_e      (full softmax of the scores s = logits + bias)
 *   f_e = counts_e / (T k)                 (share of the token copies routed to e)
 *   L_aux = alpha * E * sum_e f_e P_e
 * logits [T][E] fp32, bias [E] or NULL, counts [E] int32 (from moe_route_topk) ->
 * prob_mean [E] fp32 (or NULL), aux_loss [1] fp32 (device). Fixed-order reductions
 * (deterministic). ws: >= 256 + 4*(E*min(512, ceil(T/8)) + ceil(E/32)) bytes, 256-byte aligned. T >= 1. */
int moe_route_balance(const float* logits, const float* bias, const int32_t* counts, int64_t T,
                      int32_t E, int32_t k, float alpha, float* prob_mean, float* aux_loss, void* ws,
                      size_t ws_bytes, moe_stream_t stream);

/* moe_route_topk and moe_route_balance in one pass over the scores (the balance statistics
 * fused into the routing kernel: the Pangu Ultra MoE tech-report article's load-balancing
 * section computes them from the same router scores). Each warp takes the full softmax of its
 * token's scores from the registers the top-k reads, so the scores are read once.
 * logits [T][E] fp32, bias [E] fp32 or NULL -> topk_idx [T][k], topk_w [T][k], counts [E]
 * (zeroed and filled), prob_mean [E] (or NULL), aux_loss [1]: the same bits as moe_route_topk
 * followed by moe_route_balance with the same alpha. T >= 1; ws as for moe_route_balance
 * (>= 256 + 4*(E*min(512, ceil(T/8)) + ceil(E/32)) bytes, 256-byte aligned). */
int moe_route_topk_balance(const float* logits, const float* bias, int64_t T, int32_t E, int32_t k,
                           float alpha, int32_t* topk_idx, float* topk_w, int32_t* counts, float* prob_mean,
                           float* aux_loss, void* ws, size_t ws_bytes, moe_stream_t stream);

/* Gradient of grad * L_aux w.r.t. the scores, ADDED into dlogits [T][E] (counts constant):
 *   dlogits[t,e] += grad * alpha * E / (T*T*k) * p_te * (counts_e - sum_e' counts_e' p_te'). */
int moe_route_balance_bwd(const float* logits, const float* bias, const int32_t* counts, int64_t T,
                          int32_t E, int32_t k, float alpha, float grad, float* dlogits,
                          moe_stream_t stream);

/* Sequence-level form of the balance statistics (same pages): the T tokens fall into
 * G = T / group_len groups of consecutive tokens (one sequence each; T % group_len == 0,
 * G <= 65535), each with its own term, and the loss is their mean:
 *   P_ge = (1/group_len) sum_{t in g} softmax(s_t)_e,   f_ge = counts_ge / (group_len k)
 *   L_aux = alpha * E / G * sum_g sum_e f_ge P_ge
 * group_len = T is the micro-batch form above. topk_idx [T][k] -> counts [G][E] int32 (each
 * group's top-k choices), prob_mean [G][E] fp32 (or NULL), aux_loss [1] fp32. For the
 * global-batch (data-parallel group) and expert-parallel-group forms the caller sums counts
 * (and averages prob_mean) over the ranks of the group and passes the summed counts to the
 * backward with group_len = the group's token count and n_groups = 1.
 * ws: >= 256 + 4*G*(E*min(32, ceil(group_len/64)) + 1) bytes, 256-byte aligned. */
int moe_route_balance_seq(const float* logits, const float* bias, const int32_t* topk_idx, int64_t T,
                          int32_t E, int32_t k, int64_t group_len, float alpha, float* prob_mean,
                          int32_t* counts, float* aux_loss, void* ws, size_t ws_bytes,
                          moe_stream_t stream);

/* Gradient of grad * L_aux (sequence-level form) w.r.t. the scores, ADDED into dlogits:
 *   dlogits[t,e] += grad * alpha * E / (n_groups * group_len^2 * k) * p_te *
 *                   (c_ge - sum_e' c_ge' p_te'),   g = t / group_len,
 * counts c [ceil(T/group_len)][E] (constants of the gradient). */
int moe_route_balance_seq_bwd(const float* logits, const float* bias, const int32_t* counts, int64_t T,
                              int32_t E, int32_t k, int64_t group_len, int64_t n_groups, float alpha,
                              float grad, float* dlogits, moe_stream_t stream);

/* ---------------------------------------------------------------- whole layer */
typedef struct moe_layer_params {
  const float* w_r;  /* [d][E] fp32, or NULL when the caller passes logits_in */
  const float* bias; /* [E] fp32 constant score bias, or NULL */
  const void* w13;   /* [E][2f][d] */
  const void* w2;    /* [E][d][f] */
  const void* ws13;  /* [S][2f_s][d] or NULL */
  const void* ws2;   /* [S][d][f_s] or NULL */
} moe_layer_params;

typedef struct moe_layer_saved { /* caller-allocated; written by moe_layer_fwd, read by _bwd */
  float* logits;     /* [T][E]: x W_r (without bias); unused when logits_in is given */
  int32_t* topk_idx; /* [T][k] */
  float* topk_w;     /* [T][k] */
  int32_t* counts;   /* [E] */
  int32_t* offsets;  /* [E+1] */
  int32_t* dest;     /* [T*k] */
  int32_t* row_src;  /* [T*k] */
  float* w_perm;     /* [T*k] */
  void* x_perm;      /* [T*k, d], or NULL: not kept (see below) */
  void* z;           /* [T*k, 2f] */
  void* h;           /* [T*k, f], or NULL: not kept (the backward recomputes h from z) */
  void* z_sh;        /* [S*T, 2f_s] or NULL when S == 0 */
  void* h_sh;        /* [S*T, f_s], or NULL (not kept, or S == 0) */
} moe_layer_saved;
/* Selective recompute (Pangu Ultra MoE tech-report article, memory section: permutation and
 * activation recomputed instead of saved; Huawei MoE training-operator article, Selective R/S):
 * with saved->x_perm, saved->h and saved->h_sh NULL the forward keeps them in the workspace
 * only; the saved activations shrink by T*k*(d+f) + S*T*f_s elements. Results are identical.
 * With dims->rearrange = MOE_REARRANGE_GATHER (bf16, dropless) the rearrangement is fused
 * into the expert GEMMs instead (Huawei MoE training-operator article, "VectorSort": cut
 * repeated data movement): FWD1 and the dW13 product gather their x rows, the dX chain's
 * first product and the dW2 product their dY rows, straight from x / dy by row_src. x_perm
 * is then written only when the caller passes it, and dY is never rearranged in memory.
 * Otherwise the backward re-permutes x when saved->x_perm is NULL. */

typedef struct moe_layer_grads { /* caller-allocated outputs of moe_layer_bwd */
  void* dx;        /* [T, d]; includes the router term when w_r is given */
  void* dw13;      /* [E][2f][d] */
  void* dw2;       /* [E][d][f] */
  void* dws13;     /* [S][2f_s][d] or NULL when S == 0 */
  void* dws2;      /* [S][d][f_s] or NULL when S == 0 */
  float* dw_r;     /* [d][E] fp32, required when w_r is given, else ignored */
  float* dlogits;  /* [T][E] fp32 gradient w.r.t. the scores; required when logits_in was
                      given, optional (NULL) otherwise */
} moe_layer_grads;

/* Forward of one layer: router (unless logits_in), route, permute, grouped SwiGLU,
 * combine. logits_in [T][E] fp32 or NULL. y [T, d]. No host synchronisation. */
int moe_layer_fwd(const moe_layer_params* params, const void* x, const float* logits_in,
                  const moe_dims* dims, const moe_layer_saved* saved, void* y,
                  void* ws, size_t ws_bytes, moe_stream_t stream);

/* Backward of one layer from dy [T, d]: permute dY, expert dX chain, dgate -> score
 * gradient, combine dX (+ router term x-gradient when w_r is given), expert dW products,
 * router dW_r. The top-k indices are constants (not differentiated); the bias gets no
 * gradient. `saved` must hold the values moe_layer_fwd wrote for the same x. */
int moe_layer_bwd(const moe_layer_params* params, const moe_layer_saved* saved, const void* x,
                  const void* dy, const moe_dims* dims, const moe_layer_grads* grads,
                  void* ws, size_t ws_bytes, moe_stream_t stream);

/* ---------------------------------------------------------------- tracing */
/* Per-phase launch timing: while enabled, every kernel launch of the library is bracketed by
 * a pair of CUDA events on its stream (a few microseconds of host work per launch, no device
 * synchronisation). moe_trace_enable(1) clears the record and starts; (0) stops and clears.
 * moe_trace_read waits for the recorded events and fills up to max_entries entries, one per
 * phase that launched at least once (name is a static string; launches = kernel launches). */
typedef struct moe_trace_entry {
  const char* name;
  int64_t launches;
  double total_ms;
} moe_trace_entry;
int moe_trace_enable(int on);
int moe_trace_read(moe_trace_entry* out, int max_entries, int* n_out);

/* Failure-detection check: runs one bounded wait on a barrier that nothing completes, with
 * the given limit in nanoseconds, so that it records MOE_ERR_DEVICE_TIMEOUT in the error word
 * and returns without hanging (read it with moe_get_device_error). */
int moe_debug_timeout_probe(void* ws, size_t ws_bytes, uint64_t limit_ns, moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
