/*
 * moe_b300.h -- C ABI of the single-GPU MoE-layer forward for B300 (sm_103a).
 *
 * The forward pass is cut into the five steps that the expert-parallelism
 * tutorial "专家并行：混合专家模型的分布式训练方案" states in §2.1 (gate
 * decision, dispatch plan, token exchange, local expert compute, token
 * return), with the capacity rule of its §2.2 and the auxiliary loss of its
 * §5.1; the fine-grained EP deployment guide "细粒度专家并行部署实践与优化指南"
 * gives the same steps as pseudo-code in §七 (top-k of the gate
 * probabilities, dispatch, per-expert compute, gather back).  On one GPU the
 * two All-to-All exchanges become a row permutation and un-permutation in HBM.
 *
 *   moe_route      router linear layer, softmax over E, top-k     (§1.1, §2.1 step 1)
 *   moe_dispatch   capacity, slot ranks, drops, row permutation   (§2.1 steps 2-3, §2.2)
 *   moe_expert_ffn per-expert w1 -> activation -> w2, gate scale  (§2.1 step 4)
 *   moe_combine    gate-weighted sum back into token order        (§2.1 step 5)
 *   moe_aux_loss   L_aux = alpha * E * sum_i f_i * P_i            (§5.1)
 *
 * Routing variants from the ms-swift pages: moe_route_ex (group-limited
 * top-k, per-token log-sum-exp) and moe_z_loss (router z-loss).
 *
 * Backward (the layer is trained through the same steps in reverse: the
 * tutorial's §5.1 aux loss acts through its gradient, and the guide's 步骤三
 * item 3 returns the gradients by the reverse exchange; the pages give no
 * formula, so each call computes a derivative of the forward):
 *   moe_combine_bwd, moe_act_bwd, moe_route_bwd, moe_router_grads (or
 *   moe_grad_x + moe_router_wgrad), moe_expert_wgrad_rows (or moe_expert_wgrad on the
 *   packed transposes of moe_pack_segments_t),
 *   moe_expert_dgrad (the data-gradient GEMMs, B operand MN-major) and
 *   moe_expert_up_z (the forward keeping the pre-activation).
 *
 * Conventions shared by every call
 * --------------------------------
 * Ownership   The caller allocates and owns every buffer (inputs, outputs,
 *             intermediates and workspaces).  The library never allocates
 *             device or host memory and never synchronises the stream on the
 *             compute calls.
 * Pointers    Every array argument is a DEVICE pointer, row-major, 16-byte
 *             aligned (torch allocations are).  Sizes are element counts.
 * Streams     Work is enqueued on `stream` and runs asynchronously.
 * Errors      Bad arguments and launch failures come back synchronously as a
 *             moe_status; nothing is enqueued when a call returns an error.
 *             Problems found on the device (an expert id out of range, a
 *             pipeline wait that ran past its time limit) set a sticky device
 *             status word that moe_check() reads and clears.  No kernel traps.
 * Indices     int32: T*k < 2^31, E <= 256, 1 <= k <= min(E, 16).
 * Shapes      d % 64 == 0 and F % 64 == 0 (16-byte rows for the vector
 *             moves, 64-element K blocks for the tensor-core GEMMs).
 * Dtypes      x, w1, w2, h, y_perm and y share one dtype (MOE_F32 or
 *             MOE_BF16); the router weight, bias, gates and prob sums are
 *             fp32.  bf16 data is accumulated in fp32 and rounded once per
 *             stored tensor; the fp32 path uses no TF32 and no bf16.
 * Residual    Adding the layer input back (the residual path that dropped
 *             tokens take, §2.2) is the caller's job: a dropped slot
 *             contributes zero to y.
 */
#ifndef MOE_B300_H
#define MOE_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; declared here so the header needs no CUDA
 * headers.  NULL is the legacy default stream. */
typedef struct CUstream_st* moe_stream_t;

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,   /* NULL pointer, size out of range, bad enum */
    MOE_ERR_UNSUPPORTED = 2,   /* valid but not implemented (shape rule, dtype) */
    MOE_ERR_WORKSPACE = 3,     /* ws NULL or ws_bytes below moe_workspace_bytes() */
    MOE_ERR_CUDA = 4,          /* a CUDA runtime/driver call or launch failed */
    MOE_ERR_TIMEOUT = 5        /* (moe_check) a device-side wait hit its limit */
} moe_status;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype;

typedef enum {
    MOE_ACT_GELU = 0,      /* exact erf GELU: z * (1 + erf(z / sqrt 2)) / 2        */
    MOE_ACT_SWIGLU = 1,    /* silu(z[0:F]) * z[F:2F]; w1[e] rows 0..F-1 gate, F..2F-1 up */
    MOE_ACT_IDENTITY = 2   /* h = z; for checks (identity experts)                 */
} moe_act;

typedef enum {
    MOE_CALL_ROUTE = 0,
    MOE_CALL_DISPATCH = 1,
    MOE_CALL_FFN = 2,
    MOE_CALL_ROUTER_WGRAD = 3,
    MOE_CALL_ROUTER_GRADS = 4
} moe_call;

/* ---------------------------------------------------------------- host --- */

/* Expert capacity of the tutorial's §2.2: round((T / E) * cf), rounded half
 * away from zero in double precision, no minimum.  cf <= 0 selects dropless
 * routing and returns T.  Returns -1 when T < 0 or E < 1. */
int64_t moe_capacity(int64_t T, int E, double cf);

/* Rows of the permuted buffers (x_perm, h, y_perm, row_token, row_gate):
 * the largest possible number of kept slots, min(T * k, E * cap).
 * Returns -1 on invalid arguments. */
int64_t moe_perm_rows_max(int64_t T, int k, int E, int64_t cap);

/* Bytes of device workspace the given call needs at these sizes (0 = none;
 * pass ws = NULL then).  Returns 0 for an unknown call. */
size_t moe_workspace_bytes(moe_call call, int64_t T, int d, int E, int k, int F,
                           moe_act act, moe_dtype dtype);

/* Static text for a status code. */
const char* moe_status_string(moe_status s);

/* ABI revision of this header (bumped on any incompatible change). */
int moe_abi_version(void);
#define MOE_ABI_VERSION 1

/* ------------------------------------------------------------- compute --- */

/* Router: tutorial §1.1 (a lightweight linear layer scores every expert),
 * §2.1 step 1 (each token picks its Top-K experts); guide §七 takes top-k of
 * the softmaxed gate probabilities.
 *   x          [T, d]  xdt (F32 or BF16)
 *   w_router   [E, d]  fp32;  b_router [E] fp32 or NULL
 *   logits l[t,e] = sum_c x[t,c] w_router[e,c] + b[e]  (fp32 accumulation)
 *   p[t,:]     = softmax over all E experts
 * Outputs (all written, caller-owned):
 *   topk_idx   [T, k]  int32: experts ordered by (logit desc, index asc);
 *                      ties go to the lower expert index; j is the k-rank
 *   topk_gate  [T, k]  fp32: p[t, idx]; divided by sum_j p[t, idx[t,j]] when
 *                      renorm != 0
 *   prob_sum   [E]     fp32: sum_t p[t,e], bitwise reproducible run to run:
 *                      a fixed-order sum, or (bf16 x, E <= 64) per-block
 *                      sums added as 64-bit fixed point (resolution 2^-32,
 *                      integer adds, so the order does not matter)
 *   ws         >= moe_workspace_bytes(MOE_CALL_ROUTE, T, d, E, k, ...) bytes
 * T == 0 is allowed (prob_sum becomes zeros). */
moe_status moe_route(const void* x, moe_dtype xdt, const float* w_router, const float* b_router,
                     int64_t T, int d, int E, int k, int renorm,
                     int32_t* topk_idx, float* topk_gate, float* prob_sum,
                     void* ws, size_t ws_bytes, moe_stream_t stream);

/* moe_route with the routing variants.
 * Group-limited routing, from "ms-swift MoE模型加速：Megatron并行实测提速10倍"
 * §3.2 (EP bullet): the router first picks the token's expert group, then
 * runs Top-k inside it.  That page fixes no more; the readings taken: the E
 * experts form n_group contiguous groups of E / n_group (the EP placement of
 * the same section); a group's score is its largest logit; the topk_group
 * groups of highest score are kept (equal scores: lower group index); the k
 * experts are then chosen among the kept groups' experts exactly as
 * moe_route orders them.  The softmax, the gates (and their renormalisation)
 * and prob_sum stay those over all E experts.  n_group = 1 is moe_route.
 *   n_group     1..32, dividing E;  topk_group 1..n_group;
 *               k <= topk_group * E / n_group (else MOE_ERR_INVALID_ARG)
 *   lse         [T] fp32 or NULL: log sum_e exp(l[t,e]) per token, the
 *               input of moe_z_loss
 *   logits      [T, E] fp32 or NULL: the logits (bias included), the input
 *               of moe_route_bwd
 * Other arguments, outputs and workspace as moe_route. */
moe_status moe_route_ex(const void* x, moe_dtype xdt, const float* w_router, const float* b_router,
                        int64_t T, int d, int E, int k, int renorm, int n_group, int topk_group,
                        int32_t* topk_idx, float* topk_gate, float* prob_sum, float* lse, float* logits,
                        void* ws, size_t ws_bytes, moe_stream_t stream);

/* Dispatch: tutorial §2.1 steps 2-3 (dispatch plan, token exchange) and
 * §2.2 (capacity, overflow tokens dropped).  Assignments (t, j) are granted
 * expert slots in k-rank-then-token order -- every first choice in token
 * order, then every second choice, ... -- and an assignment whose place in
 * its expert's queue is >= cap is dropped.  The exchange becomes a gather of
 * x rows into expert-contiguous segments.
 *   topk_idx [T,k] int32, topk_gate [T,k] fp32 (from moe_route)
 *   x        [T, d] xdt
 * Outputs:
 *   counts   [E]    assignments per expert before drops
 *   kept     [E]    min(counts, cap)
 *   offsets  [E+1]  exclusive prefix sum of kept; offsets[E] = kept slots A
 *   slot_row [T,k]  row of x_perm holding (t, j), or -1 when dropped;
 *                   slot_row - offsets[e] is the place in expert e's queue
 *   row_token[rows_max], row_gate[rows_max], x_perm[rows_max, d]: rows
 *                   0..A-1 filled (token id, gate, copy of x[token]); rows
 *                   A..rows_max-1 are left untouched.  x_perm may be NULL:
 *                   then no rows are copied (for moe_expert_up_gathered,
 *                   which reads x through row_token itself)
 *   n_dropped[1]    sum_e max(0, counts[e] - cap)
 *   rows_max = moe_perm_rows_max(T, k, E, cap); cap >= 0.
 * An expert id outside [0, E) in topk_idx sets the device status (the
 * assignment is ignored). */
moe_status moe_dispatch(const int32_t* topk_idx, const float* topk_gate, int64_t T, int k, int E,
                        int64_t cap, const void* x, moe_dtype xdt, int d,
                        int32_t* counts, int32_t* kept, int32_t* offsets, int32_t* slot_row,
                        int32_t* row_token, float* row_gate, void* x_perm, int32_t* n_dropped,
                        void* ws, size_t ws_bytes, moe_stream_t stream);

/* Expert up-projection: tutorial §2.1 step 4 (each expert is an FFN run on
 * the tokens it received); the expert shape d -> d_ff -> d with w1
 * column-split and w2 row-split is the one the ETP page
 * "ETP专家并行加速MoE模型：ms-swift中稀疏架构的极致优化" describes.
 * For every expert e and row r in [offsets[e], offsets[e] + kept[e]):
 *   z = w1[e] . x_perm[r]        (w1 [E, N1, d], nn.Linear layout; N1 = 2F for
 *                                 SwiGLU, F otherwise)
 *   h[r, :F] = act(z)            fp32 accumulate, one rounding to dtype
 * BF16 runs on the tcgen05 tensor cores (TMA-fed, TMEM accumulators); F32 on
 * CUDA cores in true fp32.  rows_max is the row count of x_perm and h.
 * Rows outside the kept segments are not written. */
moe_status moe_expert_up(const void* x_perm, const int32_t* offsets, const int32_t* kept,
                         int E, int d, int F, moe_act act, moe_dtype dtype, const void* w1,
                         int64_t rows_max, void* h, moe_stream_t stream);

/* Row permutation: dst[i] = src[index[i]] for i < n (rows of d elements of
 * dtype; rows 16-byte multiples, 16-byte aligned buffers).  The pages' §2.1
 * token exchange regroups received rows by expert; the expert-parallel
 * layer uses this to turn rows grouped by source rank into rows grouped by
 * local expert and back. */
moe_status moe_permute_rows(const void* src, const int32_t* index, int64_t n, int d, moe_dtype dtype, void* dst,
                            moe_stream_t stream);

/* moe_expert_up that also keeps the pre-activation for the backward:
 *   z [rows_max, N1] bf16 = w1[e] . x_perm[r] before the activation (SwiGLU:
 *   gate columns 0..F-1, up columns F..2F-1), rows < offsets[E] written.
 * BF16 only (MOE_ERR_UNSUPPORTED otherwise); the 1-SM kernel always runs. */
moe_status moe_expert_up_z(const void* x_perm, const int32_t* offsets, const int32_t* kept, int E, int d, int F,
                           moe_act act, moe_dtype dtype, const void* w1, int64_t rows_max, void* h, void* z,
                           moe_stream_t stream);

/* moe_expert_up reading its A rows straight from x: row r of the permuted
 * order is x[row_token[r]] (row_token from moe_dispatch), so the dispatch can
 * skip materialising x_perm (the tutorial's §5.3 packs tokens for contiguous
 * transfer; here the GEMM's producer copies the rows in place).
 *   x [T, d] bf16, 16-byte aligned, T * d * 2 < 2^32 bytes (else
 *   MOE_ERR_UNSUPPORTED); row_token [rows_max]; other arguments as
 *   moe_expert_up.  BF16 only (MOE_ERR_UNSUPPORTED otherwise). */
moe_status moe_expert_up_gathered(const void* x, int64_t T, const int32_t* row_token, const int32_t* offsets,
                                  const int32_t* kept, int E, int d, int F, moe_act act, moe_dtype dtype,
                                  const void* w1, int64_t rows_max, void* h, moe_stream_t stream);

/* Expert down-projection with the gate scale of the combine folded in:
 *   y_perm[r, :] = row_gate[r] * (w2[e] . h[r, :F])     (w2 [E, d, F])
 * fp32 accumulate and gate product, one rounding to dtype.  Same segment
 * rules as moe_expert_up. */
moe_status moe_expert_down(const void* h, const int32_t* offsets, const int32_t* kept,
                           int E, int d, int F, moe_dtype dtype, const void* w2,
                           const float* row_gate, int64_t rows_max, void* y_perm,
                           moe_stream_t stream);

/* moe_expert_up followed by moe_expert_down on the same stream.
 * ws may be NULL (moe_workspace_bytes(MOE_CALL_FFN, ...) is 0). */
moe_status moe_expert_ffn(const void* x_perm, const int32_t* offsets, const int32_t* kept,
                          int E, int d, int F, moe_act act, moe_dtype dtype,
                          const void* w1, const void* w2, const float* row_gate,
                          int64_t rows_max, void* h, void* y_perm,
                          void* ws, size_t ws_bytes, moe_stream_t stream);

/* Combine: tutorial §2.1 step 5 (outputs return to their original token
 * positions) with the guide's §七 gather-back.  The gate weights are already
 * inside y_perm, so
 *   y[t] = sum_{j : slot_row[t,j] >= 0} y_perm[slot_row[t,j]]
 * summed in j order in fp32 and rounded once; a token with every slot
 * dropped gets a zero row.  y [T, d] has dtype `dtype`. */
moe_status moe_combine(const void* y_perm, const int32_t* slot_row, int64_t T, int k, int d,
                       moe_dtype dtype, void* y, moe_stream_t stream);

/* Auxiliary load-balance loss, tutorial §5.1:
 *   L = alpha * E * sum_e f_e * P_e,  f_e = counts[e] / T,  P_e = prob_sum[e] / T
 * (f counts every choice before capacity drops).  Computed in fp64 on the
 * device, stored as fp32 to loss[0] (device pointer).  T must be >= 1.
 * Passing kept[] (from moe_dispatch) as counts gives the post-drop variant,
 * where f_e counts only the slots that survived the capacity cut. */
moe_status moe_aux_loss(const int32_t* counts, const float* prob_sum, int64_t T, int E,
                        float alpha, float* loss, moe_stream_t stream);

/* moe_combine and moe_aux_loss in one launch (the first warp of the combine
 * computes the loss, with the same arithmetic as moe_aux_loss): the two
 * closing steps of the forward.  Arguments as in the two calls; T >= 1. */
moe_status moe_combine_aux(const void* y_perm, const int32_t* slot_row, int64_t T, int k, int d, moe_dtype dtype,
                           void* y, const int32_t* counts, const float* prob_sum, int E, float alpha, float* loss,
                           moe_stream_t stream);

/* Router z-loss.  "ETP专家并行加速MoE模型：ms-swift中稀疏架构的极致优化", section
 * on dynamic routing, names a routing z-loss that spreads the router's
 * choices but gives no formula; this is the router z-loss of ST-MoE (Zoph et
 * al. 2022, eq. 5):
 *   loss = beta * (1/T) * sum_t lse[t]^2,   lse from moe_route_ex
 * Summed in fp64 in a fixed order on the device, stored as fp32 to loss[0]
 * (device pointer).  T must be >= 1. */
moe_status moe_z_loss(const float* lse, int64_t T, float beta, float* loss, moe_stream_t stream);

/* ------------------------------------------------------------ backward --- */
/* Gradients of L = <dy, y> + aux_weight * L_aux + z_weight * L_z.  The top-k
 * choice, the capacity cut and f_e carry no gradient; a dropped slot's gate
 * gets none either.  bf16 layers only (MOE_ERR_UNSUPPORTED otherwise); fp32
 * results where noted.  A training step runs, after the forward (with
 * moe_route_ex keeping logits):
 *   do_perm, dgate   = moe_combine_bwd(dy, ...)
 *   z                = kept by moe_expert_up_z in the forward, or recomputed:
 *                      moe_expert_up(x_perm, ..., IDENTITY, F := N1, w1)
 *   dz               = moe_expert_dgrad_act(do_perm, ..., w2, z)  (the da GEMM
 *                      with moe_act_bwd in its epilogue; identity: moe_expert_dgrad)
 *   dx_perm          = moe_expert_dgrad(dz, ..., K = N1, N = d, w1)
 *   dw2[e]           = moe_expert_wgrad_rows(do_perm, h, M = d, N = F)
 *   dw1[e]           = moe_expert_wgrad_rows(dz, x_perm, M = N1, N = d)
 *                      (or moe_expert_wgrad on moe_pack_segments_t copies)
 *   dl               = moe_route_bwd(logits, topk_idx, dgate, counts, ...)
 *   dx, dW, db       = moe_router_grads(dx_perm, slot_row, dl, w_router, x)
 *                      (tensor cores; or moe_grad_x + moe_router_wgrad)       */

/* Data-gradient GEMM on the weights as stored (no transposed copy):
 *   out[r, n] = sum_k a[r, k] * w[e][k][n]   for kept rows r of expert e
 * a [rows_max, K] (segments as from moe_dispatch), w [E, K, N] (N contiguous:
 * w2 as [E, d, F] gives da from do_perm; w1 as [E, N1, d] gives dx_perm from
 * dz), out [rows_max, N]; bf16, fp32 accumulation, one rounding.
 * K % 64 == 0, N % 64 == 0. */
moe_status moe_expert_dgrad(const void* a, const int32_t* offsets, const int32_t* kept, int E, int K, int N,
                            moe_dtype dtype, const void* w, int64_t rows_max, void* out, moe_stream_t stream);

/* The da GEMM with the activation backward in its epilogue:
 *   da = do_perm[r] . w2[e] (fp32, never stored), dz = act'(z) * da  as
 *   moe_act_bwd, from the kept pre-activation z [rows_max, N1]
 * dz [rows_max, N1] bf16.  act GELU or SWIGLU; d % 64 == 0, F % 64 == 0. */
moe_status moe_expert_dgrad_act(const void* do_perm, const int32_t* offsets, const int32_t* kept, int E, int d,
                                int F, moe_act act, moe_dtype dtype, const void* w2, const void* z, int64_t rows_max,
                                void* dz, moe_stream_t stream);

/* w [E, R, C] -> wt [E, C, R] (2-byte elements; R, C multiples of 64;
 * 16-byte aligned). */
moe_status moe_transpose_experts(const void* w, int E, int R, int C, moe_dtype dtype, void* wt,
                                 moe_stream_t stream);

/* Combine backward.  For every kept slot r = slot_row[t, j] (gate g_r =
 * row_gate[r], y_perm[r] = g_r * o_r from moe_expert_down):
 *   do_perm[r]  = g_r * dy[t]             bf16 [rows_max, d]
 *   dgate[t, j] = <dy[t], y_perm[r]> / g_r = <dy[t], o_r>    fp32 [T, k]
 * dgate of a dropped slot is 0.  dy [T, d] bf16; d % 64 == 0. */
moe_status moe_combine_bwd(const void* dy, const int32_t* slot_row, const float* row_gate, const void* y_perm,
                           int64_t T, int k, int d, moe_dtype dtype, void* do_perm, float* dgate,
                           moe_stream_t stream);

/* Activation backward over the kept rows r < offsets[E]:
 *   GELU     dz = da * (Phi(z) + z phi(z))                        dz [rows, F]
 *   SwiGLU   dz[:, :F] = da * z_up * silu'(z_gate), dz[:, F:] = da * silu(z_gate)   dz [rows, 2F]
 *   IDENTITY dz = da
 * z [rows, N1] is the pre-activation (moe_expert_up with IDENTITY on w1), da
 * [rows, F] the gradient of the activation output.  bf16, F % 64 == 0. */
moe_status moe_act_bwd(const void* z, const void* da, const int32_t* offsets, int E, int F, moe_act act,
                       moe_dtype dtype, int64_t rows_max, void* dz, moe_stream_t stream);

/* Columns of the packed transposed operands of moe_expert_wgrad:
 * rows_max + 64 E rounded up to 64 (each segment is padded to 64). */
int64_t moe_wgrad_cols(int64_t rows_max, int E);

/* dst [C, ld] (2-byte elements) from the expert segments of src [rows_max, C]:
 * expert e's row offsets[e] + i lands in column 64 * kstart[e] + i, where
 * kstart[e] = sum over e' < e of ceil(kept[e'] / 64); the padding columns of
 * each segment are zero.  ld >= moe_wgrad_cols(rows_max, E), ld % 64 == 0,
 * C % 64 == 0.  Columns past the last segment are left untouched. */
moe_status moe_pack_segments_t(const void* src, const int32_t* offsets, const int32_t* kept, int E, int C,
                               int64_t rows_max, int64_t ld, moe_dtype dtype, void* dst, moe_stream_t stream);

/* Per-expert weight gradient on the tensor cores:
 *   dw[e] = at[:, seg_e] . bt[:, seg_e]^T      [E, M, N], fp32 accumulation
 * at [M, ld] and bt [N, ld] (dtype bf16) come from moe_pack_segments_t
 * (seg_e = expert e's packed, zero-padded columns); an expert with no rows
 * gets zeros.  dw_dtype: MOE_F32, or MOE_BF16 (the weights' own type, one
 * rounding).  M % 64 == 0, N % 64 == 0, ld % 64 == 0. */
moe_status moe_expert_wgrad(const void* at, const void* bt, const int32_t* kept, int E, int M, int N, int64_t ld,
                            moe_dtype dtype, void* dw, moe_dtype dw_dtype, moe_stream_t stream);

/* The same weight gradient read straight from the row-major activations (no
 * packed copies):
 *   dw[e] = sum over rows r in [offsets[e], offsets[e] + kept[e]) of
 *           a[r, :]^T b[r, :]                   [E, M, N], fp32 accumulation
 * a [rows_max, M] and b [rows_max, N] (dtype bf16): do_perm and h give dw2
 * (M = d, N = F), dz and x_perm give dw1 (M = N1, N = d).  Only the rows of
 * the segments are read into the sums; rows between or past them may hold
 * anything.  An expert with no rows (and every expert when rows_max == 0)
 * gets zeros.  dw_dtype MOE_F32 or MOE_BF16 (one rounding).  M % 64 == 0,
 * N % 64 == 0; offsets[e] + kept[e] <= rows_max. */
moe_status moe_expert_wgrad_rows(const void* a, const void* b, const int32_t* offsets, const int32_t* kept, int E,
                                 int M, int N, int64_t rows_max, moe_dtype dtype, void* dw, moe_dtype dw_dtype,
                                 moe_stream_t stream);

/* Router backward to the logits, per token (logits [T, E] from moe_route_ex,
 * topk_idx and dgate [T, k], counts [E] = f_e * T: counts for the pre-drop
 * aux loss, kept for the post-drop one):
 *   dp[e_j] += (dgate_j - sum_i dgate_i g_i) / S   (renorm; S = sum of the k
 *              chosen probabilities, g = p / S)    or  dgate_j
 *   dp[e]   += aux_coef * counts[e] / T^2          (aux_coef = aux_weight * alpha * E)
 *   dl      = p * (dp - <p, dp>) + z_coef * (2 / T) * lse * p   (z_coef = z_weight * beta)
 * dl fp32 [T, E]. */
moe_status moe_route_bwd(const float* logits, const int32_t* topk_idx, const float* dgate, const int32_t* counts,
                         int64_t T, int E, int k, int renorm, float aux_coef, float z_coef, float* dl,
                         moe_stream_t stream);

/* Input gradient: dx[t] = sum over kept j of dx_perm[slot_row[t, j]] +
 * sum_e dl[t, e] w_router[e] (fp32 sums, one rounding to dtype).
 * dx_perm [rows_max, d] and dx [T, d] in dtype; dl [T, E]; w_router [E, d];
 * d % 64 == 0 and 16-byte aligned dx_perm, w_router, dx (else UNSUPPORTED). */
moe_status moe_grad_x(const void* dx_perm, const int32_t* slot_row, const float* dl, const float* w_router,
                      int64_t T, int k, int E, int d, moe_dtype dtype, void* dx, moe_stream_t stream);

/* Router weight gradient: dW[e, c] = sum_t dl[t, e] x[t, c] (fp32 [E, d]) and,
 * when db != NULL, db[e] = sum_t dl[t, e] (fp32 [E]); token splits summed in a
 * fixed order (bitwise reproducible).  ws >=
 * moe_workspace_bytes(MOE_CALL_ROUTER_WGRAD, T, d, E, ...) bytes; T >= 1;
 * d % 64 == 0 and x 16-byte aligned (else UNSUPPORTED). */
moe_status moe_router_wgrad(const float* dl, const void* x, moe_dtype xdt, int64_t T, int E, int d, float* dW,
                            float* db, void* ws, size_t ws_bytes, moe_stream_t stream);

/* The input gradient and the router weight gradient of moe_grad_x and
 * moe_router_wgrad in one call, their two contractions on the tensor cores:
 *   dx[t] = rn(sum_e dl[t, e] w_router[e] + sum over kept j of dx_perm[slot_row[t, j]])
 *   dW    = dl^T x   (fp32 [E, d]),   db[e] = sum_t dl[t, e]   (fp32 [E])
 * The fp32 dl and w_router enter the bf16 MMAs as hi + lo parts (hi = rn(v),
 * lo = rn(v - hi)): dl . W takes hi.hi + lo.hi + hi.lo, dl^T x takes
 * hi + lo (x is bf16), fp32 accumulation; the relative error of the parts
 * is at most 2^-16 (~2^-17 seen), far below dx's bf16 rounding.  Sums run in a fixed order
 * (bitwise reproducible).  dtype (x, dx_perm, dx) MOE_BF16; d % 64 == 0;
 * 16-byte aligned x, dx_perm, w_router, dx, dW, ws.  ws >=
 * moe_workspace_bytes(MOE_CALL_ROUTER_GRADS, T, d, E, ...) bytes (it holds
 * the bf16 parts, the fp32 dl . W and the split weight-gradient partials).
 * T == 0 zeroes dW and db. */
moe_status moe_router_grads(const void* dx_perm, const int32_t* slot_row, const float* dl, const float* w_router,
                            const void* x, int64_t T, int k, int E, int d, moe_dtype dtype, void* dx, float* dW,
                            float* db, void* ws, size_t ws_bytes, moe_stream_t stream);

/* ------------------------------------------------- no-allocation variant --- */

/* moe_dispatch without a caller workspace.  The pages have no counterpart to
 * this entry point: it exists for callers that cannot allocate device memory
 * where they run the layer -- a plugin enqueue callback of an inference
 * engine that must not call cudaMalloc, a process whose device memory is all
 * handed out by its own pool, a latency-critical loop that cannot take the
 * device-wide synchronisation an allocation may cause.
 *
 * Same arguments, outputs and errors as moe_dispatch, minus ws / ws_bytes.
 * Its scratch (the per-chunk expert histograms) is a fixed 256 KiB array in
 * the library's device memory, which every GPU that loads the library holds
 * until the process exits.  Limit: moe_workspace_bytes(MOE_CALL_DISPATCH,
 * T, d, E, k, ...) <= 262144, i.e. ceil(T*k / c) * E <= 65536 with chunks of
 * c = 256 assignments up to T*k = 65536 and c = 1024 above (for example
 * T*k <= 262144 at E = 256); larger calls return MOE_ERR_WORKSPACE with a
 * message on stderr and enqueue nothing.  It calls no cudaMalloc, cudaFree
 * or allocating library routine.
 *
 * The first call on a device with T*k > 0 looks up the array's device
 * address with that device current (once per device); make that first call
 * before any stream capture.  Every call shares the one array and the array keeps the last
 * call's contents: each call overwrites every histogram cell it reads, so
 * nothing needs clearing, but calls that overlap on the GPU (different
 * streams, or different host threads, with no ordering between them) race on
 * the array and must not be issued. */
moe_status moe_dispatch_noalloc(const int32_t* topk_idx, const float* topk_gate, int64_t T, int k, int E,
                                int64_t cap, const void* x, moe_dtype xdt, int d,
                                int32_t* counts, int32_t* kept, int32_t* offsets, int32_t* slot_row,
                                int32_t* row_token, float* row_gate, void* x_perm, int32_t* n_dropped,
                                moe_stream_t stream);

/* ---------------------------------------------------------- diagnostics --- */

/* Synchronises `stream`, then reads and clears the device status word of the
 * current device: MOE_OK, MOE_ERR_TIMEOUT (a pipeline wait ran past its
 * limit), MOE_ERR_INVALID_ARG (an out-of-range expert id reached dispatch),
 * or MOE_ERR_CUDA (the stream reported an error). */
moe_status moe_check(moe_stream_t stream);

/* Time limit of every device-side wait, in SM clock cycles (default 4e9,
 * about two seconds).  A wait that runs past it records MOE_ERR_TIMEOUT and
 * its kernel winds down cleanly.  0 restores the default. */
void moe_set_wait_limit(uint64_t cycles);

/* Kernel family of the bf16 expert GEMMs: 0 (default) automatic, 1 one SM
 * per 128-token x 256-column tile, 2 CTA pairs (two SMs per 256-weight-row x
 * up-to-256-token tile).  Process-wide; for tests and tuning.
 * MOE_ERR_INVALID_ARG for any other value. */
moe_status moe_set_gemm_kernel(int kind);

/* Output-tile width of the one-SM bf16 expert GEMMs: 128, 192 or 256 columns, or 0
 * (the default) to pick per call the width whose tiles best fill whole waves
 * of the SMs.  Process-wide; for tests and tuning.  MOE_ERR_INVALID_ARG for
 * any other value. */
moe_status moe_set_gemm_tile_n(int bn);

/* Tile order of the forward and data-gradient bf16 expert GEMMs inside each
 * expert: 0 (default) automatic (M-fastest: the blocks running together
 * share a weight tile), 1 M-fastest, 2 N-fastest (they share a row tile).
 * The results do not depend on it.  Process-wide; for tests and tuning.
 * MOE_ERR_INVALID_ARG otherwise. */
moe_status moe_set_gemm_order(int order);

/* Last wave of the forward bf16 expert GEMMs with 256-column tiles (GELU,
 * identity and gate epilogues): 1 (default) lets a launch whose tiles end in
 * a wave that would leave at least half of the SMs idle run that wave's R
 * tiles as 2R units of 128 columns, one per SM; 0 keeps whole tiles.  The
 * results do not depend on it (every output is the same dot product in the
 * same K order).  Process-wide; for tests and tuning.  MOE_ERR_INVALID_ARG
 * for any other value. */
moe_status moe_set_gemm_tail_halves(int on);

/* Programmatic dependent launch between the library's kernels: 1 (default)
 * launches each kernel after the first of a call as a programmatic dependent
 * of the one before it (its set-up overlaps that kernel's end; it waits for
 * that kernel's results before reading them), 0 plain stream order.  The
 * results do not depend on it.  Process-wide, read at each launch (a CUDA
 * graph keeps what was set when it was captured); for tests and tuning.
 * MOE_ERR_INVALID_ARG for any other value. */
moe_status moe_set_launch_overlap(int on);

/* Output of the forward expert GEMMs (moe_expert_up, moe_expert_down,
 * moe_expert_ffn; the up projection of moe_expert_up_z keeps per-thread
 * stores) and of moe_expert_dgrad: 1 (default) writes each whole block of 32
 * rows x 64 columns of h, y_perm or dx_perm through shared memory with one
 * TMA store when the launch has at
 * least 3 row tiles of 128 per expert on average (below that the GEMM streams
 * its weights and keeps per-thread stores), 0 always per-thread 16-byte
 * stores.  The results do not depend on it.  Process-wide; for tests and
 * tuning.  MOE_ERR_INVALID_ARG for any other value. */
moe_status moe_set_gemm_tma_store(int on);

/* Router kernel for bf16 x: 0 (default) automatic (the tensor-core router
 * for E <= 128), 1 the tensor-core router wherever it applies, 2 the
 * CUDA-core router for E <= 8 (d a multiple of 256, at most 4096: one fused
 * kernel for logits, softmax, top-k and per-block probability sums, then the
 * fixed-order sum of the blocks' rows) wherever it applies.  Both give the
 * routing the pages define within fp32 rounding (identical selections away
 * from near-ties).  Process-wide; for tests and tuning.  MOE_ERR_INVALID_ARG
 * for any other value. */
moe_status moe_set_router_kernel(int kind);

/* Tile order of the weight-gradient GEMMs (moe_expert_wgrad,
 * moe_expert_wgrad_rows) inside each expert: 0 (default) automatic
 * (N-fastest), 1 M-fastest, 2 N-fastest.  The results do not depend on it.
 * Process-wide; for tests and tuning.  MOE_ERR_INVALID_ARG otherwise. */
moe_status moe_set_wgrad_order(int order);

/* Launches one block that waits, under the current limit, on a barrier that
 * nothing ever completes, so that a test can watch the time-limit path end
 * in MOE_ERR_TIMEOUT from moe_check() with the context still usable. */
moe_status moe_selftest_wait_timeout(moe_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_B300_H */
