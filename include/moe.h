/*
 * moe.h -- C ABI of the B300 (sm_103a) MoE layer hot path.
 *
 * One Mixture-of-Experts layer on one GPU, in the four steps the Ultralytics
 * glossary page "Expert Parallelism" gives in its section "How tokens move between
 * GPUs" (German edition: "Wie Tokens zwischen GPUs uebertragen werden"):
 *   1. routing   -- moe_route       score every expert per token, keep the top k
 *   2. dispatch  -- moe_dispatch    count, cap, and permute hidden states into the
 *                                   contiguous per-expert (per-rank) send layout
 *   3. compute   -- moe_expert_ffn  run each expert on the rows it received
 *   4. combine   -- moe_combine     return outputs to token order, weighted by the
 *                                   router scores, and sum
 * plus the bias-based balancing step of the section "Load balancing and capacity"
 * (moe_bias_update).  Expert-parallel ranks are logical to these calls: the expert
 * -> rank map yields the per-rank counts and offsets an all-to-all would use as its
 * splits, and nothing leaves the GPU.  Ranks on separate devices exchange, between
 * moe_dispatch and moe_expert_ffn, the send buffer's chunk of each (rank, expert)
 * pair (rows expert_start[e] .. + kept_counts[e]); a receiving rank lays its rows out
 * expert by expert and calls moe_expert_ffn with a configuration of its local
 * experts only (their counts and starts, their weights); the results go back to the
 * rows they came from before moe_combine.  The Python package's ep module does this
 * with point-to-point messages.
 *
 * Conventions (all calls):
 *   - Every pointer argument is a DEVICE pointer unless its comment says "host".
 *     The caller allocates and owns every buffer; no call allocates device memory.
 *     Scratch memory comes only from the caller's workspace (moe_workspace_size).
 *   - Calls are asynchronous and ordered on `stream` (a cudaStream_t passed as
 *     void*; NULL = the legacy default stream).  No call synchronises the host and
 *     nothing is read back to the host: counts stay on the device.
 *   - Arguments are validated on the host before anything is launched; a rejected
 *     call launches nothing and returns MOE_ERR_INVALID_ARG (bad sizes, null or
 *     misaligned pointers), MOE_ERR_WORKSPACE (workspace too small),
 *     MOE_ERR_UNSUPPORTED (device is not compute capability 10.3).  A failed
 *     launch returns MOE_ERR_CUDA.  No exception crosses this interface.
 *   - Activation buffers (x, xperm, yperm, yshared, out, expert weights) have the
 *     element type cfg->act_dtype and must be 16-byte aligned; `hidden` and `d_ff`
 *     must be multiples of 8.  Row-major throughout.
 *   - Router logits must be finite; NaN logits give unspecified routing.
 *   - Buffers written by one call must not alias buffers it reads.
 */
#ifndef MOE_B300_H
#define MOE_B300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,
  MOE_ERR_UNSUPPORTED = 2,
  MOE_ERR_WORKSPACE = 3,
  MOE_ERR_CUDA = 4
} moe_status;

enum { MOE_DTYPE_F32 = 0, MOE_DTYPE_BF16 = 1 };
enum { MOE_SCORE_SOFTMAX = 0, MOE_SCORE_SIGMOID = 1 };
enum { MOE_RANK_CONTIGUOUS = 0, MOE_RANK_ROUND_ROBIN = 1 };
enum { MOE_DISPATCH_PACKED = 0, MOE_DISPATCH_CAPACITY_PADDED = 1 };

/* Layer configuration (host struct, passed by const pointer; read during the call
 * only).  Limits: 1 <= tokens; 8 <= hidden, hidden % 8 == 0;
 * 1 <= num_experts <= 256; 1 <= top_k <= min(8, num_experts);
 * 1 <= num_ranks <= num_experts (num_experts % num_ranks == 0 for the contiguous
 * map); num_groups divides num_experts; 1 <= topk_groups <= num_groups and
 * topk_groups * (num_experts / num_groups) >= top_k; d_ff >= 8, d_ff % 8 == 0;
 * shared_d_ff == 0 or a multiple of 8; num_experts * 2 * d_ff, num_experts * hidden
 * and 2 * shared_d_ff each at most 2^31 - 1 (weight rows take 32-bit coordinates). */
typedef struct {
  int32_t tokens;          /* N: tokens in the batch */
  int32_t hidden;          /* d: hidden size of a token */
  int32_t num_experts;     /* E: routed experts */
  int32_t top_k;           /* k: experts kept per token */
  int32_t num_ranks;       /* R: logical expert-parallel ranks ("GPUs" on the page) */
  int32_t rank_map;        /* MOE_RANK_CONTIGUOUS: rank = e / (E/R) (experts 0..E/R-1 on
                              rank 0, as in the page's example); MOE_RANK_ROUND_ROBIN:
                              rank = e % R */
  int32_t score_fn;        /* MOE_SCORE_SOFTMAX or MOE_SCORE_SIGMOID (+ selection bias) */
  int32_t normalize_topk;  /* nonzero: combine weights renormalised over the k kept */
  int32_t num_groups;      /* expert groups (one per node); 1 = no group limit */
  int32_t topk_groups;     /* groups a token may use; 1 when num_groups == 1 */
  float capacity_factor;   /* > 0: per-expert cap C = ceil(cf * N * k / E); <= 0: none */
  int32_t d_ff;            /* F: routed expert intermediate size */
  int32_t shared_d_ff;     /* Fs: always-on shared expert size, 0 = none */
  int32_t act_dtype;       /* MOE_DTYPE_F32 or MOE_DTYPE_BF16 (activations and expert
                              weights); the router weight and logits are always fp32 */
  int32_t dispatch_mode;   /* MOE_DISPATCH_PACKED: capacity goes to assignments in token
                              order and the send buffer is packed (N*k rows).
                              MOE_DISPATCH_CAPACITY_PADDED (needs capacity_factor > 0):
                              every expert owns C consecutive rows (E*C rows, padding
                              unused), and capacity goes to all first choices in token
                              order, then all second choices, and so on */
} moe_config;

/* Rows of the send buffer (xperm, yperm) and length of perm_src for `cfg`: N*k for
 * MOE_DISPATCH_PACKED, E*C for MOE_DISPATCH_CAPACITY_PADDED.  `rows` is a HOST
 * pointer. */
MOE_API moe_status moe_send_rows(const moe_config* cfg, int64_t* rows);

/* Bytes of workspace that every call below needs for `cfg` (one size serves all
 * calls; a larger workspace is fine).  `bytes` is a HOST pointer.  The workspace is
 * device memory, 256-byte aligned, owned by the caller; its contents on entry do not
 * matter and on exit are unspecified, except for the first int32, a sticky device
 * status word: zero it once after allocating the workspace; a kernel of moe_route
 * or moe_expert_ffn that gives up a bounded internal wait sets it nonzero (that
 * call's outputs are then invalid) and no call clears it.  Read it once the stream
 * has passed the calls of interest.  Calls sharing one workspace must not overlap
 * on the GPU. */
MOE_API moe_status moe_workspace_size(const moe_config* cfg, size_t* bytes);

/* Routing.  Ultralytics glossary "Expert Parallelism", section "How tokens move
 * between GPUs", step 1 (the router scores each token against every expert and keeps
 * the k best) and step 4 (outputs are weighted by the router scores); section "Load
 * balancing and capacity" (a per-expert bias added to the scores changes only which
 * experts are selected; each token reaches experts on at most 4 of 8 nodes).
 *
 *   x         [N, d]  act_dtype   hidden states
 *   w_router  [E, d]  fp32        router weight (nn.Linear layout)
 *   b_router  [E]     fp32        router bias, or NULL
 *   sel_bias  [E]     fp32        selection-only bias (sigmoid scoring), or NULL
 *   logits    [N, E]  fp32        out: x . w_router^T + b_router (fp32-accurate)
 *   topk_idx  [N, k]  int32       out: selected experts, best first
 *   topk_w    [N, k]  fp32        out: combine weights
 * Softmax: experts are ranked by logit; weight = softmax probability over all E
 * (renormalised over the k kept if normalize_topk).  Sigmoid: s = S(logit) (a fixed
 * fp32 sigmoid), ranked by s + sel_bias; weight = s (no bias), renormalised over the
 * k kept if normalize_topk.  Group limit: group score = sum of the two best ranking
 * keys in the group; only the topk_groups best groups are eligible.  Ties break
 * toward the lower expert / group index. */
MOE_API moe_status moe_route(const moe_config* cfg, const void* x, const float* w_router,
                     const float* b_router, const float* sel_bias, float* logits,
                     int32_t* topk_idx, float* topk_w, void* workspace,
                     size_t workspace_bytes, void* stream);

/* Dispatch.  Same page, step 2 (each token's hidden state goes to the rank holding
 * its expert) and the page's counting example (assignments per expert and per
 * device); section "Load balancing and capacity" (capacity factor: an expert takes
 * at most cf times its even share, overflow skips that expert); bowenzhou.top
 * "专家并行", exercise 2 (each expert's buffer is reserved at the mean times 1.25:
 * the capacity-padded layout).  Deterministic: assignments a = t*k + j compete in
 * token order (packed) or choice-major order (padded).
 *
 *   topk_idx      [N, k]     int32      from moe_route
 *   x             [N, d]     act_dtype  hidden states
 *   xperm         [S, d]     act_dtype  out: send buffer (S = moe_send_rows): packed,
 *                                       rows [0, num_kept) written, ordered by rank, then
 *                                       expert, then priority; padded, expert e's kept rows
 *                                       at expert_start[e] + [0, kept_counts[e])
 *   expert_counts [E]        int32      out: routed assignments per expert (pre-cap)
 *   kept_counts   [E]        int32      out: min(count, C)
 *   expert_start  [E]        int32      out: first xperm row of each expert
 *   rank_counts   [R]        int32      out: kept rows per logical rank
 *   rank_offsets  [R + 1]    int32      out: exclusive prefix of rank_counts
 *   slot_of       [N*k]      int32      out: xperm row of assignment a, -1 if dropped
 *   perm_src      [S]        int32      out: assignment held by xperm row s, -1 for a row
 *                                       holding none
 *   num_kept      [1]        int32      out: assignments kept (rows written to xperm)
 * xperm may be NULL to compute the routing tables only (x is then ignored). */
MOE_API moe_status moe_dispatch(const moe_config* cfg, const int32_t* topk_idx, const void* x,
                        void* xperm, int32_t* expert_counts, int32_t* kept_counts,
                        int32_t* expert_start, int32_t* rank_counts, int32_t* rank_offsets,
                        int32_t* slot_of, int32_t* perm_src, int32_t* num_kept,
                        void* workspace, size_t workspace_bytes, void* stream);

/* Dispatch without any device allocation by the caller.  The pages have no
 * counterpart to this call; it exists for callers that cannot call cudaMalloc or
 * own a workspace -- for example a runtime whose memory is planned ahead of time by
 * an allocator it does not control, or code on a path where an allocation (which may
 * synchronise the device) is not allowed.  Same arguments, results and ordering as
 * moe_dispatch, minus the workspace: its scratch (a per-chunk expert histogram of
 * ceil(N*k / 2048) * num_experts int32) lives in a static device array of 65536
 * int32 (256 KiB) inside the library, which every GPU that loads the library keeps
 * until the process exits.  Larger layers are rejected with MOE_ERR_WORKSPACE (use
 * moe_dispatch).  Every call looks up the array's device address with the current
 * device (a host-side query, so after a device reset the next call uses the new
 * context's copy of the array); the first call on a device may load the library's
 * device code there, so make it before any stream capture.  All calls share the one
 * array: calls that overlap on the GPU (on different streams) race and give wrong
 * results.  Leftover contents from an earlier call are never read, so nothing needs
 * clearing.  Allocates nothing. */
MOE_API moe_status moe_dispatch_noalloc(const moe_config* cfg, const int32_t* topk_idx,
                                        const void* x, void* xperm, int32_t* expert_counts,
                                        int32_t* kept_counts, int32_t* expert_start,
                                        int32_t* rank_counts, int32_t* rank_offsets,
                                        int32_t* slot_of, int32_t* perm_src, int32_t* num_kept,
                                        void* stream);

/* Expert compute.  Same page, step 3 (each rank runs its local experts on the
 * tokens it received); fudan-mlsys-cn chapter 10, section 10.5 (a shared expert sees
 * every token).  Each expert is a SwiGLU feed-forward block:
 *   h = silu(X Wg^T) * (X Wu^T),  Y = h Wd^T
 *
 *   xperm          [S, d]         act_dtype  from moe_dispatch (S = moe_send_rows)
 *   expert_start   [E], kept_counts [E]  int32  from moe_dispatch (read on device)
 *   w_gate_up      [E, 2F, d]     act_dtype  rows 0..F-1 gate Wg, F..2F-1 up Wu
 *   w_down         [E, d, F]      act_dtype  Wd
 *   x              [N, d]         act_dtype  input of the shared expert (NULL if none)
 *   shared_gate_up [2Fs, d], shared_down [d, Fs]  act_dtype, NULL if shared_d_ff == 0
 *   yperm          [S, d]         act_dtype  out: the kept rows written
 *   yshared        [N, d]         act_dtype  out: shared expert output (NULL if none)
 * bf16: tensor-core products with fp32 accumulation; h is rounded to bf16.
 * fp32: fp32 products and accumulation. */
MOE_API moe_status moe_expert_ffn(const moe_config* cfg, const void* xperm, const int32_t* expert_start,
                          const int32_t* kept_counts, const void* w_gate_up, const void* w_down,
                          const void* x, const void* shared_gate_up, const void* shared_down,
                          void* yperm, void* yshared, void* workspace, size_t workspace_bytes,
                          void* stream);

/* Self-test of the device-side failure handling (the pages have no counterpart).
 * Same arguments and validation as moe_expert_ffn with bf16 activations, but it
 * always runs the prefill tensor-core kernels and makes CTA 0 of the first GEMM arm
 * one pipeline slot whose data is never loaded.  That CTA's bounded wait (about 2 s)
 * runs out, it records a nonzero code in the workspace status word, waits (bounded)
 * for its own copies and MMAs, frees its tensor memory and exits; every other CTA
 * completes normally and the CUDA context stays usable.  Outputs are invalid.
 * Returns MOE_ERR_UNSUPPORTED for fp32 layers. */
MOE_API moe_status moe_selftest_ffn_stall(const moe_config* cfg, const void* xperm,
                                          const int32_t* expert_start, const int32_t* kept_counts,
                                          const void* w_gate_up, const void* w_down,
                                          const void* x, const void* shared_gate_up,
                                          const void* shared_down, void* yperm, void* yshared,
                                          void* workspace, size_t workspace_bytes, void* stream);

/* Combine.  Same page, step 4 (outputs return to token order, weighted by the router
 * scores and summed); section "Load balancing and capacity" (a skipped token passes
 * through the residual connection unchanged).
 *   out[t] = residual[t] + yshared[t] + sum_{j kept} topk_w[t,j] * yperm[slot_of[t,j]]
 * summed in fp32 in the order written (j ascending), rounded once to act_dtype.  A
 * token with no kept choice and no shared expert gets out[t] == residual[t] exactly.
 *   yperm [S, d], slot_of [N*k], topk_w [N, k], residual [N, d] or NULL,
 *   yshared [N, d] or NULL, out [N, d]. */
MOE_API moe_status moe_combine(const moe_config* cfg, const void* yperm, const int32_t* slot_of,
                       const float* topk_w, const void* residual, const void* yshared,
                       void* out, void* stream);

/* Bias-based balancing.  Same page, section "Load balancing and capacity": after a
 * step, lower the selection bias of overloaded experts and raise it for underloaded
 * ones.  For each expert e (fp32, in place):
 *   sel_bias[e] -= step  if expert_counts[e] * E > N * k   (above the mean load)
 *   sel_bias[e] += step  if expert_counts[e] * E < N * k
 * equal load leaves it unchanged.  expert_counts [E] int32 (from moe_dispatch),
 * sel_bias [E] fp32. */
MOE_API moe_status moe_bias_update(const moe_config* cfg, const int32_t* expert_counts, float* sel_bias,
                           float step, void* stream);

/* ---- INT8 all-to-all payload ------------------------------------------------
 * bowenzhou.top note "专家并行", section "深入推导：all-to-all 通信模型与 DeepSeek-V3
 * 的 EP 配置" (DeepSeek-V3's two-level EP): INT8-quantised communication halves the
 * all-to-all traffic again.  The pages fix no format; this library's format is
 * symmetric with one fp32 scale per row:
 *   s   = max_i |v_i| / 127                (fp32 divide)
 *   r   = 1 / s                            (fp32 divide, once per row)
 *   q_i = rint(v_i * r), clamped to +-127   (fp32 multiply, round half to even)
 *   a row of zeros has s = 0 and all q = 0
 *   received value = (float)q_i * s         (one fp32 multiply, then rounded once to
 *                                           act_dtype)
 * A row then travels as `hidden` int8 bytes plus one fp32 scale.  Rows must be
 * finite.  The four calls below replace moe_dispatch's permute and moe_combine on a
 * path whose send and return buffers hold this format:
 *   moe_dispatch_q8 -> moe_dequant_rows -> moe_expert_ffn -> moe_quant_rows ->
 *   moe_combine_q8.
 * Send-buffer rows: S = moe_send_rows(cfg); a row holds an assignment iff
 * perm_src[row] >= 0 (from moe_dispatch_q8); rows with perm_src < 0 are neither read
 * nor written. */

/* moe_dispatch with an INT8 send buffer: the same counts, capacity and slot tables
 * (every int32 output identical to moe_dispatch's), and instead of xperm
 *   xperm_q [S, hidden] int8   codes of the kept tokens' rows, 16-byte aligned
 *   xscale  [S]         fp32   their scales
 * Each token row is quantised once and written to every slot it was kept in. */
MOE_API moe_status moe_dispatch_q8(const moe_config* cfg, const int32_t* topk_idx, const void* x,
                                   int8_t* xperm_q, float* xscale, int32_t* expert_counts,
                                   int32_t* kept_counts, int32_t* expert_start,
                                   int32_t* rank_counts, int32_t* rank_offsets, int32_t* slot_of,
                                   int32_t* perm_src, int32_t* num_kept, void* workspace,
                                   size_t workspace_bytes, void* stream);

/* Quantise the send-buffer rows that hold an assignment (the expert side of the
 * return trip): rows [S, hidden] act_dtype -> q [S, hidden] int8 (16-byte aligned),
 * scale [S] fp32. */
MOE_API moe_status moe_quant_rows(const moe_config* cfg, const void* rows, const int32_t* perm_src,
                                  int8_t* q, float* scale, void* stream);

/* Receiver side: rows[r, i] = (float)q[r, i] * scale[r], stored as act_dtype, for the
 * send-buffer rows that hold an assignment.  q [S, hidden] int8, scale [S] fp32,
 * rows [S, hidden] act_dtype (16-byte aligned). */
MOE_API moe_status moe_dequant_rows(const moe_config* cfg, const int8_t* q, const float* scale,
                                    const int32_t* perm_src, void* rows, void* stream);

/* moe_combine reading an INT8 return payload: expert output element = (float)q * s
 * of its slot's row (fp32 multiply), then the same fp32 sum as moe_combine:
 *   out[t] = residual[t] + yshared[t] + sum_{j kept, ascending} topk_w[t,j] * y_j.
 * yperm_q [S, hidden] int8 (16-byte aligned), yscale [S] fp32; the other arguments as
 * in moe_combine. */
MOE_API moe_status moe_combine_q8(const moe_config* cfg, const int8_t* yperm_q, const float* yscale,
                                  const int32_t* slot_of, const float* topk_w, const void* residual,
                                  const void* yshared, void* out, void* stream);

/* ---- Backward pass ----------------------------------------------------------
 * Gradients of the layer output (the forward calls above, bias update aside) for a
 * FIXED selection: the top-k choice, capacity drops and group limit are piecewise
 * constant in the inputs and pass no gradient; the selection-only bias gets none (the
 * sign rule of moe_bias_update moves it).  With dout = dL/dout [N, hidden] act_dtype:
 *   moe_combine_backward    dyperm, dtopk_w
 *   moe_expert_ffn_backward dxperm, dx_shared, every expert weight gradient
 *   moe_route_backward      dlogits, dx_router, dw_router, db_router
 *   moe_dispatch_backward   dx = dout + dx_shared + dx_router + sum_j dxperm[slot_of]
 * The forward's own buffers (logits, topk_idx, topk_w, slot_of, expert_start,
 * kept_counts, xperm, yperm) are the inputs; they must be those of the same call. */

/* Bytes of the activations a training forward keeps for the backward:
 * h [S, F] + [N, Fs], then g|u [S, 2F] + [N, 2Fs], bf16 (S = moe_send_rows). */
MOE_API moe_status moe_saved_size(const moe_config* cfg, size_t* bytes);

/* moe_expert_ffn for training: the same outputs, and the SwiGLU activations h and the
 * gate/up pre-activations g|u of every row written to `saved` (moe_saved_size bytes,
 * 16-byte aligned), so that moe_expert_ffn_backward need not recompute them.  bf16
 * layers only (fp32: MOE_ERR_UNSUPPORTED); always the prefill tensor-core kernels. */
MOE_API moe_status moe_expert_ffn_save(const moe_config* cfg, const void* xperm,
                                       const int32_t* expert_start, const int32_t* kept_counts,
                                       const void* w_gate_up, const void* w_down, const void* x,
                                       const void* shared_gate_up, const void* shared_down,
                                       void* yperm, void* yshared, void* saved, size_t saved_bytes,
                                       void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of the workspace moe_expert_ffn_backward and moe_route_backward need (one size
 * serves both): the status word, then the gate/up and h activations and [dg | du]
 * (bf16, in the send-buffer layout) or the router weight gradient's split logit
 * gradient and bias partial sums, whichever is larger.  `bytes` is a HOST pointer. */
MOE_API moe_status moe_backward_workspace_size(const moe_config* cfg, size_t* bytes);

/* Combine backward.  Same page, step 4, differentiated: for each kept choice,
 *   dyperm[slot_of[t,j]] = topk_w[t,j] * dout[t]          (act_dtype, one rounding)
 *   dtopk_w[t,j]         = sum_i dout[t,i] * yperm[slot,i] (fp32; 0 for dropped j)
 * dout [N, hidden], yperm / dyperm [S, hidden] act_dtype (16-byte aligned); slot_of
 * [N*k] int32; topk_w, dtopk_w [N, k] fp32.  Rows of dyperm that hold no assignment
 * are not written. */
MOE_API moe_status moe_combine_backward(const moe_config* cfg, const void* dout, const void* yperm,
                                        const int32_t* slot_of, const float* topk_w, void* dyperm,
                                        float* dtopk_w, void* stream);

/* Expert FFN backward (bf16 layers; fp32 returns MOE_ERR_UNSUPPORTED).  For each
 * send-buffer row of expert e (and each token for the shared expert), with
 * g = Wg x, u = Wu x, h = silu(g) * u, y = Wd h:
 *   dh = Wd^T dy;  dg = dh * u * silu'(g);  du = dh * silu(g)
 *   dx = Wg^T dg + Wu^T du;  dWd[e] += dy h^T;  dWg[e] += dg x^T;  dWu[e] += du x^T
 * g, u and h are recomputed from xperm (tensor cores, fp32 accumulation; g, u, h and
 * [dg | du] rounded to bf16).
 *   xperm, expert_start, kept_counts, w_gate_up, w_down, x, shared_*  as moe_expert_ffn
 *   dyperm [S, hidden]  from moe_combine_backward;  dout [N, hidden] (the shared
 *                       expert's dy; NULL without a shared expert)
 *   dxperm [S, hidden]  out: input gradient of the kept rows
 *   dx_shared [N, hidden] out (NULL without a shared expert)
 *   dw_gate_up [E, 2F, hidden], dw_down [E, hidden, F]  out (experts with no kept rows
 *                       get zeros); dshared_gate_up [2Fs, hidden], dshared_down
 *                       [hidden, Fs] out (NULL without a shared expert)
 *   saved               the activations moe_expert_ffn_save kept in the forward of the
 *                       same layer call, or NULL to recompute g, u and h here
 *   workspace           moe_backward_workspace_size bytes, 256-byte aligned; its
 *                       first int32 is a sticky status word (caller zeroes it; nonzero
 *                       if a kernel gave up a bounded wait). */
MOE_API moe_status moe_expert_ffn_backward(const moe_config* cfg, const void* xperm,
                                           const int32_t* expert_start, const int32_t* kept_counts,
                                           const void* w_gate_up, const void* w_down, const void* x,
                                           const void* shared_gate_up, const void* shared_down,
                                           const void* dyperm, const void* dout, void* dxperm,
                                           void* dx_shared, void* dw_gate_up, void* dw_down,
                                           void* dshared_gate_up, void* dshared_down,
                                           const void* saved, void* workspace,
                                           size_t workspace_bytes, void* stream);

/* Router backward.  The combine weights as functions of the logits (moe_route):
 *   softmax, renormalised:   dl_j = w_j (dw_j - sum_i w_i dw_i) on the selection, 0 off it
 *   softmax, unnormalised:   dl_e = p_e (dw_e - sum_j w_j dw_j), dw_e = 0 off the selection
 *   sigmoid, renormalised:   dl_j = s_j (1 - s_j) (dw_j - sum_i w_i dw_i) / sum_sel s
 *   sigmoid, unnormalised:   dl_j = s_j (1 - s_j) dw_j
 * (s = the selection sigmoid of moe_route, p = softmax over all experts), then
 *   dx_router = dl . w_router  [N, hidden] fp32 (NULL to skip)
 *   dw_router = dl^T x [E, hidden] fp32 (16-byte aligned) and db_router = sum_t dl
 *   [E] fp32 (both or neither NULL)
 * logits [N, E] fp32 and topk_idx [N, k] from moe_route; dtopk_w from
 * moe_combine_backward; dlogits [N, E] fp32 out.  workspace: the backward workspace
 * (moe_backward_workspace_size bytes, 256-byte aligned; may be NULL when dw_router is
 * NULL); its contents are not kept between calls, its first int32 is the device status
 * word (nonzero if a kernel gave up a bounded wait).  With bf16 activations and at least
 * 128 tokens dw_router is one tensor-core GEMM over an exact three-term bf16 split of dl
 * (fp32 accumulation); db_router and the fp32 layers' dw_router are fixed-order fp32 sums
 * over the tokens. */
MOE_API moe_status moe_route_backward(const moe_config* cfg, const void* x, const float* w_router,
                                      const float* logits, const int32_t* topk_idx,
                                      const float* dtopk_w, float* dlogits, float* dx_router,
                                      float* dw_router, float* db_router, void* workspace,
                                      size_t workspace_bytes, void* stream);

/* Dispatch backward: the permute's transpose plus the residual, shared-expert and
 * router paths, summed in fp32 and rounded once:
 *   dx[t] = dout[t] + dx_shared[t] + dx_router[t] + sum_{j kept, ascending} dxperm[slot_of[t,j]]
 * dxperm [S, hidden], dout / dx_shared (nullable) / dx [N, hidden] act_dtype;
 * dx_router [N, hidden] fp32 (nullable). */
MOE_API moe_status moe_dispatch_backward(const moe_config* cfg, const void* dxperm,
                                         const int32_t* slot_of, const void* dout,
                                         const void* dx_shared, const float* dx_router, void* dx,
                                         void* stream);

/* Static, NUL-terminated description of a status code (host pointer). */
MOE_API const char* moe_status_string(moe_status status);

#ifdef __cplusplus
}
#endif

#endif /* MOE_B300_H */
