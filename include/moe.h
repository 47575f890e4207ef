/*
 * moe.h -- C ABI of libmoe.so, a B300 (sm_103a) single-GPU Mixture-of-Experts
 * layer forward.
 *
 * The operations and their notation come from "MoE 与专家并行"
 * (hs-black.github.io/posts/scaling-moe):
 *   - 从稠密 FFN 到 MoE: SwiGLU expert FFN(u) = W_down (SiLU(W_gate u) ⊙ W_up u)
 *     and the layer output h'_t = u_t + sum_i g_{i,t} FFN_i(u_t);
 *   - 路由器：打分、top-k、加权求和: H = U W_r, scores, top-k, gates, the noisy
 *     top-k router, and the single-GPU shapes listing (permute by expert,
 *     grouped FFN, index_add back into token order);
 *   - softmax 门控还是 sigmoid 门控: softmax / sigmoid scoring, with or without
 *     renormalisation over the selected experts;
 *   - 专家容量与丢 token: capacity C = ceil(CF * T * k / E), slots filled in
 *     token order with every token's first choice before any second choice,
 *     overflow dropped (the token keeps its residual only);
 *   - 负载均衡辅助损失：推导与梯度: f_i, P_i and E * sum_i f_i P_i (sigmoid P_i
 *     from s_i / sum_j s_j);
 *   - 专家计算：padding、block-sparse 与 grouped GEMM: one grouped GEMM over the
 *     variable-length expert segments, gate and up fused into one [h, 2 d_e]
 *     product, then SiLU * up, then down.
 * The capacity formula also appears, for top-1, in the router / expert-
 * parallel tutorial at aissn.com/133.html (section 工程难点 2).
 *
 * Conventions shared by every entry point
 *   Notation: T tokens, h hidden size, E experts, k experts per token, d_e
 *   expert intermediate size, A = number of kept (token, expert) pairs.
 *   Layouts are row-major and dense.  "act dtype" is the config's dtype
 *   (MOE_F32: float, MOE_BF16: bfloat16) for activations and weights; router
 *   logits, gates, scores and statistics are float32.
 *   Memory: every array argument is a DEVICE pointer, 16-byte aligned, owned
 *   by the caller, unless stated otherwise.  The library never allocates,
 *   frees or synchronises (moe_get_device_status excepted) and keeps no
 *   global state apart from the static histogram of moe_dispatch_noalloc;
 *   all work is enqueued on the caller's stream in order.
 *   Workspace: `ws` is caller-owned device scratch of moe_workspace_size()
 *   bytes, 256-byte aligned, zero-filled once after allocation.  It carries
 *   the device status word and the per-block partial sums one stage hands to
 *   the next, so the stage calls of one layer must use the same `ws`, and
 *   calls that share a `ws` must not overlap on the GPU.
 *   Errors: argument and shape errors return MOE_ERR_INVALID_ARG or
 *   MOE_ERR_UNSUPPORTED before anything is enqueued; a failed launch returns
 *   MOE_ERR_CUDA; errors only the device can see (an expert id out of range,
 *   inconsistent expert offsets, a pipeline wait that timed out) set the
 *   status word in `ws` and the offending element is skipped -- read it with
 *   moe_get_device_status().  moe_last_error() gives a one-line message for
 *   the last non-OK return of the calling host thread.
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t; /* a cudaStream_t; NULL = legacy default stream */

typedef enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,   /* null / misaligned pointer, bad shape, k > E, ... */
  MOE_ERR_UNSUPPORTED = 2,   /* valid MoE config outside the supported ranges */
  MOE_ERR_CUDA = 3,          /* a CUDA call or launch failed */
  MOE_ERR_DEVICE = 4         /* the device status word is set (moe_get_device_status) */
} moe_status;

typedef enum moe_score_fn { MOE_SCORE_SOFTMAX = 0, MOE_SCORE_SIGMOID = 1 } moe_score_fn;
typedef enum moe_dtype { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype;
typedef enum moe_priority {
  MOE_PRIORITY_CHOICE_MAJOR = 0, /* all first choices (tokens in order), then all second choices, ... */
  MOE_PRIORITY_TOKEN_MAJOR = 1   /* token by token, a token's choices in rank order */
} moe_priority;

/* Device status codes written into the workspace status word. */
enum {
  MOE_DEV_OK = 0,
  MOE_DEV_BAD_EXPERT_ID = 1,  /* moe_dispatch saw idx outside [0, E); that pair was dropped */
  MOE_DEV_TIMEOUT = 2,        /* a pipeline wait in the grouped GEMM gave up; outputs are invalid */
  MOE_DEV_BAD_ROW = 3,        /* moe_combine saw slot_row outside [-1, T*k); that pair was skipped */
  MOE_DEV_BAD_OFFSETS = 4     /* moe_expert_ffn saw non-monotone or out-of-range offsets; nothing written */
};

typedef struct moe_config {
  int64_t T;              /* tokens, >= 0; T * k < 2^31 */
  int32_t h;              /* hidden size, >= 1, multiple of 8 */
  int32_t E;              /* experts, 1..1024 */
  int32_t k;              /* experts per token, 1..min(E, 16) */
  int32_t d_e;            /* expert intermediate size, >= 1, multiple of 8 */
  float capacity_factor;  /* CF; <= 0 means no capacity limit (C = T) */
  int32_t capacity;       /* > 0 overrides the formula with this C */
  int32_t score_fn;       /* moe_score_fn */
  int32_t renorm;         /* nonzero: g_j = s_j / sum of the k selected s; zero: g_j = s_j */
  int32_t noisy;          /* nonzero: noisy top-k router (W_noise, eps required) */
  int32_t priority;       /* moe_priority: order in which capacity slots are filled */
  int32_t dtype;          /* moe_dtype of activations and weights */
  int32_t n_shared;       /* shared experts (every token, no router), 0..16; 0 = none */
  int32_t d_shared;       /* their intermediate size (multiple of 8) when n_shared > 0 */
  int32_t n_group;        /* group-limited routing: 0 or 1 = off; else 2..32 equal, contiguous expert
                           * groups (E % n_group == 0), see moe_route */
  int32_t topk_group;     /* groups kept per token when n_group > 1: 1..n_group, k % topk_group == 0,
                           * k <= topk_group * E / n_group */
} moe_config;

/* Library version string, e.g. "moe-b300 0.1 sm_103a". */
const char* moe_version(void);

/* Human-readable name of a status code (static storage). */
const char* moe_status_string(moe_status status);

/* One-line message for the last non-OK return on the calling host thread ("" if none). */
const char* moe_last_error(void);

/* Expert capacity C (host only, no CUDA call).  C = ceil(CF * T * k / E)
 * evaluated exactly on the float32 value of CF; CF <= 0: C = T; cfg->capacity
 * > 0: C = cfg->capacity.  Section 专家容量与丢 token. */
moe_status moe_capacity(const moe_config* cfg, int64_t* C);

/* Bytes of device workspace the calls below need for this config (host only). */
moe_status moe_workspace_size(const moe_config* cfg, size_t* bytes);

/* Router: logits, scores, top-k and gates for every token.
 * Section 路由器：打分、top-k、加权求和 and section softmax 门控还是 sigmoid 门控;
 * the selection bias is section 无辅助损失的负载均衡 (loss-free balancing).
 *   U        [T, h] act dtype         token hidden states
 *   W_r      [h, E] act dtype         router weight (column i = expert i's centroid)
 *   b_r      [E] float32 or NULL      per-expert additive logit bias
 *   sel_bias [E] float32 or NULL      loss-free balancing bias: when given, the top-k is
 *                                     taken on score + sel_bias (score = softmax or sigmoid,
 *                                     float32) while the gates stay the scores; NULL: the
 *                                     top-k is taken on the logits
 *   W_noise  [h, E] act dtype         noisy router only (cfg->noisy), else ignored
 *   eps      [T, E] float32           noisy router only: the N(0,1) draws
 *   logits_in [T, E] float32 or NULL  stage mode: use these final logits as they
 *                                     are (U, W_r, b_r, W_noise, eps ignored)
 *   logits_out [T, E] float32 or NULL receives the final logits
 *                                     H = U W_r + b_r + eps * softplus(U W_noise)
 *   idx      [T, k] int32 out         selected experts, highest logit first, ties
 *                                     to the lower expert id
 *   gate     [T, k] float32 out       g_j (renormalised over the k or not, cfg->renorm)
 * Logits accumulate in float32 from the act-dtype inputs; selection compares
 * the float32 logits.  Also leaves per-block sums of the scores (sigmoid:
 * s_i / sum_j s_j) in `ws` for moe_combine's P_i.
 * Group-limited routing (cfg->n_group > 1; section 设备受限与节点受限路由, node-limited
 * routing with the nodes read as expert groups): group q holds experts
 * [q*E/n_group, (q+1)*E/n_group); each group is scored by the float32 sum of its
 * k/topk_group highest affinities (the score, or score + sel_bias when sel_bias is
 * given); the topk_group best groups are kept (ties to the lower group id), and the
 * top-k above is taken over their experts only. */
moe_status moe_route(const moe_config* cfg, const void* U, const void* W_r, const float* b_r,
                     const float* sel_bias, const void* W_noise, const float* eps,
                     const float* logits_in, float* logits_out, int32_t* idx, float* gate, void* ws,
                     moe_stream_t stream);

/* Bytes of the packed router weights of this config (host only, no CUDA call): 2 * N * h with
 * N = E (noisy router: 2E) rounded up to a multiple of 16, when the config's router runs on the
 * tensor cores (bf16 and N <= 256); 0 otherwise (moe_route then reads W_r as it is). */
moe_status moe_router_pack_size(const moe_config* cfg, size_t* bytes);

/* One-time packing of the router weights for the tensor-core router (section 路由器：打分、
 * top-k、加权求和: H = U W_r, and the noise projection U W_noise of the noisy router).
 *   W_r      [h, E] bf16               as for moe_route
 *   W_noise  [h, E] bf16               noisy router only (cfg->noisy), else ignored
 *   W_r_packed [N, h] bf16 out         caller-owned, moe_router_pack_size() bytes, 16-byte
 *                                      aligned: row n < E is column n of W_r, row E + n (noisy)
 *                                      column n of W_noise, the remaining rows zero
 * Run it once after the weights change; moe_route_packed and moe_layer_forward (args->W_r_packed)
 * then skip the per-call packing.  MOE_ERR_UNSUPPORTED when moe_router_pack_size() is 0. */
moe_status moe_pack_router(const moe_config* cfg, const void* W_r, const void* W_noise, void* W_r_packed,
                           moe_stream_t stream);

/* moe_route from packed router weights (moe_pack_router): the same results as moe_route with
 * the weights that were packed, bit for bit.  No stage mode (logits_in).  One kernel: the
 * router GEMM on the tensor cores with the scores, top-k, gates and the P / z partials in its
 * epilogue. */
moe_status moe_route_packed(const moe_config* cfg, const void* U, const void* W_r_packed, const float* b_r,
                            const float* sel_bias, const float* eps, float* logits_out, int32_t* idx,
                            float* gate, void* ws, moe_stream_t stream);

/* One step of the loss-free balancing bias (section 无辅助损失的负载均衡):
 *   bias[i] += u * sign(mean(counts_routed) - counts_routed[i]),
 * the sign taken exactly on the integer counts.  counts_routed [E] int32 (e.g. from
 * moe_dispatch), bias [E] float32 updated in place; one small kernel on `stream`. */
moe_status moe_balance_bias_update(const moe_config* cfg, const int32_t* counts_routed, float u,
                                   float* bias, moe_stream_t stream);

/* Capacity-limited dispatch: per-expert histogram, prefix sums, slots, drop
 * mask, offsets, and the row copy X[row] = U[token].
 * Section 专家容量与丢 token and the permute of the shapes listing.
 *   U        [T, h] act dtype
 *   idx      [T, k] int32             from moe_route (any values; ids outside
 *                                     [0, E) set MOE_DEV_BAD_EXPERT_ID and drop)
 *   counts_routed [E] int32 out       pairs that chose expert e (before drops)
 *   counts_kept   [E] int32 out       min(counts_routed[e], C)
 *   offsets  [E+1] int32 out          exclusive prefix sum of counts_kept; A = offsets[E]
 *   slot_row [T*k] int32 out          row of pair (t, j) = t*k + j in X, or -1 if dropped
 *   row_token [T*k] int32 out         token of each row; only the first A are written
 *   X        [T*k, h] act dtype out   expert inputs, segment e = rows offsets[e]..offsets[e+1],
 *                                     in slot (priority) order; only the first A rows written
 *   n_dropped [1] int64 out           T*k - A
 * All of it is integer work and bit-exact: the n-th pair (in cfg->priority
 * order) that chose expert e takes slot n and is kept iff n < C.
 * X may be NULL: then only the routing metadata is written (for moe_expert_ffn_gather). */
moe_status moe_dispatch(const moe_config* cfg, const void* U, const int32_t* idx,
                        int32_t* counts_routed, int32_t* counts_kept, int32_t* offsets,
                        int32_t* slot_row, int32_t* row_token, void* X, int64_t* n_dropped,
                        void* ws, moe_stream_t stream);

/* moe_dispatch for callers that cannot allocate device memory.
 *
 * The pages have no counterpart to this call; it is a deployment variant of
 * moe_dispatch.  Some callers are not allowed to allocate device memory at
 * all: an engine that reserves its whole device memory up front and forbids
 * allocation once it is serving, a plugin whose host framework hands it tensors
 * but offers no scratch allocator, or code that must not pay for an allocation
 * (nor risk one failing) on the hot path.  This entry point needs no `ws`: the
 * only scratch dispatch uses, the per-chunk expert histogram, sits in a
 * file-scope device array inside libmoe of MOE_NOALLOC_HIST_MAX int32 (4 MiB).
 * Every GPU that loads the library keeps that array until the process exits.
 * The call makes no cudaMalloc or cudaFree and calls no allocating routine.
 *
 *   Arguments and results are those of moe_dispatch, bit for bit, except:
 *   status   [1] int32 device out or NULL: zeroed by the call, then set to a
 *            MOE_DEV_* code (an expert id outside [0, E) -> MOE_DEV_BAD_EXPERT_ID,
 *            that pair dropped).  NULL: device-side errors are not reported.
 *   Size limit: ceil(T*k / 4096) * E <= MOE_NOALLOC_HIST_MAX, else
 *            MOE_ERR_UNSUPPORTED before anything is enqueued (for E = 1024 that
 *            is T*k <= 4 Mi pairs).
 *   Shared scratch: every call on a device uses the same array and leaves its
 *            contents behind; each call rewrites all it reads, so no clearing is
 *            needed between calls.  Calls whose work overlaps on the GPU (on
 *            streams with no ordering between them) race on the array and give
 *            wrong results: order them on one stream or with events.
 *   First call per device: it looks up the array's device address on the
 *            current device (cudaGetSymbolAddress) and caches it with the id of
 *            the current context.  Make that first call before any stream
 *            capture begins.  A call from another context (after
 *            cudaDeviceReset, or with a context the caller made current) looks
 *            the address up again; make such a call outside stream capture too.
 *   The current device must be the device that `stream` and every pointer
 *   belong to. */
#define MOE_NOALLOC_HIST_MAX (1 << 20)
moe_status moe_dispatch_noalloc(const moe_config* cfg, const void* U, const int32_t* idx,
                                int32_t* counts_routed, int32_t* counts_kept, int32_t* offsets,
                                int32_t* slot_row, int32_t* row_token, void* X, int64_t* n_dropped,
                                int32_t* status, moe_stream_t stream);

/* Grouped SwiGLU expert FFN over the expert segments of X.
 * Section 从稠密 FFN 到 MoE (the expert) and section 专家计算：padding、block-sparse
 * 与 grouped GEMM (one grouped GEMM for gate|up, SiLU * up, one for down).
 *   X        [T*k, h] act dtype       rows 0..A-1 valid (from moe_dispatch)
 *   offsets  [E+1] int32              expert segments (device-resident; no host read)
 *   W_gate   [E, d_e, h] act dtype    W_gate[e] in R^{d_e x h}
 *   W_up     [E, d_e, h] act dtype
 *   W_down   [E, h, d_e] act dtype    W_down[e] in R^{h x d_e}
 *   act      [T*k, d_e] act dtype out SiLU(X W_gate^T) * (X W_up^T), rounded to act dtype
 *   Y        [T*k, h] act dtype out   act W_down^T, rounded to act dtype
 * Accumulation is float32.  bf16 runs on the tcgen05 tensor cores (operands
 * staged by TMA, accumulators in tensor memory); float32 on the CUDA cores.
 * Rows >= A of act and Y are not written. */
moe_status moe_expert_ffn(const moe_config* cfg, const void* X, const int32_t* offsets,
                          const void* W_gate, const void* W_up, const void* W_down,
                          void* act, void* Y, void* ws, moe_stream_t stream);

/* moe_expert_ffn with the dispatch's row copy fused into the first GEMM (bf16 configs; section
 * 专家计算：padding、block-sparse 与 grouped GEMM, and the permute of the shapes listing):
 *   U        [T, h] bf16               token rows
 *   row_token [T*k] int32              from moe_dispatch: row r of the expert input is U[row_token[r]]
 *                                      (ids outside [0, T) read row 0 and set MOE_DEV_BAD_ROW)
 *   offsets, W_gate, W_up, W_down, act, Y   as in moe_expert_ffn
 * No X is read or written: the first GEMM's producer loads each 128 x 64 A tile straight from the
 * token rows of U (32 four-row TMA gathers into the swizzled layout of a tiled load).  act and Y
 * are bit-identical to moe_expert_ffn on X[r] = U[row_token[r]].  It is slower than the
 * materialised X when the first GEMM has many column tiles (each re-reads the gathered rows). */
moe_status moe_expert_ffn_gather(const moe_config* cfg, const void* U, const int32_t* row_token,
                                 const int32_t* offsets, const void* W_gate, const void* W_up,
                                 const void* W_down, void* act, void* Y, void* ws, moe_stream_t stream);

/* Shared experts (section 细粒度专家与共享专家, the shared-expert isolation of
 * DeepSeekMoE / V3): cfg->n_shared SwiGLU experts that every token passes
 * through, outside the router.
 *   U            [T, h] act dtype
 *   W_gate_shared, W_up_shared [n_shared, d_shared, h] act dtype
 *   W_down_shared               [n_shared, h, d_shared] act dtype
 *   act_shared   [n_shared, T, d_shared] act dtype out   SiLU(G) * Up of each shared expert
 *   Y_shared     [n_shared, T, h] act dtype out   FFN_s(u_t), rounded to act dtype
 * The same grouped kernels as moe_expert_ffn, with one segment of all T rows. */
moe_status moe_shared_ffn(const moe_config* cfg, const void* U, const void* W_gate_shared,
                          const void* W_up_shared, const void* W_down_shared, void* act_shared,
                          void* Y_shared, void* ws, moe_stream_t stream);

/* Combine and load statistics.
 * Section 从稠密 FFN 到 MoE (h'_t = u_t + sum g FFN), the index_add of the
 * shapes listing, section 负载均衡辅助损失：推导与梯度 (f, P, aux) and section
 * Router z-loss 与数值稳定 (z_loss).
 *   U        [T, h] act dtype
 *   Y        [T*k, h] act dtype       from moe_expert_ffn
 *   Y_shared [n_shared, T, h] or NULL from moe_shared_ffn (ignored when cfg->n_shared is 0)
 *   slot_row [T*k] int32, gate [T, k] float32, counts_routed [E] int32
 *   out      [T, h] act dtype out     u_t + sum_s Y_shared[s, t] + sum over kept j (ascending)
 *                                     of gate[t,j] * Y[row], float32 accumulation, one rounding
 *   f        [E] float32 out          counts_routed[i] / (T*k)
 *   P        [E] float32 out          (1/T) sum_t s_{i,t}, from the partial sums moe_route
 *                                     left in this `ws`
 *   aux      [1] float32 out          E * sum_i f_i P_i (the balance loss with alpha = 1)
 *   z_loss   [1] float32 out or NULL  (1/T) sum_t (log sum_j exp H_{t,j})^2 over the final
 *                                     router logits (the router z-loss with c_z = 1), from the
 *                                     per-block sums moe_route left in this `ws` */
moe_status moe_combine(const moe_config* cfg, const void* U, const void* Y, const void* Y_shared,
                       const int32_t* slot_row, const float* gate, const int32_t* counts_routed,
                       void* out, float* f, float* P, float* aux, float* z_loss, void* ws,
                       moe_stream_t stream);

/* ---- Backward of the router side (section 路由器：打分、top-k、加权求和, how the
 * router learns: dL/dg_{i,t} = delta_t^T FFN_i(u_t); section 负载均衡辅助损失：
 * 推导与梯度, 梯度往哪推; section Router z-loss 与数值稳定). */

/* Backward of moe_combine for the upstream gradient dO = dL/dout:
 *   dO       [T, h] act dtype
 *   Y, slot_row, gate                 as given to moe_combine
 *   d_gate   [T, k] float32 out       dO_t . Y[row] for kept pairs (float32 sum), 0 if dropped
 *   dY       [T*k, h] act dtype out   row r of a kept pair (t, j): gate[t,j] * dO_t, rounded
 *                                     once; rows of dropped pairs and rows >= A untouched */
moe_status moe_combine_backward(const moe_config* cfg, const void* dO, const void* Y,
                                const int32_t* slot_row, const float* gate, float* d_gate, void* dY,
                                void* ws, moe_stream_t stream);

/* Gradient of the loss with respect to the router logits H (the top-k set held fixed):
 *   dH = (dg/dH)^T d_gate + w_aux * d(E sum_i f_i P_i)/dH + w_z * dL_z/dH
 *   logits   [T, E] float32           the final logits (moe_route's logits_out)
 *   idx      [T, k] int32, d_gate [T, k] float32 (from moe_combine_backward)
 *   counts_routed [E] int32           for f_i = counts / (T k); may be NULL when w_aux = 0
 *   w_aux, w_z                        weights of the balance loss (alpha) and of the z-loss (c_z)
 *   dH       [T, E] float32 out
 * The gate part follows cfg->score_fn and cfg->renorm (gates from the scores, also under a
 * loss-free selection bias); sigmoid P uses s / sum_j s_j. */
moe_status moe_route_backward(const moe_config* cfg, const float* logits, const int32_t* idx,
                              const float* d_gate, const int32_t* counts_routed, float w_aux,
                              float w_z, float* dH, moe_stream_t stream);

/* ---- Backward of the experts and of the permute (section 专家计算：padding、
 * block-sparse 与 grouped GEMM: the experts' backward is grouped GEMMs too, one
 * group for the input gradients and one for the weight gradients). */

/* Backward of moe_expert_ffn for dY = dL/dY (bf16 configs; float32 returns MOE_ERR_UNSUPPORTED).
 *   X, offsets, W_gate, W_up, W_down  as given to moe_expert_ffn
 *   act      [T*k, d_e] bf16           moe_expert_ffn's act (for dW_down)
 *   dY       [T*k, h] bf16             rows 0..A-1 read (e.g. from moe_combine_backward)
 *   d_act    [T*k, d_e] bf16 out       dY W_down[e]
 *   dG, dUp  [T*k, d_e] bf16 out       d_act * Up * SiLU'(G), d_act * SiLU(G), with G = X W_gate^T
 *                                      and Up = X W_up^T recomputed
 *   dX       [T*k, h] bf16 out         dG W_gate[e] + dUp W_up[e]
 *   dW_gate, dW_up [E, d_e, h] float32 out   dG^T X, dUp^T X over each expert's rows
 *   dW_down  [E, h, d_e] float32 out   dY^T act over each expert's rows (experts with no rows: 0)
 * Rows >= A of the row outputs are not written.  All products run on the tensor cores
 * (bf16 operands, float32 accumulation); the weights are read MN-major where the product
 * contracts over their other dimension. */
moe_status moe_expert_ffn_backward(const moe_config* cfg, const void* X, const int32_t* offsets,
                                   const void* W_gate, const void* W_up, const void* W_down,
                                   const void* act, const void* dY, void* d_act, void* dG, void* dUp,
                                   void* dX, float* dW_gate, float* dW_up, float* dW_down, void* ws,
                                   moe_stream_t stream);

/* Backward of the residual and the permute: dU_t = dO_t + sum over kept j (choice order) of
 * dX[row(t, j)], float32 accumulation, one rounding.  dO [T, h], dX [T*k, h], slot_row [T*k],
 * dU [T, h] out (act dtype).  The router's contribution dH W_r^T is not included. */
moe_status moe_dispatch_backward(const moe_config* cfg, const void* dO, const void* dX,
                                 const int32_t* slot_row, void* dU, void* ws, moe_stream_t stream);

/* Backward of the router linear H = U W_r + b_r (+ eps * softplus(U W_noise)), bf16 configs:
 *   dH       [T, E] float32           from moe_route_backward
 *   dU_router [T, h] bf16 out         dH W_r^T (+ dN W_noise^T), dN = dH * eps * sigmoid(U W_noise)
 *   dW_r     [h, E] float32 out       U^T dH;   dW_noise [h, E] float32 out (noisy): U^T dN
 *   db_r     [E] float32 out or NULL  sum over tokens of dH
 * The products run on the tensor cores with dH (and dN) rounded to bf16; the noise logits
 * are recomputed. */
moe_status moe_router_input_backward(const moe_config* cfg, const void* U, const void* W_r,
                                     const void* W_noise, const float* eps, const float* dH,
                                     void* dU_router, float* dW_r, float* dW_noise, float* db_r,
                                     void* ws, moe_stream_t stream);

/* Every input and output of one layer forward (pointer meanings as above). */
typedef struct moe_layer_args {
  const void* U; const void* W_r; const float* b_r; const void* W_noise; const float* eps;
  const void* W_gate; const void* W_up; const void* W_down;
  float* logits_out;                          /* NULL: logits are not written */
  int32_t* idx; float* gate;
  int32_t* counts_routed; int32_t* counts_kept; int32_t* offsets;
  int32_t* slot_row; int32_t* row_token; int64_t* n_dropped;
  void* X; void* act; void* Y;
  void* out; float* f; float* P; float* aux;
  float* z_loss;                              /* NULL: the z-loss is not written */
  const float* sel_bias;                      /* NULL: no loss-free selection bias */
  const void* W_gate_shared; const void* W_up_shared; const void* W_down_shared;
  void* act_shared; void* Y_shared;           /* used when cfg->n_shared > 0 */
  const void* W_r_packed;                     /* NULL, or W_r (and W_noise) from moe_pack_router:
                                               * then the router skips its per-call packing */
} moe_layer_args;

/* The whole layer: moe_route, moe_dispatch, moe_expert_ffn, (moe_shared_ffn,)
 * moe_combine in order on `stream`, with no host synchronisation in between.
 * args->X == NULL (bf16 configs): the dispatch copies no rows and the expert FFN runs as
 * moe_expert_ffn_gather, reading the token rows of U directly (the results are identical). */
moe_status moe_layer_forward(const moe_config* cfg, const moe_layer_args* args, void* ws,
                             moe_stream_t stream);

/* ---- FP8 dispatch and up-projection (section 低精度通信) -------------------------------
 * The activations entering the up-projection travel and multiply as FP8 E4M3 codes with one
 * power-of-two scale per row; the down projection, the shared experts and the combine stay bf16.
 * Row rule (all calls below): s = the smallest integer >= -127 with amax(row) <= 448 * 2^s,
 * scale = 2^s (float32, exact), code = E4M3(x * 2^-s) rounded to nearest even.  bf16 configs
 * only, with h % 16 == 0 (MOE_ERR_UNSUPPORTED otherwise). */

/* Quantise rows: src [rows, cols] bf16 -> dst [rows, cols] E4M3 bytes, scale [rows] float32.
 * cols % 8 == 0; src and dst 16- and 8-byte aligned.  For the expert weights: W_gate and W_up
 * as [E * d_e, h] (one scale per output channel), once, before the layer runs. */
moe_status moe_quantize_fp8(int64_t rows, int32_t cols, const void* src, uint8_t* dst, float* scale,
                            moe_stream_t stream);

/* moe_dispatch with FP8 rows: the same routing metadata (bit-exact with moe_dispatch), and
 *   X8       [T*k, h] E4M3 out         X8[row] = codes of U[row_token[row]]
 *   x_scale  [T*k] float32 out         the scale of that token row
 * Each token row is quantised once and copied to its kept slots. */
moe_status moe_dispatch_fp8(const moe_config* cfg, const void* U, const int32_t* idx,
                            int32_t* counts_routed, int32_t* counts_kept, int32_t* offsets,
                            int32_t* slot_row, int32_t* row_token, uint8_t* X8, float* x_scale,
                            int64_t* n_dropped, void* ws, moe_stream_t stream);

/* moe_expert_ffn with the FP8 up-projection:
 *   X8, x_scale                        from moe_dispatch_fp8
 *   W_gate8, W_up8 [E, d_e, h] E4M3    s_gate, s_up [E * d_e] float32: from moe_quantize_fp8
 *   W_down   [E, h, d_e] bf16          act [T*k, d_e] bf16 out, Y [T*k, h] bf16 out
 * G = (X8 W_gate8^T) * x_scale[row] * s_gate[col] (and Up alike) on the tensor cores
 * (kind::f8f6f4, float32 accumulation of exact products), act = SiLU(G) * Up rounded to bf16,
 * Y = act W_down^T as in moe_expert_ffn. */
moe_status moe_expert_ffn_fp8(const moe_config* cfg, const uint8_t* X8, const float* x_scale,
                              const int32_t* offsets, const uint8_t* W_gate8, const uint8_t* W_up8,
                              const float* s_gate, const float* s_up, const void* W_down, void* act,
                              void* Y, void* ws, moe_stream_t stream);

/* The FP8 operands of moe_layer_forward_fp8. */
typedef struct moe_fp8_args {
  uint8_t* X8; float* x_scale;                    /* [T*k, h], [T*k] outputs of the dispatch */
  const uint8_t* W_gate8; const uint8_t* W_up8;   /* [E, d_e, h] */
  const float* s_gate; const float* s_up;         /* [E * d_e] */
} moe_fp8_args;

/* moe_layer_forward with moe_dispatch_fp8 and moe_expert_ffn_fp8 in place of moe_dispatch and
 * moe_expert_ffn (args->X, args->W_gate and args->W_up are not used). */
moe_status moe_layer_forward_fp8(const moe_config* cfg, const moe_layer_args* args,
                                 const moe_fp8_args* fp8, void* ws, moe_stream_t stream);

/* Gradients and scratch of one layer backward (bf16 configs).  Scratch is caller-owned. */
typedef struct moe_layer_grads {
  const void* dO;        /* [T, h]   dL/dout */
  float w_aux, w_z;      /* weights of E*sum f P and of the z-loss in the loss */
  float* d_gate;         /* [T, k] scratch */
  void* dY;              /* [T*k, h] scratch */
  float* dH;             /* [T, E] out: dL/d(router logits) */
  void* d_act; void* dG; void* dUp;   /* [T*k, d_e] scratch */
  void* dX;              /* [T*k, h] scratch */
  void* dU_router;       /* [T, h] scratch */
  void* d_act_shared; void* dG_shared; void* dUp_shared;  /* [T, d_shared] scratch (n_shared > 0) */
  void* dX_shared;       /* [n_shared, T, h] scratch */
  void* dU;              /* [T, h] out: dL/dU */
  float* dW_gate; float* dW_up; float* dW_down;          /* out, float32, shapes of the weights */
  float* dW_r; float* db_r; float* dW_noise;             /* out [h, E], [E] or NULL, [h, E] (noisy) */
  float* dW_gate_shared; float* dW_up_shared; float* dW_down_shared;  /* out (n_shared > 0) */
} moe_layer_grads;

/* The whole backward for L = <dO, out> + w_aux E sum_i f_i P_i + w_z L_z, the routing decisions
 * of the forward held fixed: moe_combine_backward, moe_route_backward, moe_expert_ffn_backward,
 * the shared experts' backward, moe_router_input_backward, moe_dispatch_backward, in order on
 * `stream`.  `a` holds the forward's inputs and the tensors it saved (logits_out must have been
 * requested; act, Y, X, act_shared, idx, gate, slot_row, offsets, counts_routed). */
moe_status moe_layer_backward(const moe_config* cfg, const moe_layer_args* a, const moe_layer_grads* g,
                              void* ws, moe_stream_t stream);


/* Synchronises `stream`, returns the device status word of `ws` in *code
 * (MOE_DEV_*) and clears it.  Returns MOE_ERR_DEVICE if the word was set. */
moe_status moe_get_device_status(void* ws, moe_stream_t stream, int32_t* code);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H_ */
