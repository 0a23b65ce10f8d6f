/*
 * moe.h -- C ABI of libmoe_b300.so: the forward pass of a token-choice top-k
 * Mixture-of-Experts SwiGLU FFN layer on one B300 (sm_103a).
 *
 * The layer, as the pages define it:
 *   route    z = W_r h (+ b_r); p = softmax(z) or sigmoid(z); q = p + bias;
 *            S = TopK(q, k); g = p_S / sum(p_S) (or g = p_S, Switch style)
 *   dispatch regroup the (token, slot) pairs by expert
 *   experts  E_i(x) = W_down_i (SiLU(W_gate_i x) * W_up_i x), one grouped GEMM
 *   combine  y_t = sum_shared E_s(h_t) + sum_{i in S_t} g_{t,i} E_i(h_t)
 *
 * Pages cited (title, section):
 *   [P1] "MOE 专家选择与路由机制"            [P2] "MoE：router 怎样选 expert"
 *   [P3] pwwt.cn MoE blog, §2.1 Top-K      [P4] "拆解 MoE：单个 Token 如何经过专家层"
 *   [P5] "【大模型】MoE（专家混合模型）简介"
 *
 * Conventions shared by every entry point
 *   Memory     All tensor pointers are DEVICE pointers, row-major and contiguous,
 *              16-byte aligned. Rows of h, x_disp, W_* and outputs need a byte
 *              stride that is a multiple of 16: d and ffn multiples of 8 (bf16)
 *              or 4 (fp32).
 *   Ownership  The caller allocates and owns every buffer, the workspace
 *              included. The library allocates no device memory and keeps no
 *              per-call state.
 *   Async      Work is enqueued on `stream`; nothing synchronises. MOE_OK means
 *              the arguments were valid and every launch was accepted. Failures
 *              detected on the device (a bounded wait that ran out) are recorded
 *              in the workspace's status word; read them with moe_read_status.
 *   Errors     No exceptions cross the ABI. Bad shapes, k < 1, k > N, null
 *              required pointers or misaligned pointers return
 *              MOE_ERR_INVALID_ARG before anything is launched. T == 0 returns
 *              MOE_OK with no launch.
 *   dtype      MOE_BF16: h, W_*, x_disp, y_rows, y_shared, out are bf16 and the
 *              GEMMs run on the bf16 tensor cores with fp32 accumulation.
 *              MOE_F32: the same tensors are fp32 and the GEMMs run as tf32.
 *              logits and gates are always fp32; indices are int32.
 */
#ifndef MOE_B300_H
#define MOE_B300_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,   /* bad shape, null or misaligned pointer ([P2] sparse_moe raises on bad shapes) */
  MOE_ERR_UNSUPPORTED = 2,   /* valid request the library does not implement */
  MOE_ERR_WORKSPACE = 3,     /* workspace missing or smaller than moe_workspace_size() */
  MOE_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed */
  MOE_ERR_TIMEOUT = 5,       /* device side: a bounded wait ran out (read via moe_read_status) */
  MOE_ERR_DEVICE_CHECK = 6   /* device side: an index check failed (read via moe_read_status) */
} moe_status;

typedef enum { MOE_BF16 = 0, MOE_F32 = 1 } moe_dtype;

/* [P1] §二 第二步 (softmax); [P2] 最常见的 router (sigmoid, as in DeepSeek-V3). */
typedef enum { MOE_SCORE_SOFTMAX = 0, MOE_SCORE_SIGMOID = 1 } moe_score;

/* [P1] §二 第三步 g = p / sum_S p (SELECTED); [P2] Switch top-1 keeps the full
 * softmax probability, [P3] §2.1 scatters top_probs unrenormalised (NONE). */
typedef enum { MOE_NORM_SELECTED = 0, MOE_NORM_NONE = 1 } moe_norm;

typedef struct {
  int64_t T;          /* tokens (flattened batch x sequence, [P1] §三 steps 1-2) */
  int32_t d;          /* hidden width */
  int32_t N;          /* routed experts, 1..1024 */
  int32_t k;          /* experts per token, 1..min(N, 16) */
  int32_t ffn;        /* routed expert FFN width F */
  int32_t ffn_shared; /* shared expert FFN width; 0 = no shared expert ([P1] §八) */
  int32_t dtype;      /* moe_dtype */
  int32_t score;      /* moe_score */
  int32_t norm;       /* moe_norm */
} moe_config;

/* Bytes of device workspace that moe_forward needs for `cfg` (the largest
 * need of any entry point; every entry point accepts a workspace this size).
 * Returns 0 for an invalid config. Layout is private to the library. */
size_t moe_workspace_size(const moe_config* cfg);

/* Stage 1+2: router logits, scores, top-k selection and gates.
 * [P1] §二 第一步-第三步; [P2] 最常见的 router; [P4] first and second steps.
 *   h          [T, d]  (dtype) hidden states; may be NULL, then logits_in is used
 *   W_r        [N, d]  (dtype) router weight (rows score one expert each)
 *   b_r        [N] fp32 or NULL: router bias added to the logits
 *   sel_bias   [N] fp32 or NULL: per-expert selection bias. It is added to the
 *              score for SELECTION only; gates use the un-biased scores
 *              ([P1] §五 auxiliary-loss-free balancing; [P4] bias paragraph)
 *   logits_in  [T, N] fp32, read iff h == NULL (route given logits, as [P2]
 *              sparse_moe takes logits)
 *   logits_out [T, N] fp32 or NULL: the logits z
 *   idx        [T, k] int32 out: selected experts, by descending selection
 *              score; equal scores go to the lower expert index first
 *   gate       [T, k] fp32 out: gate weight of each selected expert
 *   ws         workspace of moe_workspace_size(cfg) bytes, 256-byte aligned.
 *              Required for bf16 routing from h with N <= 256 (it holds the
 *              tensor-core GEMM's partial logits; MOE_ERR_WORKSPACE without
 *              it); optional otherwise. When given, device-side failures are
 *              recorded in its status word.
 * bf16 routing from h with N <= 256 computes the logits on the tensor cores
 * (fp32 accumulation; a small batch splits the sum over d into slices that are
 * added in a fixed order); fp32 inputs, N > 256 and routing from logits
 * compute them on CUDA cores. Scores, bias, top-k and gates then run in one
 * warp-per-token kernel for every source of logits.
 */
moe_status moe_route(const moe_config* cfg, const void* h, const void* W_r,
                     const float* b_r, const float* sel_bias,
                     const float* logits_in, float* logits_out,
                     int32_t* idx, float* gate,
                     void* ws, size_t ws_bytes, cudaStream_t stream);

/* Stage 3+4: regroup (token, slot) pairs by expert and gather their rows.
 * [P1] §三 Token Dispatch (tokens of one expert listed in ascending order);
 * [P5] §3 ② Dispatch. Deterministic: rows ordered by (expert, token).
 *   h          [T, d] (dtype); idx [T, k] int32 from moe_route (each row holds
 *              k distinct experts in [0, N))
 *   counts     [N] int32 out: rows per expert
 *   offsets    [N+1] int32 out: exclusive prefix sum of counts
 *   row_token  [T*k] int32 out: token of each dispatched row
 *   inv        [T*k] int32 out: inv[t*k + j] = dispatched row of (t, slot j)
 *   x_disp     [T*k, d] (dtype) out: x_disp[r] = h[row_token[r]]; may be NULL
 *              to skip the gather
 *   ws         scratch for the per-block histograms (see moe_workspace_size)
 */
moe_status moe_dispatch(const moe_config* cfg, const void* h, const int32_t* idx,
                        int32_t* counts, int32_t* offsets, int32_t* row_token,
                        int32_t* inv, void* x_disp,
                        void* ws, size_t ws_bytes, cudaStream_t stream);

/* Dispatch for callers that cannot allocate device memory. The pages have no
 * counterpart to this entry point; it exists for callers that have no device
 * allocator to provide moe_dispatch's workspace (a plain C/C++ host program
 * embedding the library without a framework, or a runtime that forbids device
 * allocation after start-up because it can synchronise the device or exceed a
 * fixed memory budget).
 *   Same arguments, layouts and results as moe_dispatch, without the
 *   workspace. The per-block histograms live in a fixed array inside the
 *   library's device image (1 MiB, reserved on every GPU that loads the
 *   library until the process exits). Nothing is allocated: no cudaMalloc,
 *   no cudaFree, no allocating library routine.
 *   Limit: ceil(T / 256) * N <= 262144 (e.g. T <= 65536 with N <= 1024);
 *   larger requests return MOE_ERR_WORKSPACE before anything is launched.
 *   The first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current; make that first call
 *   before any stream capture. The address is cached with the id of the
 *   device's context: after a device reset the next call looks it up again,
 *   so make that call before any capture too.
 *   All calls share the one array: calls whose work overlaps on the GPU (on
 *   different streams, or from several host threads) race and corrupt each
 *   other's results. Serialise them. Out-of-range expert indices are skipped
 *   as in moe_dispatch, but this variant has no device status word: such a
 *   call gives counts that sum to fewer than T*k pairs and no other signal.
 */
moe_status moe_dispatch_noalloc(const moe_config* cfg, const void* h, const int32_t* idx,
                                int32_t* counts, int32_t* offsets, int32_t* row_token,
                                int32_t* inv, void* x_disp, cudaStream_t stream);

/* Expert capacity ([P1] §六 Expert Capacity): C = ceil(capacity_factor * T *
 * k / N), the most (token, slot) pairs one expert keeps. Evaluated on the host
 * in double precision in that order ((capacity_factor * T) * k, then / N) and
 * rounded up; writes *capacity. Requires T >= 0, 1 <= k <= N, a finite
 * capacity_factor >= 0 and a result <= 2^31 (the range moe_dispatch_capacity
 * accepts); otherwise MOE_ERR_INVALID_ARG and *capacity is left unchanged.
 * No CUDA call. */
moe_status moe_expert_capacity(int64_t T, int32_t k, int32_t N, double capacity_factor,
                               int64_t* capacity);

/* Dispatch with an expert capacity ([P1] §六 Expert Capacity: C =
 * ceil(capacity_factor * T * k / N); tokens beyond it may be dropped, the
 * policy is left to the implementation). Each expert keeps its first
 * `capacity` (token, slot) pairs in token order; the rest are dropped:
 * inv[t*k + j] = -1 and no row is written for them. counts/offsets describe the
 * kept rows only (sum counts = kept pairs). Otherwise as moe_dispatch.
 * capacity in [0, 2^31]; 0 drops every pair. */
moe_status moe_dispatch_capacity(const moe_config* cfg, int64_t capacity, const void* h,
                                 const int32_t* idx, int32_t* counts, int32_t* offsets,
                                 int32_t* row_token, int32_t* inv, void* x_disp, void* ws,
                                 size_t ws_bytes, cudaStream_t stream);

/* Stage 5+6: every expert's SwiGLU FFN over its dispatched rows, as one
 * grouped GEMM pair on the tensor cores (tcgen05, TMA-fed).
 * [P1] §一 E_i(h) = W_down (SiLU(W_gate h) * W_up h); [P1] §十二 Grouped GEMM;
 * [P5] §3 ③ and §8 Kernel row.
 *   x_disp     [T*k, d] (dtype), rows grouped by expert as moe_dispatch writes
 *   offsets    [N+1] int32 device array from moe_dispatch
 *   W_gate, W_up [N, ffn, d]; W_down [N, d, ffn] (dtype)
 *   y_rows     [T*k, d] (dtype) out: y_rows[r] = E_e(x_disp[r]) for row r of expert e
 *   h, Ws_gate [ffn_shared, d], Ws_up [ffn_shared, d], Ws_down [d, ffn_shared],
 *   y_shared   [T, d] (dtype) out: the shared expert over all tokens
 *              ([P1] §八); all five are ignored (may be NULL) when
 *              cfg->ffn_shared == 0
 *   ws         holds the [T*k, ffn] (and [T, ffn_shared]) activations
 */
moe_status moe_expert_ffn(const moe_config* cfg, const void* x_disp,
                          const int32_t* offsets, const void* W_gate,
                          const void* W_up, const void* W_down, void* y_rows,
                          const void* h, const void* Ws_gate, const void* Ws_up,
                          const void* Ws_down, void* y_shared,
                          void* ws, size_t ws_bytes, cudaStream_t stream);

/* moe_expert_ffn with the routed rows read straight from h: dispatched row r
 * is h[row_token[r]] (the row_token of moe_dispatch, which can then skip its
 * x_disp copy). The gate/up pass fetches each 128-row tile with TMA gather4
 * loads, four rows per instruction. bf16 only (MOE_ERR_UNSUPPORTED for fp32).
 * It saves the [T*k, d] dispatched copy (memory and its HBM round trip) but
 * issues 32 gather loads per pipeline stage instead of one 16 KB box, which
 * made the grouped GEMM ~2.5x slower on B300; moe_forward uses the copy.
 * Otherwise as moe_expert_ffn. */
moe_status moe_expert_ffn_gather(const moe_config* cfg, const void* h, const int32_t* row_token,
                                 const int32_t* offsets, const void* W_gate, const void* W_up,
                                 const void* W_down, void* y_rows, const void* Ws_gate,
                                 const void* Ws_up, const void* Ws_down, void* y_shared, void* ws,
                                 size_t ws_bytes, cudaStream_t stream);

/* Stage 7: weighted scatter-ADD of every expert output back to its token.
 * [P2] 选好以后: outputs are added, never overwritten or concatenated;
 * [P5] §3 ④ Gather; [P1] §八 shared-expert term.
 *   out[t] = y_shared[t] + sum_{j<k} gate[t,j] * y_rows[inv[t*k+j]]
 *   accumulated in fp32 in slot order, stored in dtype.
 *   y_shared may be NULL (no shared term). out [T, d] (dtype).
 */
moe_status moe_combine(const moe_config* cfg, const void* y_rows,
                       const int32_t* inv, const float* gate,
                       const void* y_shared, void* out, cudaStream_t stream);

/* The whole layer: route -> dispatch -> grouped SwiGLU (+ shared) -> combine.
 * [P1] §十四 moe_forward returns (output, logits); [P2] sparse_moe.
 *   out        [T, d] (dtype) out
 *   logits_out [T, N] fp32 or NULL
 *   idx, gate  [T, k] out (as moe_route); counts [N] int32 out or NULL
 *   Ws_*       NULL when cfg->ffn_shared == 0
 *   ws         at least moe_workspace_size(cfg) bytes
 * Only enqueues work on `stream`: no host synchronisation and no allocation,
 * so after one eager call (which sets up per-device launch caches) the call
 * can be captured in a CUDA graph and replayed on the same buffers.
 */
moe_status moe_forward(const moe_config* cfg, const void* h, const void* W_r,
                       const float* b_r, const float* sel_bias,
                       const void* W_gate, const void* W_up, const void* W_down,
                       const void* Ws_gate, const void* Ws_up, const void* Ws_down,
                       void* out, float* logits_out, int32_t* idx, float* gate,
                       int32_t* counts, void* ws, size_t ws_bytes,
                       cudaStream_t stream);

/* Group-limited selection ([P2] 跨设备时，为什么还要先选组？): the N experts form
 * n_group contiguous groups of N / n_group; each group is scored by its
 * largest selection score (rule 0) or the sum of its top_m scores (rule 1);
 * the topk_group best groups are kept (equal scores: lower group index); the
 * other groups' experts are masked with -inf and the top-k runs over the rest. */
typedef struct {
  int32_t n_group;     /* 1..32, divides N */
  int32_t topk_group;  /* 1..n_group; topk_group * N / n_group >= k ("too few candidates") */
  int32_t rule;        /* 0 = group max, 1 = sum of the group's top_m scores */
  int32_t top_m;       /* 1..min(8, N / n_group), used by rule 1 */
} moe_group_config;

/* moe_route with group-limited selection; arguments as moe_route plus `grp`.
 * Scores, bias and gates are as in moe_route (gates from the un-biased scores
 * of the selected experts). Invalid group settings, including fewer than k
 * candidates in the kept groups, return MOE_ERR_INVALID_ARG. bf16 routing
 * from h with N <= 256 needs the workspace (moe_workspace_size) for the
 * tensor-core GEMM's partial logits, as moe_route does. */
moe_status moe_route_grouped(const moe_config* cfg, const moe_group_config* grp, const void* h,
                             const void* W_r, const float* b_r, const float* sel_bias,
                             const float* logits_in, float* logits_out, int32_t* idx,
                             float* gate, void* ws, size_t ws_bytes, cudaStream_t stream);

/* Routing side statistics of one routing decision ([P1] §五 load-balancing
 * loss and router z-loss; [P1] §十三 per-expert load and routing entropy).
 *   logits [T, N] fp32 (moe_route's logits_out), idx [T, k] int32 (moe_route)
 *   stats  [3 + 2N] fp32 out: L_bal, L_z, entropy, P_0..P_{N-1}, f_0..f_{N-1}
 *          f_i = share of the T*k routed pairs sent to expert i;
 *          P_i = mean over tokens of the router probability of expert i
 *          (softmax; for a sigmoid router the scores divided by their sum);
 *          L_bal = N * sum_i f_i P_i (1 when both are uniform);
 *          L_z = mean over tokens of (log sum_i exp z_ti)^2;
 *          entropy = mean over tokens of -sum_i p_ti log p_ti.
 *   Deterministic (fixed summation order). ws (moe_workspace_size bytes):
 *   per-block partial sums and the counter that picks the block closing the
 *   final reduction; calls sharing one workspace must not overlap on the GPU.
 *   Too small a workspace returns MOE_ERR_WORKSPACE. */
moe_status moe_route_stats(const moe_config* cfg, const float* logits, const int32_t* idx,
                           float* stats, void* ws, size_t ws_bytes, cudaStream_t stream);

/* moe_forward with an expert capacity: dropped (token, slot) pairs contribute
 * nothing; gates are not renormalised over the kept experts; a token whose
 * pairs are all dropped gets the shared expert's output only (zero without
 * one), i.e. only its residual path in the surrounding block. counts = kept
 * rows per expert. */
moe_status moe_forward_capacity(const moe_config* cfg, int64_t capacity, const void* h,
                                const void* W_r, const float* b_r, const float* sel_bias,
                                const void* W_gate, const void* W_up, const void* W_down,
                                const void* Ws_gate, const void* Ws_up, const void* Ws_down,
                                void* out, float* logits_out, int32_t* idx, float* gate,
                                int32_t* counts, void* ws, size_t ws_bytes, cudaStream_t stream);

/* The layer with Expert Choice routing ([P1] §九 routing table; [P2] last
 * section): scores p = softmax (or sigmoid, cfg->score) of the logits; every
 * expert picks the `capacity` tokens with the highest p for it (equal scores:
 * lower token index); y_t = [shared] + sum over experts e that picked t of
 * p_{t,e} E_e(h_t). A token may be picked by no expert (output: shared expert
 * or zero) or by several. cfg->k is the average experts per token the
 * workspace is sized for: require capacity * N <= T * k and capacity <= T.
 *   tokens_out [N, capacity] int32 or NULL: each expert's picked tokens in
 *              ascending order; gates_out [N, capacity] fp32 or NULL: their p
 *   sel_bias and cfg->norm do not apply. ws: moe_workspace_size(cfg) bytes. */
moe_status moe_forward_expert_choice(const moe_config* cfg, int64_t capacity, const void* h,
                                     const void* W_r, const float* b_r, const void* W_gate,
                                     const void* W_up, const void* W_down, const void* Ws_gate,
                                     const void* Ws_up, const void* Ws_down, void* out,
                                     float* logits_out, int32_t* tokens_out, float* gates_out,
                                     void* ws, size_t ws_bytes, cudaStream_t stream);

/* Synchronises `stream`, copies the workspace's device status word into
 * *device_status (MOE_OK, MOE_ERR_TIMEOUT or MOE_ERR_DEVICE_CHECK) and clears
 * it. Returns MOE_ERR_CUDA if the synchronisation or copy fails. */
moe_status moe_read_status(void* ws, size_t ws_bytes, int32_t* device_status,
                           cudaStream_t stream);

/* Test hook for the failure path: launches one CTA that waits on an mbarrier
 * nothing ever arrives on, for at most `budget_ns` nanoseconds (clamped to
 * 1 s), then records MOE_ERR_TIMEOUT in the workspace status word and returns.
 * Never traps and never hangs. */
moe_status moe_selftest_wait_timeout(uint64_t budget_ns, void* ws, size_t ws_bytes,
                                     cudaStream_t stream);

/* Human-readable name of a status code. */
const char* moe_status_string(int32_t status);

#ifdef __cplusplus
}
#endif

#endif /* MOE_B300_H */
