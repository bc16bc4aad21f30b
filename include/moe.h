/*
 * moe.h -- C ABI of libmoe.so, the forward pass of a mixture-of-experts
 * layer on one B300 GPU (sm_103a):
 *
 *   y_t = sum over the top-k experts i of g_i(x_t) * Expert_i(x_t)
 *   ("Expert Parallelism in LLMs: How All-to-All Token Dispatch, Capacity
 *    Factors, and Parallel Folding Scale MoE Architectures", section
 *    "The Distributed MoE Dilemma: Dense vs. Sparse Sharding", the MoE
 *    layer equation)
 *
 * The five calls follow that page's section "The Execution Pipeline":
 *   moe_route            step 1, router gating and top-k selection
 *   moe_dispatch_layout  step 2, local permutation layout, plus the
 *                        per-rank send counts of step 3's all-to-all-v
 *   moe_permute          step 2, the physical reorder into the
 *                        expert-contiguous buffer
 *   moe_grouped_ffn      step 4, batched GEMM per local expert (SwiGLU)
 *   moe_combine          step 6, un-permutation and weighted reduction
 * On one GPU the dispatch and combine all-to-alls (steps 3 and 5) are the
 * identity: the expert-contiguous buffer is the send buffer, split by
 * rank_send_counts / rank_send_displs.
 * Further down: router statistics and the bias step, the dispatch matrix,
 * the static-capacity layout, and the backward pass of every step.
 *
 * Conventions shared by every call
 *  - Pointers are DEVICE pointers unless marked "host".  The caller owns
 *    every buffer, including workspaces; the library keeps no allocation
 *    between calls and never allocates, synchronises or copies to the host.
 *  - Every call is asynchronous on `stream` (NULL = the legacy default
 *    stream).  A return of MOE_OK means the work was enqueued.
 *  - Errors the host can see (null pointer, bad size, misaligned pointer,
 *    unsupported shape or dtype) return MOE_ERR_INVALID or
 *    MOE_ERR_UNSUPPORTED and launch nothing.  A failed launch returns
 *    MOE_ERR_CUDA.
 *  - Errors only the device can see are written to the optional `status`
 *    word (one int32 in device memory, 0 = OK): the first error code wins
 *    (atomic compare-and-swap from 0).  The caller clears it and reads it
 *    when it chooses.  Kernels never trap: out-of-range data is skipped and
 *    reported, and every wait on another warp is bounded in time.
 *  - Matrices are row-major.  "K-major" means the reduction dimension is
 *    contiguous.  Rows of activations must start on 16-byte boundaries:
 *    D * sizeof(element) must be a multiple of 16, and base pointers must be
 *    16-byte aligned (256-byte for buffers read by the tensor-memory
 *    accelerator, noted per call).
 *  - Pair id p = t * k + j names slot j (0 = highest score) of token t.
 */
#ifndef MOE_H_
#define MOE_H_

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

/* Same underlying type as cudaStream_t. */
typedef struct CUstream_st* moe_stream_t;

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID = 1,     /* bad argument, detected on the host           */
  MOE_ERR_UNSUPPORTED = 2, /* valid request outside what this build runs    */
  MOE_ERR_CUDA = 3,        /* a CUDA runtime or driver call failed          */
  MOE_ERR_TIMEOUT = 4,     /* device: a bounded wait expired                */
  MOE_ERR_INDEX = 5        /* device: an expert id outside [0, E), or a
                              buffer row id outside the buffer            */
} moe_status;

typedef enum { MOE_BF16 = 0, MOE_F32 = 1 } moe_dtype;

/* How router logits become selection keys and gates. */
typedef enum {
  /* key = logit; gate = softmax over the k selected logits,
   * g_t = Softmax(TopK(W_g x_t, k)) ("Expert Parallelism in LLMs",
   * The Execution Pipeline, step 1). */
  MOE_SCORE_SOFTMAX_TOPK = 0,
  /* key = logit; gate = softmax over all E experts, taken at the selected
   * ones (the top-1 Switch-style gate). */
  MOE_SCORE_SOFTMAX_FULL = 1,
  /* s = sigmoid(logit) rounded once to fp32, key = s + sel_bias[e] in
   * fp32 (bias steers selection only; the selection is exact on these
   * keys); gate = s_j / sum of the selected s, with s from the fp32
   * sigmoid there (within 3.5 fp32 ulp) ("Expert Parallelism in LLMs",
   * Modern Dropless Dynamic Dispatch: bias terms on routing scores for
   * auxiliary-loss-free balance). */
  MOE_SCORE_SIGMOID_BIAS = 2
} moe_score;

/* Router configuration.  Group-limited selection (n_groups > 1): experts
 * form n_groups contiguous groups; a group's score is the fp32 sum of its
 * group_score_topk largest keys (largest first); the topk_groups best
 * groups stay eligible and the top-k is taken inside them ("Expert
 * Parallelism and All-to-All", Three ways the system fights back: a token
 * reaches at most a few nodes, chosen before the per-expert selection).
 * Ties: equal keys go to the lower expert index, equal group scores to the
 * lower group index.  n_groups = 1 disables grouping. */
typedef struct {
  int32_t T;                /* tokens                                   */
  int32_t D;                /* hidden size                              */
  int32_t E;                /* experts, 1..256                          */
  int32_t k;                /* experts per token, 1..min(E, 32)         */
  int32_t dtype;            /* moe_dtype of x and w_r                   */
  int32_t score;            /* moe_score                                */
  int32_t n_groups;         /* 1 = no grouping; must divide E           */
  int32_t topk_groups;      /* groups kept, 1..n_groups                 */
  int32_t group_score_topk; /* keys summed per group, 1..E/n_groups     */
} moe_route_cfg;

/* Bytes of scratch moe_route needs for `cfg` (partial fp32 logits of the
 * split-K router GEMM).  Returns 0 for an invalid cfg. */
MOE_API size_t moe_route_workspace_size(const moe_route_cfg* cfg);

/* Kernels one moe_route call launches for `cfg`: 1 when E <= 32 and
 *   bf16: E <= 8, or W_r padded to 8, 16 or 32 rows takes at most 96 KiB,
 *         or T <= 16 x the current device's SM count (blocks of up to 16
 *         tokens compute the logits on the warp-level MMA, operands read
 *         straight from global memory, then select);
 *   fp32: W_r padded to 8, 16 or 32 rows takes at most 96 KiB (one warp per
 *         token computes the logits on the CUDA cores from W_r in shared
 *         memory and selects);
 * also 1 in bf16 for E <= 64 with a softmax score, no groups and k <= 2
 * when the router GEMM runs as one K split (moe_route_workspace_size is
 * then T * E * 4 bytes; it splits K while its 128-token row blocks are
 * fewer than half the SMs): it selects in its epilogue; else 2 (the router
 * GEMM, then the select kernel); 0 for an invalid cfg or T = 0.  Host
 * only. */
MOE_API int32_t moe_route_launches(const moe_route_cfg* cfg);

/* moe_route -- router GEMM, score, top-k and gates
 * ("Expert Parallelism in LLMs", The Execution Pipeline, step 1 "Router
 *  Gating and Softmax Selection"; "All-to-All Communication", phase 1
 *  "Routing decision").
 *   cfg           host pointer
 *   x             [T, D] dtype, row-major, 256-byte aligned
 *   w_r           [E, D] dtype, row-major (K-major), 256-byte aligned
 *   logit_offset  [E] fp32 or NULL: added to every token's logits in fp32
 *                 before scoring (it moves both selection and gates)
 *   sel_bias      [E] fp32 or NULL: selection bias, sigmoid mode only
 *   topk_idx      [T, k] int32 out: expert ids, slot 0 = best key
 *   topk_gate     [T, k] fp32 out
 *   logits_out    [T, E] fp32 out or NULL: the exact logits (after the
 *                 offset) that selection used
 *   workspace     >= moe_route_workspace_size(cfg) bytes, 16-byte aligned
 * logits = fp32(x . w_r^T) accumulated in fp32 (bf16 inputs on the tensor
 * cores for MOE_BF16; fp32 FMA for MOE_F32). */
MOE_API moe_status moe_route(const moe_route_cfg* cfg, const void* x, const void* w_r,
                     const float* logit_offset, const float* sel_bias,
                     int32_t* topk_idx, float* topk_gate, float* logits_out,
                     void* workspace, size_t workspace_bytes,
                     int32_t* status, moe_stream_t stream);

/* Bytes of scratch moe_dispatch_layout needs (per-chunk expert
 * histograms).  Returns 0 for invalid sizes. */
MOE_API size_t moe_dispatch_layout_workspace_size(int32_t T, int32_t k, int32_t E);

/* Kernels one moe_dispatch_layout (or moe_dispatch_layout_noalloc) call
 * launches: 1 when one block does the whole layout (T*k <= 16384 pairs and
 * E <= 256), else 3 (histogram, scan, assignment; 1 for T = 0); 0 for
 * invalid sizes.  Host only. */
MOE_API int32_t moe_dispatch_layout_launches(int32_t T, int32_t k, int32_t E);

/* moe_dispatch_layout -- binning of the T*k (token, expert) pairs into an
 * expert-contiguous buffer ("Expert Parallelism in LLMs", The Execution
 * Pipeline, step 2 "Local Token Permutation"; "All-to-All Communication",
 * the expert_parallel_dispatch listing: destination = expert /
 * experts_per_device, bincount of destinations as the send counts), with
 * the capacity clamp C = ceil(CF * k * T / E) ("Expert Parallelism in
 * LLMs", Static Capacity Factors and Token Dropping).
 *   R             virtual expert-parallel ranks; must divide E; rank r owns
 *                 experts [r*E/R, (r+1)*E/R)
 *   capacity      rows per expert; <= 0 means dropless
 *   topk_idx      [T*k] int32 in
 *   expert_counts [E] out: kept pairs per expert = min(routed, capacity)
 *   expert_offsets[E+1] out: exclusive scan of expert_counts
 *   dst_row       [T*k] out: buffer row of pair p, -1 if dropped
 *   src_pair      [T*k] out: pair id held by buffer row r, r < n_kept
 *                 (entries past n_kept are left unwritten)
 *   n_kept, n_dropped   [1] out each
 *   rank_send_counts, rank_send_displs  [R] out: rows bound for each rank
 *                 and where they start (the all-to-all-v split arguments)
 *   workspace     >= moe_dispatch_layout_workspace_size(T, k, E) bytes
 * Pairs are visited in pair-id order: within an expert, rows ascend with p,
 * and a pair is kept iff fewer than `capacity` earlier pairs chose the same
 * expert.  Ids outside [0, E) are dropped and raise MOE_ERR_INDEX in
 * `status`.  Integer results are deterministic. */
MOE_API moe_status moe_dispatch_layout(int32_t T, int32_t k, int32_t E, int32_t R,
                               int32_t capacity, const int32_t* topk_idx,
                               int32_t* expert_counts, int32_t* expert_offsets,
                               int32_t* dst_row, int32_t* src_pair,
                               int32_t* n_kept, int32_t* n_dropped,
                               int32_t* rank_send_counts,
                               int32_t* rank_send_displs,
                               void* workspace, size_t workspace_bytes,
                               int32_t* status, moe_stream_t stream);

/* moe_dispatch_layout_noalloc -- moe_dispatch_layout for callers that
 * cannot allocate device memory: a plugin inside a host engine that owns the
 * whole device memory pool and passes it only input and output buffers, or
 * a service that forbids cudaMalloc after start-up because an allocation
 * can synchronise the device.  The pages have no counterpart; this is a
 * deployment convenience.  Same arguments, outputs and results as
 * moe_dispatch_layout, minus the workspace: the scratch is a static device
 * array of MOE_NOALLOC_LAYOUT_SCRATCH_BYTES inside the library, held by
 * every GPU that loads it until exit.
 *  - Requires ceil(T*k / 2048) * E * 4 <= MOE_NOALLOC_LAYOUT_SCRATCH_BYTES,
 *    else returns MOE_ERR_UNSUPPORTED without launching.
 *  - The first call on each device (with that device current) looks up the
 *    array's device address and caches it for that device's current CUDA
 *    context; make it before any stream capture.  After the context is
 *    destroyed and re-created (cudaDeviceReset) the next call looks the
 *    address up again, so make that call before any capture too.  A failed
 *    lookup returns MOE_ERR_CUDA.
 *  - All calls share the array; overlapping calls on the GPU (unordered
 *    streams) race.  No cudaMalloc, cudaFree or other allocating call. */
#define MOE_NOALLOC_LAYOUT_SCRATCH_BYTES (1u << 20)
MOE_API moe_status moe_dispatch_layout_noalloc(
    int32_t T, int32_t k, int32_t E, int32_t R, int32_t capacity,
    const int32_t* topk_idx, int32_t* expert_counts, int32_t* expert_offsets,
    int32_t* dst_row, int32_t* src_pair, int32_t* n_kept, int32_t* n_dropped,
    int32_t* rank_send_counts, int32_t* rank_send_displs, int32_t* status,
    moe_stream_t stream);

/* moe_permute -- xp[dst_row[t*k + j]] = x[t] for every kept pair
 * ("Expert Parallelism in LLMs", The Execution Pipeline, step 2: tokens
 * physically reordered into contiguous per-destination buffers).  Each
 * token row with a kept pair is read once and written to each of its kept
 * destinations (a scatter by dst_row, so x is read once rather than once per
 * pair); the row of a token whose pairs were all dropped is not read.
 *   x         [T, D] dtype in, 16-byte aligned
 *   dst_row   [T*k] int32 in (moe_dispatch_layout's): < 0 = dropped
 *   xp        [max_rows, D] dtype out, 16-byte aligned; rows not named by
 *             dst_row are left unwritten
 *   max_rows  rows of xp.  A row id >= max_rows is never written: the pair
 *             is skipped and MOE_ERR_INDEX is raised in `status` (nullable).
 */
MOE_API moe_status moe_permute(int32_t T, int32_t k, int32_t D, int32_t dtype,
                       const void* x, const int32_t* dst_row, void* xp,
                       int32_t max_rows, int32_t* status,
                       moe_stream_t stream);

/* Bytes of scratch moe_grouped_ffn needs: the SwiGLU hidden activations
 * H [max_rows, F] in the compute dtype, then (bf16) one 32-bit counter per
 * 128-row block (ceil(max_rows / 128) + E) and one tile ticket, which the
 * call zeroes itself on the stream. */
MOE_API size_t moe_grouped_ffn_workspace_size(int32_t E, int32_t D, int32_t F,
                                      int32_t max_rows, int32_t dtype);

/* moe_grouped_ffn_variant -- which implementation moe_grouped_ffn runs for
 * this size: 1 = fp32 FMA kernel, one launch of one block per row with its
 * H row in shared memory (MOE_F32, F <= 12288); 4 = fp32 FMA kernels, up
 * then down (MOE_F32, F > 12288, two launches); 2 = one
 * persistent tcgen05 launch with a 128-row tile on each SM (cooperative);
 * 3 = one persistent tcgen05 launch of SM pairs (2-CTA clusters,
 * cta_group::2) with 256-row tiles claimed in order, taken when the experts
 * average at least 384 rows (max_rows >= 384 E), F % 256 == 0 and
 * E <= 256; 0 for arguments moe_grouped_ffn rejects or max_rows = 0.
 * Host only. */
MOE_API int32_t moe_grouped_ffn_variant(int32_t E, int32_t D, int32_t F,
                                        int32_t max_rows, int32_t dtype);

/* moe_grouped_ffn -- per-expert SwiGLU over ragged expert segments
 * ("Expert Parallelism in LLMs", The Execution Pipeline, step 4 "Local
 *  Expert Computation": the rows of one expert packed into one GEMM;
 *  Modern Dropless Dynamic Dispatch: ragged grouped GEMM over exact
 *  per-expert counts).  For every expert e and row r in
 *  [expert_offsets[e], expert_offsets[e+1]):
 *     H[r]  = SiLU(xp[r] . W1_e^T) * (xp[r] . W3_e^T)   (rounded to dtype)
 *     yp[r] = H[r] . W2_e^T
 *   xp      [max_rows, D] dtype, 256-byte aligned
 *   w13     [E, 2F, D] dtype: rows 0..F-1 of each expert are W1 (gate),
 *           rows F..2F-1 are W3 (up); K-major; 256-byte aligned
 *   w2      [E, D, F] dtype, K-major; 256-byte aligned
 *   yp      [max_rows, D] dtype out; rows >= expert_offsets[E] untouched
 *   max_rows  rows allocated in xp / yp (>= expert_offsets[E]; T*k works)
 *   max_ctas  MOE_BF16: at most this many CTAs (one per SM); <= 0 means one
 *             per SM of the device.  Fewer leave SMs to other streams.
 * Expert offsets are read on the device: no host synchronisation.
 * MOE_BF16 runs on the tcgen05 tensor cores with fp32 accumulation and
 * needs D % 64 == 0 and F % 128 == 0 (else MOE_ERR_UNSUPPORTED).  It is one
 * persistent launch for both projections in which tiles of the down
 * projection wait (bounded) for the up-projection tiles of their rows held
 * by other CTAs.  With one SM per tile the CTAs walk a fixed schedule, so
 * the launch is cooperative: CUDA makes every CTA resident at once, and a
 * device that cannot host the grid fails the call with MOE_ERR_CUDA instead
 * of stalling.  Experts with many rows run on SM pairs instead
 * (moe_grouped_ffn_variant), which claim tiles in order and need no
 * co-residency; max_ctas is then rounded down to whole pairs, one pair (2
 * CTAs) at least.  MOE_F32 runs fp32 FMA (max_ctas unused). */
MOE_API moe_status moe_grouped_ffn(int32_t E, int32_t D, int32_t F, int32_t max_rows,
                           int32_t dtype, const void* xp,
                           const int32_t* expert_offsets, const void* w13,
                           const void* w2, void* yp, void* workspace,
                           size_t workspace_bytes, int32_t max_ctas,
                           int32_t* status, moe_stream_t stream);

/* moe_combine -- y[t] = sum over kept slots j of
 * topk_gate[t, j] * yp[dst_row[t*k + j]], accumulated in fp32 in slot
 * order, rounded once to dtype ("Expert Parallelism in LLMs", The Execution
 * Pipeline, step 6 "Unpermutation and Weighted Reduction"; dropped pairs
 * contribute nothing, "Static Capacity Factors and Token Dropping").  The
 * residual connection is not added.  A token with no kept pair gets zeros.
 *   yp        [max_rows, D] dtype, 16-byte aligned
 *   dst_row   [T*k] int32 in: < 0 = dropped
 *   topk_gate [T, k] fp32 in
 *   y         [T, D] dtype out, 16-byte aligned
 *   max_rows  rows of yp.  A row id >= max_rows is never read: the pair
 *             contributes nothing and MOE_ERR_INDEX is raised in `status`
 *             (nullable). */
MOE_API moe_status moe_combine(int32_t T, int32_t k, int32_t D, int32_t dtype,
                       const void* yp, const int32_t* dst_row,
                       const float* topk_gate, void* y, int32_t max_rows,
                       int32_t* status, moe_stream_t stream);

/* moe_expert_capacity -- C_expert = ceil(CF * k * T / E) with the capacity
 * factor given as the exact ratio CF = cf_num / cf_den (1.25 = 5 / 4)
 * ("Expert Parallelism in LLMs", Static Capacity Factors and Token
 * Dropping), evaluated in exact integer arithmetic.  Returns the capacity
 * to pass to moe_dispatch_layout, or -1 for cf_num < 0, cf_den <= 0, T < 0,
 * k < 1, E < 1 or a result above INT32_MAX.  Host only. */
MOE_API int32_t moe_expert_capacity(int64_t cf_num, int64_t cf_den, int32_t T,
                                    int32_t k, int32_t E);

/* ------------------------------------------------------------------------
 * Router statistics and load balancing
 * ------------------------------------------------------------------------ */

/* Bytes of scratch moe_router_stats needs (per-block partial sums).
 * Returns 0 for invalid sizes. */
MOE_API size_t moe_router_stats_workspace_size(int32_t T, int32_t E);

/* moe_router_stats -- the auxiliary load-balancing loss of one routing
 * decision ("Expert Parallelism in LLMs", Static Capacity Factors and Token
 * Dropping: L_aux = alpha * E * sum_i f_i * P_i, f_i the fraction of tokens
 * dispatched to expert i, P_i the router probability allocated to it).
 *   score          moe_score of the routing: the router probability of a
 *                  token is the softmax of its E logits (softmax modes) or
 *                  its E sigmoid scores normalised to sum to 1 (sigmoid
 *                  mode)
 *   logits         [T, E] fp32 in: the logits selection used (moe_route's
 *                  logits_out)
 *   topk_idx       [T, k] int32 in: the routing decision
 *   f              [E] fp32 out: routed pairs of expert i / (T*k), counted
 *                  before any capacity drop
 *   P              [E] fp32 out: mean over the T tokens of the router
 *                  probability of expert i
 *   counts_routed  [E] int32 out or NULL: routed pairs per expert
 *   aux_loss       [1] fp32 out: alpha * E * sum_i f_i P_i
 *   workspace      >= moe_router_stats_workspace_size(T, E) bytes, 16-byte
 *                  aligned
 * Probabilities are evaluated in fp32, rounded to multiples of 2^-32 and
 * summed exactly as 64-bit integers (T < 2^31): the results do not depend on
 * the order of the additions and are deterministic.  Ids outside [0, E) are
 * skipped and raise MOE_ERR_INDEX in `status`.  E <= 256,
 * 1 <= k <= min(E, 32). */
MOE_API moe_status moe_router_stats(int32_t T, int32_t E, int32_t k,
                                    int32_t score, const float* logits,
                                    const int32_t* topk_idx, float alpha,
                                    float* f, float* P, int32_t* counts_routed,
                                    float* aux_loss, void* workspace,
                                    size_t workspace_bytes, int32_t* status,
                                    moe_stream_t stream);

/* moe_router_bias_update -- one step of auxiliary-loss-free balancing on the
 * selection bias of MOE_SCORE_SIGMOID_BIAS ("Expert Parallelism in LLMs",
 * Modern Dropless Dynamic Dispatch: bias terms on the routing scores,
 * adjusted dynamically to keep the experts' load balanced).  The pages do
 * not give the rule; this is the plainest one that moves every expert
 * toward the mean load T*k/E:
 *     bias[e] += gamma  if counts_routed[e] * E < T * k   (underloaded)
 *     bias[e] -= gamma  if counts_routed[e] * E > T * k   (overloaded)
 * (exact integer comparison, one fp32 add per expert).
 *   counts_routed  [E] int32 in (moe_router_stats' output)
 *   bias           [E] fp32 in/out */
MOE_API moe_status moe_router_bias_update(int32_t T, int32_t k, int32_t E,
                                          const int32_t* counts_routed,
                                          float gamma, float* bias,
                                          moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Dispatch bookkeeping beyond the compact layout
 * ------------------------------------------------------------------------ */

/* moe_dispatch_matrix -- pairs sent from each virtual source device to each
 * virtual destination device ("All-to-All Communication", the routing
 * simulation listing and its printed dispatch matrix: rows = source device,
 * columns = destination device).  Tokens form n_src equal contiguous shards
 * (token t is on source t / (T / n_src)); experts form n_dst contiguous
 * blocks (expert e lives on destination e / (E / n_dst)).
 *   topk_idx  [T*k] int32 in
 *   dst_row   [T*k] int32 in or NULL: with it, dropped pairs (dst_row < 0)
 *             are not counted; with NULL every routed pair is
 *   matrix    [n_src, n_dst] int32 out (row-major)
 * Requires T % n_src == 0, E % n_dst == 0, n_dst <= 4096.  Row sums are the
 * pairs each source sends; column sums equal moe_dispatch_layout's
 * rank_send_counts when n_dst = R.  Ids outside [0, E) are skipped and raise
 * MOE_ERR_INDEX.  Exact (integer) and deterministic. */
MOE_API moe_status moe_dispatch_matrix(int32_t T, int32_t k, int32_t E,
                                       int32_t n_src, int32_t n_dst,
                                       const int32_t* topk_idx,
                                       const int32_t* dst_row, int32_t* matrix,
                                       int32_t* status, moe_stream_t stream);

/* moe_padded_layout -- rows of the static-capacity buffer [E, C, D]
 * ("Expert Parallelism in LLMs", Static Capacity Factors and Token Dropping:
 * each expert owns a fixed buffer of C_expert rows; empty slots are
 * padding).  Expert e owns rows [e*C, (e+1)*C) and its kept pairs fill them
 * in the compact layout's order:
 *     dst_row_padded[p] = e*C + (dst_row[p] - expert_offsets[e]), or -1
 *     offsets_padded[e] = e*C, e = 0..E
 * The inputs are moe_dispatch_layout's outputs for the same capacity C.
 * moe_permute and moe_combine take dst_row_padded in place of dst_row, and
 * moe_grouped_ffn takes offsets_padded with max_rows = E*C (a padding row
 * is zero after moe_pad_fill, and SwiGLU maps it to zero).
 *   topk_idx, dst_row  [T*k] int32 in; expert_offsets [E+1] int32 in
 *   dst_row_padded     [T*k] int32 out; offsets_padded [E+1] int32 out
 * Requires capacity >= 1 and E * capacity <= INT32_MAX.  A kept row outside
 * its expert's C slots raises MOE_ERR_INDEX and is marked -1. */
MOE_API moe_status moe_padded_layout(int32_t T, int32_t k, int32_t E,
                                     int32_t capacity, const int32_t* topk_idx,
                                     const int32_t* dst_row,
                                     const int32_t* expert_offsets,
                                     int32_t* dst_row_padded,
                                     int32_t* offsets_padded, int32_t* status,
                                     moe_stream_t stream);

/* moe_pad_fill -- zero the padding rows of a padded buffer: rows
 * [e*C + expert_counts[e], (e+1)*C) of buf [E*C, D] for every expert; rows
 * holding kept pairs are not touched.
 *   expert_counts [E] int32 in (kept counts, each <= C)
 *   buf           [E*C, D] dtype in/out, 16-byte aligned */
MOE_API moe_status moe_pad_fill(int32_t E, int32_t capacity, int32_t D,
                                int32_t dtype, const int32_t* expert_counts,
                                void* buf, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Backward pass ("Expert Parallelism in LLMs", Backward Pass Symmetry: the
 * upstream gradient dL/dy is dispatched to the experts along the forward
 * dispatch pattern, the experts form their weight gradients and input
 * gradients, and the input gradients return along the combine pattern).
 * The routing decision is held fixed; gradients flow through the gates and
 * the experts.  Order of calls for one layer:
 *   moe_aligned_layout, moe_aligned_fill (forward rows Xa on 64-row
 *   aligned expert segments), moe_permute / moe_grouped_ffn / moe_combine on
 *   that layout, then
 *   moe_combine_backward -> moe_aligned_fill(dYa) ->
 *   moe_grouped_ffn_backward -> moe_permute_backward -> moe_route_backward.
 * ------------------------------------------------------------------------ */

/* moe_aligned_layout -- the training layout: expert e's rows start at
 * offsets_aligned[e], the exclusive scan of its kept count rounded up to
 * `align` (64 for moe_grouped_ffn_backward), so that no block of `align`
 * rows holds two experts.
 *     dst_row_aligned[p] = offsets_aligned[e] + (dst_row[p] - offsets[e])
 *   topk_idx, dst_row [T*k] int32 in; expert_offsets [E+1] int32 in (the
 *   compact layout's); dst_row_aligned [T*k] out (-1 if dropped);
 *   offsets_aligned [E+1] out.  Rows: offsets_aligned[E] <= T*k + (align-1)*E.
 * Requires 1 <= align <= 1024 and E <= 1024. */
MOE_API moe_status moe_aligned_layout(int32_t T, int32_t k, int32_t E,
                                      int32_t align, const int32_t* topk_idx,
                                      const int32_t* dst_row,
                                      const int32_t* expert_offsets,
                                      int32_t* dst_row_aligned,
                                      int32_t* offsets_aligned,
                                      int32_t* status, moe_stream_t stream);

/* moe_aligned_fill -- zero the padding rows of an aligned buffer: rows
 * [offsets_aligned[e] + count_e, offsets_aligned[e+1]) for every expert,
 * count_e = expert_offsets[e+1] - expert_offsets[e].
 *   buf [offsets_aligned[E], D] dtype in/out, 16-byte aligned */
MOE_API moe_status moe_aligned_fill(int32_t E, int32_t D, int32_t dtype,
                                    const int32_t* expert_offsets,
                                    const int32_t* offsets_aligned, void* buf,
                                    moe_stream_t stream);

/* moe_combine_backward -- backward of moe_combine: for every kept pair
 * (t, j) with row r = dst_row[t*k + j]:
 *     dyp[r]          = topk_gate[t, j] * dy[t]      (dtype)
 *     dgate[t, j]     = dy[t] . yp[r]                (fp32 accumulation)
 * and dgate = 0 for a dropped pair.  Rows of dyp not named by dst_row are
 * left unwritten (moe_aligned_fill zeroes an aligned buffer's padding).
 *   dy [T, D] dtype; yp, dyp [max_rows, D] dtype; dgate [T, k] fp32 out.
 * A row id >= max_rows is neither read nor written: its dgate is 0 and
 * MOE_ERR_INDEX is raised in `status` (nullable). */
MOE_API moe_status moe_combine_backward(int32_t T, int32_t k, int32_t D,
                                        int32_t dtype, const void* dy,
                                        const void* yp, const int32_t* dst_row,
                                        const float* topk_gate, void* dyp,
                                        float* dgate, int32_t max_rows,
                                        int32_t* status, moe_stream_t stream);

/* moe_permute_backward -- backward of moe_permute:
 *     dx[t] = sum over kept slots j of dxp[dst_row[t*k + j]]
 * (fp32 accumulation in slot order, rounded once to dtype; zeros for a
 * token with no kept pair).  dxp [max_rows, D], dx [T, D] dtype.  A row id
 * >= max_rows is never read and raises MOE_ERR_INDEX in `status`
 * (nullable). */
MOE_API moe_status moe_permute_backward(int32_t T, int32_t k, int32_t D,
                                        int32_t dtype, const void* dxp,
                                        const int32_t* dst_row, void* dx,
                                        int32_t max_rows, int32_t* status,
                                        moe_stream_t stream);

/* Bytes of scratch moe_grouped_ffn_backward needs: dH [max_rows, F],
 * dGU [max_rows, 2F] and H [max_rows, F] in the compute dtype. */
MOE_API size_t moe_grouped_ffn_backward_workspace_size(int32_t E, int32_t D,
                                                       int32_t F,
                                                       int32_t max_rows,
                                                       int32_t dtype);

/* moe_grouped_ffn_backward -- backward of moe_grouped_ffn on the aligned
 * layout (every expert_offsets[e] a multiple of 64; padding rows of xp and
 * dyp zero).  For expert e and its rows, with G = xp W1_e^T, U = xp W3_e^T
 * recomputed:
 *     dH   = dyp W2_e
 *     dG   = dH * U * SiLU'(G),  dU = dH * SiLU(G),  H = SiLU(G) * U
 *     dxp  = dG W1_e + dU W3_e                         (dtype out)
 *     dw2[e]  = dyp^T H,  dw13[e] = [dG | dU]^T xp      (fp32 out)
 * An expert with no rows gets zero weight gradients.  MOE_BF16: all five
 * GEMMs run on the tcgen05 tensor cores (bf16 in, fp32 accumulate).
 * MOE_F32: CUDA-core kernels, fp32 throughout, any D and F.
 *   xp, dyp [max_rows, D] dtype, 256-byte aligned (bf16); w13 [E, 2F, D]
 *   and w2 [E, D, F] dtype (the forward weights); dxp [max_rows, D] out;
 *   dw13 [E, 2F, D] and dw2 [E, D, F] fp32 out, 16-byte aligned.
 * MOE_BF16 needs D % 128 == 0 and F % 128 == 0 (else MOE_ERR_UNSUPPORTED);
 * there, unaligned offsets are detected on the device: MOE_ERR_INVALID in
 * `status` and no weight gradient is written.  MOE_F32 takes any offsets. */
MOE_API moe_status moe_grouped_ffn_backward(
    int32_t E, int32_t D, int32_t F, int32_t max_rows, int32_t dtype,
    const void* xp, const void* dyp, const int32_t* expert_offsets,
    const void* w13, const void* w2, void* dxp, float* dw13, float* dw2,
    void* workspace, size_t workspace_bytes, int32_t* status,
    moe_stream_t stream);

/* moe_route_backward -- backward of the router for the decision moe_route
 * made: from dgate [T, k] (moe_combine_backward's output)
 *     dlogits[t]  per score mode (softmax over the selected logits; softmax
 *                 over all E taken at the selected experts; selected
 *                 sigmoid scores normalised to sum 1 -- the selection bias
 *                 has no gradient path)
 *     dw_r        = dlogits^T x                   (fp32, may be NULL)
 *     dx         += dlogits w_r                   (dtype, in place, may be
 *                                                  NULL)
 *   cfg host pointer (as for moe_route); x [T, D], w_r [E, D] dtype;
 *   logits [T, E] fp32 (moe_route's logits_out); topk_idx [T, k];
 *   dlogits [T, E] fp32 out; dw_r [E, D] fp32 out;
 *   workspace >= moe_route_backward_workspace_size(cfg) bytes, 16-byte
 *   aligned (may be NULL when dw_r is NULL, and for bf16 with E and D
 *   multiples of 64 only when dx is NULL too).
 * For bf16 with E and D multiples of 64, dw_r and dx run on the tensor
 * cores: dlogits enters as two bf16 terms hi + lo (hi = bf16(dl),
 * lo = bf16(dl - hi), about 2^-17 relative) and every product accumulates
 * in fp32; x, w_r and dx must then be 16-byte aligned.  Otherwise they run
 * as fp32 sums on the CUDA cores.
 * dw_r and dx are deterministic: fixed-order fp32 sums. */
MOE_API moe_status moe_route_backward(const moe_route_cfg* cfg, const void* x,
                                      const void* w_r, const float* logits,
                                      const int32_t* topk_idx,
                                      const float* dgate, float* dlogits,
                                      float* dw_r, void* dx, void* workspace,
                                      size_t workspace_bytes, int32_t* status,
                                      moe_stream_t stream);

/* Bytes of scratch moe_route_backward needs for dw_r (per-slice partial sums
 * of the token contraction, added in a fixed order).  Returns 0 for an
 * invalid cfg. */
MOE_API size_t moe_route_backward_workspace_size(const moe_route_cfg* cfg);

/* Test hook for the bounded-wait machinery: launches one CTA that waits on
 * a shared-memory barrier nothing arrives on, gives up after `limit_ns`
 * nanoseconds, writes MOE_ERR_TIMEOUT into `status` and returns. */
MOE_API moe_status moe_selftest_bounded_wait(int32_t* status, uint64_t limit_ns,
                                     moe_stream_t stream);

/* Test hook for the selection score of MOE_SCORE_SIGMOID_BIAS: out[i] =
 * fp32(1 / (1 + exp(-l[i]))), the sigmoid evaluated in float64 and rounded
 * once to fp32, exactly as moe_route ranks experts by it before adding the
 * bias (n values, device pointers).  Selection is an integer decision taken
 * on these fp32 values; a checker that evaluates the same definition in
 * float64 agrees bit for bit except within a few float64 ulp of an fp32
 * rounding midpoint. */
MOE_API moe_status moe_selftest_sigmoid_key(const float* l, float* out,
                                            int32_t n, moe_stream_t stream);

/* Human-readable name of a status code (static string). */
MOE_API const char* moe_status_str(int32_t status);

/* ABI version of this header (incremented on any signature change). */
MOE_API int32_t moe_abi_version(void);

#define MOE_ABI_VERSION 2

#ifdef __cplusplus
}
#endif

#endif /* MOE_H_ */
