/*
 * dflash_select.h — C ABI of the DFlash 2 path selector on one GB300 GPU.
 *
 * The path selector sits between DFlash 2's one-pass block drafter and the
 * target model's verification pass (blog post "DFlash 2: Keep Drafting
 * Parallel", section "A Lightweight Path Selector"). For every sequence of a
 * batch and every draft position t of its block it
 *   1. forms the drafter's lm_head logits U_t = W h_t and keeps the K best
 *      tokens (section "The Right Tokens Are Already There": the right token
 *      is usually among the top 16);
 *   2. scores every adjacent candidate pair,
 *        S_t(a, b) = U_t(b) + < A(a) (.) H(h_t), B(b) >,
 *      with A(a) = W_A E[a], B(b) = W_B E[b], H(h) = W_H h (the pages do not
 *      say how A, B and H are parameterised; this library takes one shared
 *      token table E [V, d] and three [256, d] projections);
 *   3. walks the precomputed tables from the last verified token x0 and
 *      emits one draft path (max-sum walk by default; the literal
 *      best-successor walk on request);
 *   4. (dflash_verify_prefix) keeps the longest prefix of that path that
 *      equals the target's argmax tokens, plus the target's next token.
 *
 * Conventions of every entry point:
 *   - Tensor arguments are DEVICE pointers owned by the caller, row-major and
 *     densely packed, unless the name ends in _host. bf16 is IEEE bfloat16
 *     stored as 16-bit words.
 *   - Calls are asynchronous and ordered on the CUDA stream given as
 *     `stream` (a cudaStream_t; NULL = the legacy default stream). Output
 *     buffers are valid once the stream reaches the point of the call.
 *   - The library never aborts and never exits. A non-zero dflash_status
 *     means nothing was launched; dflash_last_error() then returns a
 *     thread-local message. Problems that only the GPU can see (a token id
 *     out of [0, V), a pipeline wait that ran out of time) are latched in a
 *     device error word that dflash_select_sync_status() reports.
 *   - Draft positions are numbered t = 0 .. L-1 (the pages' positions
 *     1 .. L); x0 precedes position 0.
 */
#ifndef DFLASH_SELECT_H
#define DFLASH_SELECT_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    DFLASH_OK = 0,
    DFLASH_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misaligned buffer */
    DFLASH_ERR_UNSUPPORTED = 2,   /* shape outside the supported set, or not an sm_103 GPU */
    DFLASH_ERR_CUDA = 3,          /* a CUDA runtime/driver call failed */
    DFLASH_ERR_DEVICE_CHECK = 4,  /* a kernel saw an out-of-range token id */
    DFLASH_ERR_TIMEOUT = 5        /* a kernel pipeline wait exceeded its bound */
} dflash_status;

typedef enum {
    DFLASH_WALK_VITERBI = 0,  /* max-sum walk over the pair tables */
    DFLASH_WALK_GREEDY = 1,   /* from x0, follow the best successor at each step */
    DFLASH_WALK_SAMPLE = 2    /* from x0, draw each step from softmax(S_t(prev, .) / temperature)
                                 (dflash_select_run_sampled only) */
} dflash_walk;

/* Shapes fixed for the lifetime of a handle.
 * Supported: 1 <= L <= 16; K in {16, 32}; K <= V; d % 64 == 0, 64 <= d <= 16384;
 * e == 256; 1 <= max_batch with max_batch * L <= 8192; V < 2^31. */
typedef struct {
    int64_t V;          /* vocabulary size (rows of W and E) */
    int32_t d;          /* drafter hidden width */
    int32_t L;          /* draft positions per block (block size - 1) */
    int32_t K;          /* candidates kept per position */
    int32_t e;          /* width of A, B and H; must be 256 */
    int32_t max_batch;  /* largest batch any run will pass; sizes the workspace */
    int32_t walk;       /* dflash_walk */
    float tie_eps;      /* margin under which tie_flags are raised, e.g. 1e-3 */
    float temperature;  /* > 0; used by DFLASH_WALK_SAMPLE */
    int32_t tables;     /* 0: compute A(a) and B(b) of the candidates in every run (the pages' form);
                           1: precompute them for every token at init, [A(v) | B(v)] for v < V as
                           V x 512 fp32 (311 MB at V = 151,936; one GEMM over E of about a
                           millisecond), and gather table rows in every run. Same results up to fp32
                           summation order; a variant of this library, not of the pages. */
    int32_t dedup;      /* 0: project every gathered row; 1: on the larger-batch path (the one that
                           runs separate merge, projection and pair-table kernels), project each
                           distinct token of the batch once (x0 and the candidates of every position
                           and sequence) and let the pair tables read its row. Identical results; needs
                           8 bytes per vocabulary token of workspace; not with tables = 1. A variant of
                           this library, not of the pages. */
} dflash_select_config;

typedef struct dflash_select_ctx *dflash_select_handle;

/* Creates a selector for the weights below (blog, "A Lightweight Path
 * Selector": U_t from the drafter's own lm_head, A/B/H of width 256).
 *   W_lm [V, d] bf16  lm_head weight        E   [V, d] bf16 token table
 *   W_A, W_B, W_H [e, d] bf16               (all 16-byte aligned)
 * The weights are borrowed, not copied: they must stay valid and unchanged
 * until dflash_select_destroy. The handle owns a device workspace sized for
 * cfg->max_batch, allocated here (the only allocation the selector makes).
 * `stream` orders the workspace initialisation. Errors: INVALID_ARG,
 * UNSUPPORTED, CUDA. */
dflash_status dflash_select_init(const dflash_select_config *cfg, const void *W_lm, const void *E,
                                 const void *W_A, const void *W_B, const void *W_H, void *stream,
                                 dflash_select_handle *out);

/* Runs the selector on B sequences (0 <= B <= max_batch; B == 0 is a no-op).
 *   hidden     [B, L, d] bf16  drafter's final hidden states (16-byte aligned)
 *   anchor     [B] int32       last verified token x0 of each sequence
 * Outputs (NULL = not wanted, except path):
 *   topk_ids   [B, L, K] int32 candidates, by logit descending then id ascending
 *   topk_vals  [B, L, K] fp32  their logits U_t
 *   pair_scores[B, L, K, K] fp32  S_t(candidate i of t-1, candidate j of t);
 *              at t = 0 row 0 holds S_0(x0, j) and rows 1..K-1 are -inf
 *   path       [B, L] int32    emitted draft tokens
 *   path_score [B] fp32        sum of the path's pair scores
 *   tie_flags  [B, L] uint8    bit 0: the walk's choice at t had a margin
 *              below tie_eps; bit 1 (t = L-1 only): the final choice did
 * Errors: INVALID_ARG (bad handle, B, pointer or alignment), CUDA. */
dflash_status dflash_select_run(dflash_select_handle h, const void *hidden, const int32_t *anchor,
                                int32_t B, int32_t *topk_ids, float *topk_vals, float *pair_scores,
                                int32_t *path, float *path_score, uint8_t *tie_flags, void *stream);

/* The selector with the sampling walk (handle created with walk =
 * DFLASH_WALK_SAMPLE). Blog "DFlash 2: Keep Drafting Parallel", section "A
 * Lightweight Path Selector": sampling draws from the same pair scores. At
 * every position the next candidate rank is drawn from
 * softmax(S_t(prev, .) / temperature) over the K candidates (prev = the rank
 * drawn at t-1, x0 at t = 0) by inverting the distribution's CDF in rank
 * order with the given uniform.
 *   u_walk      [B, L] fp32 uniforms in [0, 1)
 *   draft_probs [B, L, K] fp32 output: the distribution drawn from at each t
 *               (over the candidates in topk_ids order); needed by
 *               dflash_verify_rejection
 * Other arguments, outputs and errors as dflash_select_run; tie_flags bit 0
 * marks a uniform within tie_eps of a CDF boundary. */
dflash_status dflash_select_run_sampled(dflash_select_handle h, const void *hidden, const int32_t *anchor,
                                        int32_t B, const float *u_walk, int32_t *topk_ids, float *topk_vals,
                                        float *pair_scores, int32_t *path, float *draft_probs,
                                        float *path_score, uint8_t *tie_flags, void *stream);

/* Rejection-sampling verification of a sampled draft (same section: verified
 * by rejection sampling, the output follows the target's distribution
 * exactly). Draft token path[t] is kept when u_acc[t] < min(1, p_t(x) /
 * q_t(x)); at the first rejection the emitted token is drawn from
 * max(0, p_t - q_t) normalised (q_t is zero off the candidates), by inverting
 * its CDF in vocabulary order with u_res; when all L drafts are kept the bonus
 * token is drawn from p_L the same way.
 *   path [B, L] int32, topk_ids [B, L, K] int32, draft_probs [B, L, K] fp32
 *   (as written by dflash_select_run_sampled)
 *   target_probs [B, L+1, V] fp32  target distribution after x0, path[0], ...
 *   u_acc [B, L], u_res [B] fp32 uniforms in [0, 1)
 *   accept_len [B] int32, emitted [B, L+1] int32 (kept drafts, the drawn
 *   token, then -1)
 * 0 <= B, 1 <= L <= 16, K in {16, 32}, K <= V < 2^31. Errors: INVALID_ARG, CUDA. */
dflash_status dflash_verify_rejection(const int32_t *path, const int32_t *topk_ids, const float *draft_probs,
                                      const float *target_probs, const float *u_acc, const float *u_res,
                                      int32_t B, int32_t L, int32_t K, int64_t V, int32_t *accept_len,
                                      int32_t *emitted, void *stream);

/* Greedy verification (blog intro: the target checks the whole block in one
 * pass and keeps the right guesses; the dev.to commentary: greedy output
 * matches the target exactly).
 *   path      [B, L] int32    draft tokens
 *   target    [B, L+1] int32  target argmax token after x0, path[0], ..., path[L-1]
 *   accept_len[B] int32       n = number of leading t with path[t] == target[t]
 *   emitted   [B, L+1] int32  path[0..n-1], target[n], then -1 (NULL = not wanted)
 * 0 <= B, 1 <= L <= 16. Needs no handle. Errors: INVALID_ARG, CUDA. */
dflash_status dflash_verify_prefix(const int32_t *path, const int32_t *target, int32_t B, int32_t L,
                                   int32_t *accept_len, int32_t *emitted, void *stream);

/* dflash_select_run and dflash_verify_prefix in one call: the kernel that
 * walks a sequence's tables also checks its path against the target tokens
 * (one launch fewer per step). Same results as the two calls.
 *   target     [B, L+1] int32  target argmax token after x0, path[0], ..., path[L-1]
 *   path       [B, L] int32    draft tokens (output)
 *   accept_len [B] int32       n = number of leading t with path[t] == target[t]
 *   emitted    [B, L+1] int32  path[0..n-1], target[n], then -1 (NULL = not wanted)
 *   topk_ids, topk_vals, pair_scores, path_score, tie_flags: as dflash_select_run
 * Max-sum and greedy walks. Errors: as dflash_select_run. */
dflash_status dflash_select_run_verify(dflash_select_handle h, const void *hidden, const int32_t *anchor, int32_t B,
                                       const int32_t *target, int32_t *path, int32_t *accept_len, int32_t *emitted,
                                       int32_t *topk_ids, float *topk_vals, float *pair_scores, float *path_score,
                                       uint8_t *tie_flags, void *stream);

/* One whole draft-verify step from HOST buffers: copies hidden to the
 * handle's device staging area (the one upload) and anchor/target into a
 * mapped pinned image of the handle that the kernels read directly, runs
 * dflash_select_run_verify with
 * its results written by the walking kernel straight into a mapped pinned
 * block of the handle, together with a copy of the device error word and a
 * completion flag per sequence, waits for those flags (polling; after 3 s it
 * synchronises the stream instead), and copies path, accept_len and emitted to
 * the caller's buffers. It returns once the results are on the host: the
 * stream may still be retiring the step's last kernel, and later work on the
 * stream stays ordered after it. hidden_host should be pinned for an
 * asynchronous copy. One call at a time per handle (the staging areas are the
 * handle's).
 *   hidden_host [B, L, d] bf16, anchor_host [B], target_host [B, L+1] int32
 *   path_host [B, L], accept_host [B], emitted_host [B, L+1] int32 (outputs)
 * Returns the same errors as the two calls, and any latched device error. */
dflash_status dflash_select_step_host(dflash_select_handle h, const void *hidden_host,
                                      const int32_t *anchor_host, const int32_t *target_host,
                                      int32_t B, int32_t *path_host, int32_t *accept_host,
                                      int32_t *emitted_host, void *stream);

/* Waits for `stream`, then reports and clears the handle's device error word:
 * DFLASH_OK, DFLASH_ERR_DEVICE_CHECK or DFLASH_ERR_TIMEOUT. */
dflash_status dflash_select_sync_status(dflash_select_handle h, void *stream);

/* Per-kernel timing of later runs with CUDA events on the run's stream
 * (enable = 1 turns it on and clears the record, 0 turns it off). Covers
 * dflash_select_run and dflash_select_run_sampled. */
dflash_status dflash_select_profile(dflash_select_handle h, int32_t enable);

/* Reads the record: for kernel index k (0 = lm_head+top-K, 1 = merge,
 * 2 = projection, 3 = pair tables + walk, 4 = the fused small-batch tail that
 * replaces 1..3, 5 = the deduplication of cfg.dedup), total milliseconds and
 * launch count over the recorded runs
 * (at most 4096 runs are recorded). Waits for the recorded events.
 * n_kernels receives the number of kernel indices. */
dflash_status dflash_select_profile_read(dflash_select_handle h, double *ms_total,
                                         int64_t *launches, int32_t max_kernels,
                                         int32_t *n_kernels);

/* Number of kernel launches one dflash_select_run makes for batch B. */
int32_t dflash_select_launches_per_run(dflash_select_handle h, int32_t B);

/* The lm_head + top-K stage alone, for callers that must not allocate device
 * memory (the paper has no counterpart: it is a deployment convenience). A
 * selector handle owns a workspace that dflash_select_init allocates; some
 * hosts cannot allow that, e.g. engines that own all device memory in a
 * preallocated arena, or code paths where an allocation would synchronise the
 * device. This call allocates nothing: its scratch is one fixed 4 MiB device
 * array inside the library, present on every GPU that loads the library until
 * the process exits.
 *   W_lm      [V, d] bf16   lm_head weight (16-byte aligned)
 *   hidden    [N, d] bf16   hidden states of N positions (16-byte aligned)
 *   topk_ids  [N, K] int32  candidates, by logit descending then id ascending
 *   topk_vals [N, K] fp32   their logits (NULL = not wanted)
 *   device_status [1] int32 on the device (NULL = not wanted): 0, or the
 *             device error bits (2 = a pipeline wait ran out of time)
 * Limits: 1 <= N <= 256, K in {16, 32}, d % 64 == 0, and the partial lists
 * (min(SMs / T, ceil(V / 128)) * N * K * 8 bytes, with T = ceil(N / 128)
 * position tiles) must fit in the scratch; larger shapes return
 * DFLASH_ERR_UNSUPPORTED with the sizes in the message.
 * The first call on a device looks up the scratch's address and sets kernel
 * attributes for that device; make that first call before any stream capture.
 * Every call on a device shares the one scratch array, which keeps the last
 * call's contents; calls whose work overlaps on the GPU (different streams,
 * or host threads racing on one device) corrupt each other's results, so
 * order them on one stream. Errors: INVALID_ARG, UNSUPPORTED, CUDA. */
dflash_status dflash_lmhead_topk_noalloc(const void *W_lm, int64_t V, int32_t d, const void *hidden, int32_t N,
                                         int32_t K, int32_t *topk_ids, float *topk_vals, int32_t *device_status,
                                         void *stream);

/* ---- Vocabulary shards (the selector's lm_head split over several GPUs) ----
 * The top-K of a position over the whole vocabulary is the top-K of the union
 * of the shards' top-K lists (blog "DFlash 2: Keep Drafting Parallel",
 * sections "The Right Tokens Are Already There" and "A Lightweight Path
 * Selector": the K best tokens of the drafter's logit at each position). So a
 * GPU that holds only the rows [v0, v1) of the lm_head weight can stream them,
 * keep its own K best per position, and exchange those lists; after the
 * exchange every GPU merges the G lists and runs the rest of the selector.
 * A list entry is a 64-bit key: high word = the fp32 logit mapped to an
 * unsigned integer that preserves its order (bits ^ 0x80000000 for +x, ~bits
 * for -x, -0 taken as +0), low word = ~token_id; a larger key is a better
 * candidate (logit descending, then id ascending), and key 0 is below every
 * real one. */

/* Creates a handle that streams the lm_head rows [v0, v1) only.
 *   W_shard [v1 - v0, d] bf16  rows v0 .. v1-1 of the lm_head weight
 *   E, W_A, W_B, W_H           as dflash_select_init (E covers the whole
 *                              vocabulary: candidates of any shard are gathered)
 * cfg->V is the whole vocabulary; 0 <= v0 < v1 <= V. Such a handle runs
 * dflash_select_topk_shard and dflash_select_run_gathered, not
 * dflash_select_run. Errors: as dflash_select_init. */
dflash_status dflash_select_init_shard(const dflash_select_config *cfg, const void *W_shard, int64_t v0, int64_t v1,
                                       const void *E, const void *W_A, const void *W_B, const void *W_H,
                                       void *stream, dflash_select_handle *out);

/* The handle's shard of the lm_head pass for B sequences: writes the K best
 * keys of every position over tokens [v0, v1), sorted (best first), into
 *   shard_keys [B, L, K] uint64 (device)
 * and keeps g_t = H(h_t) in the handle for dflash_select_run_gathered. Any
 * handle works (a whole-vocabulary handle is the one-shard case).
 * Errors: INVALID_ARG, CUDA. */
dflash_status dflash_select_topk_shard(dflash_select_handle h, const void *hidden, int32_t B, uint64_t *shard_keys,
                                       void *stream);

/* The rest of the selector after the exchange: merges the G shards' lists
 *   all_keys [G, B, L, K] uint64 (device; shard g's dflash_select_topk_shard
 *            output at [g]; the shards' ranges are disjoint and together
 *            cover [0, V))
 * into the top-K of every position, then projections, pair tables and the walk,
 * with the same outputs as dflash_select_run. The gate comes from the last
 * dflash_select_topk_shard on this handle, which must have run the same batch
 * earlier on the same stream. Max-sum and greedy walks; 1 <= G <= 1024.
 * Errors: INVALID_ARG, CUDA. */
dflash_status dflash_select_run_gathered(dflash_select_handle h, const int32_t *anchor, int32_t B,
                                         const uint64_t *all_keys, int32_t G, int32_t *topk_ids, float *topk_vals,
                                         float *pair_scores, int32_t *path, float *path_score, uint8_t *tie_flags,
                                         void *stream);

/* Frees the workspace (after the device is idle) and the handle. Returns a
 * latched device error if one is pending, else DFLASH_OK. NULL is a no-op. */
dflash_status dflash_select_destroy(dflash_select_handle h);

/* Message of the last failed call on this thread ("" if none). */
const char *dflash_last_error(void);

/* Self-test of the bounded pipeline wait (no counterpart in the pages). Every
 * mbarrier wait of the library's kernels gives up after 1 s, latches the
 * device error bit 2 (reported as DFLASH_ERR_TIMEOUT) and lets the kernel
 * return. This launches a one-warp kernel whose wait can never complete, so
 * the caller can observe that path: after about 1 s `device_status` (one
 * int32 on the device, zeroed by the caller) has bit 2 set, and the context
 * stays usable. Errors: INVALID_ARG, CUDA. */
dflash_status dflash_selftest_wait_timeout(int32_t *device_status, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* DFLASH_SELECT_H */
