/*
 * spec_reject.h -- C ABI of the GB300 (sm_103a) verify-side rejection sampler
 * for speculative decoding.
 *
 * What a call computes (speculative sampling, as defined in "第12章 投机解码：以小博大"
 * §12.2.1-§12.2.4 and §12.3.2, with the flattened ragged layout of §12.3.5):
 *
 *   For request r with k_r = cu_num_draft[r+1] - cu_num_draft[r] drafts
 *   (0 <= k_r <= 32, the MAX_SPEC_LEN of §12.5.4), its k_r + 1 target rows are
 *   t_i = cu_num_draft[r] + r + i (i = 0..k_r) and its draft rows are
 *   d_i = cu_num_draft[r] + i (i < k_r).
 *     p_i = softmax(target_logits[t_i, :] / temperature[r])   (temperature on the target only)
 *     q_i = draft_probs[d_i, :], or one-hot at draft_ids[d_i] when draft_probs == NULL
 *   Sequentially over i: draft x* = draft_ids[d_i] is accepted iff
 *     uniforms[t_i, 0] * q_i(x*) < p_i(x*)        (probability min(1, p/q))
 *   and the scan stops at the first rejection j (later drafts are discarded).
 *   At j < k_r the recovered token is drawn from max(0, p_j - q_j) (one-hot q:
 *   p_j with x* removed); at j = k_r the bonus token is drawn from p_{k_r}.
 *   The draw is an inverse CDF in ascending token order with u = uniforms[t_j, 1]:
 *   the smallest v whose inclusive prefix mass exceeds u times the total.
 *   temperature[r] <= 0 (or NaN) selects the greedy path: accept iff x* equals
 *   the lowest-index argmax of the target row; the output at j is that argmax.
 *
 * Outputs: out_tokens[t_i] = x*_i for i < j, the sampled token at t_j, -1 after;
 *          out_num_accepted[r] = j (accepted drafts, the sampled token excluded).
 *
 * Conventions of every entry point:
 *   - Device pointers are device memory owned by the caller; host pointers are
 *     host memory owned by the caller.  The library allocates nothing.  The only
 *     state it keeps between calls is, per device, a cache of launch shapes (SM
 *     count and kernel occupancy, filled by the first call made with that device
 *     current, safely when several host threads make it at once) and the address
 *     of the fixed scratch array of spec_reject_sample_noalloc(); no result
 *     depends on either.
 *   - A CUDA error that earlier work left pending on the calling thread
 *     (cudaPeekAtLastError() != cudaSuccess) is reported as SPEC_ERR_CUDA before
 *     anything is launched and is left pending; SPEC_ERR_CUDA after a launch
 *     therefore means the call's own launch or copy failed.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls are
 *     asynchronous on that stream unless stated otherwise.
 *   - Errors the host can see (null pointers, bad sizes or strides, dtype,
 *     workspace too small, misaligned pointers) return synchronously and launch
 *     nothing.  Errors that depend on device data (cu_num_draft not starting at
 *     0, not non-decreasing or not ending at T - B; k_r > 32; a draft id outside
 *     [0, V)) are recorded in an error word inside the workspace, read with
 *     spec_reject_last_device_error().  A request with such an error reports
 *     out_num_accepted = -1 and -1 tokens; a batch whose cu_num_draft is
 *     inconsistent as a whole reports -1 for every request and writes no tokens.
 *     No kernel traps or asserts.
 *   - Identical inputs give bit-identical outputs (no floating-point atomics).
 */
#ifndef SPEC_REJECT_H
#define SPEC_REJECT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum spec_status {
    SPEC_OK = 0,
    SPEC_ERR_INVALID_ARG = 1,  /* null pointer, bad size / stride / alignment */
    SPEC_ERR_UNSUPPORTED = 2,  /* vocabulary too large for the chunk tables */
    SPEC_ERR_WORKSPACE = 3,    /* workspace_bytes below spec_reject_workspace_size() */
    SPEC_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed */
    SPEC_ERR_DEVICE_INPUT = 5, /* device data was invalid (see the error word) */
    SPEC_ERR_TIMEOUT = 6       /* reserved: a bounded device wait gave up */
} spec_status;

typedef enum spec_dtype { SPEC_F32 = 0, SPEC_BF16 = 1 } spec_dtype;

/* Largest vocabulary a call accepts. */
#define SPEC_REJECT_MAX_VOCAB 1048576
/* Largest number of drafts per request (MAX_SPEC_LEN). */
#define SPEC_REJECT_MAX_SPEC_LEN 32

/* Bits of the device error word (first int32 of spec_reject_last_device_error's report). */
#define SPEC_DEVERR_LAYOUT 1     /* cu_num_draft[0] != 0, cu[B] + B != T, or cu decreasing */
#define SPEC_DEVERR_SPEC_LEN 2   /* some k_r > 32 */
#define SPEC_DEVERR_DRAFT_ID 4   /* some draft id outside [0, V) */
#define SPEC_DEVERR_TIMEOUT 8    /* a bounded wait inside a kernel gave up (results invalid) */
#define SPEC_DEVERR_TREE 16      /* tree verification: a malformed tree (see spec_tree_verify_greedy) */

/*
 * Bytes of device workspace spec_reject_sample() needs for a batch of B
 * requests, T target rows and vocabulary V.  Depends on the logits dtype
 * (it sets the chunk length) and on whether explicit draft probabilities are
 * given.  Any pointer alignment is accepted; the size includes slack for
 * aligning internally.  Returns 0 for invalid sizes.
 */
size_t spec_reject_workspace_size(int32_t B, int64_t T, int32_t V, spec_dtype logits_dtype, int has_draft_probs);

/*
 * The batched rejection sampler (all steps on the GPU, asynchronous on `stream`).
 *
 *   target_logits     device, [T, V] rows `logits_row_stride` elements apart
 *                     (stride >= V, or 0 = every row aliases row 0), fp32 or bf16
 *                     per `logits_dtype`; element-aligned.  Rows whose start is
 *                     16-byte aligned stream fastest.  -inf entries are masked
 *                     tokens; NaN, +inf or an all -inf row give undefined tokens.
 *   draft_probs       device fp32 [T - B, V] rows `q_row_stride` elements apart
 *                     (>= V or 0), each row a distribution; or NULL for a
 *                     deterministic (one-hot) draft.
 *   draft_ids         device int32 [T - B] (may be NULL when T == B).
 *   cu_num_draft      device int32 [B + 1]: 0, k_0, k_0 + k_1, ..., T - B.
 *   uniforms          device fp32 [T, 2] in [0, 1): column 0 the acceptance
 *                     coin of a verify row, column 1 the sampling draw used at
 *                     the output row.  All randomness comes from here.
 *   temperature       device fp32 [B]; <= 0 (or NaN) selects the greedy path.
 *   out_tokens        device int32 [T].
 *   out_num_accepted  device int32 [B].
 *   workspace         device, at least spec_reject_workspace_size() bytes;
 *                     contents need no initialisation and are overwritten.
 */
spec_status spec_reject_sample(const void *target_logits, spec_dtype logits_dtype, int64_t T, int32_t V,
                               int64_t logits_row_stride, const float *draft_probs, int64_t q_row_stride,
                               const int32_t *draft_ids, const int32_t *cu_num_draft, int32_t B,
                               const float *uniforms, const float *temperature, int32_t *out_tokens,
                               int32_t *out_num_accepted, void *workspace, size_t workspace_bytes, void *stream);

/*
 * spec_reject_sample() with top-k / top-p applied to the target distribution, as
 * "第12章 投机解码：以小博大" §12.2.3 and §12.9 describe (temperature, then top-k, then top-p,
 * on the target only; the draft distribution is used as given).  For a sampled request
 * (temperature > 0) the target p of each of its rows is restricted to
 *   top-k: the tokens whose logit is at least the top_k[r]-th largest (ties kept), then
 *   top-p: among those, the tokens whose logit is at least that of the token at which the
 *          descending cumulative probability first reaches top_p[r] (ties kept),
 * and renormalised; that p' is used for the acceptance test, the recovered token and the
 * bonus token.  top_k[r] <= 0 or >= V, and top_p[r] >= 1 or <= 0, switch a filter off;
 * greedy requests ignore both.  top_k (int32 [B]) and top_p (fp32 [B]) are device arrays,
 * either may be NULL.  bf16 calls of 64 or more requests on 16-byte-aligned rows (without
 * diagnostics) cut each row the first-rejection pass reaches, in the block that reads it;
 * otherwise every row is cut by one thread-block cluster, at most 8 blocks of at most 20
 * chunks of 8 KB.  Both give the same cut and decisions; their draws sum the masses in
 * different orders, so an output token can differ only where the draw falls within fp32
 * rounding of a boundary between two tokens.  Each is deterministic.  The cluster limits V
 * (V <= 655360 bf16 or 327680 fp32; SPEC_ERR_UNSUPPORTED beyond, for every call with
 * filters).  row_sum and p_draft are
 * optional diagnostic outputs (device fp32 [T] and [T - B]): the restricted normaliser
 * sum over kept tokens of exp((l - m) / T_r) and p'(x*).  Same workspace as
 * spec_reject_sample().
 */
spec_status spec_reject_sample_filtered(const void *target_logits, spec_dtype logits_dtype, int64_t T, int32_t V,
                                        int64_t logits_row_stride, const float *draft_probs, int64_t q_row_stride,
                                        const int32_t *draft_ids, const int32_t *cu_num_draft, int32_t B,
                                        const float *uniforms, const float *temperature, const int32_t *top_k,
                                        const float *top_p, int32_t *out_tokens, int32_t *out_num_accepted,
                                        void *workspace, size_t workspace_bytes, void *stream, float *row_sum,
                                        float *p_draft);

/*
 * Reads the device error word of the last call that used `workspace` (waits for
 * `stream`).  Returns SPEC_OK when the device data was valid, else
 * SPEC_ERR_DEVICE_INPUT with *error_bits (SPEC_DEVERR_* bits) and
 * *first_bad_request (lowest offending request; -1 for a layout error) set.
 * Either output pointer may be NULL.  SPEC_ERR_CUDA if the copy failed.
 */
spec_status spec_reject_last_device_error(const void *workspace, void *stream, int32_t *error_bits,
                                          int32_t *first_bad_request);

/*
 * Host-buffer form of spec_reject_sample(): copies the host inputs into a
 * caller-provided device arena, runs the sampler and copies out_tokens and
 * out_num_accepted back.  Synchronous: returns after the host outputs are
 * written (or on the first error).  Host pointers may be pageable or pinned;
 * pinned memory copies fastest.  draft_probs in pinned (page-locked, device-mapped)
 * memory is not copied: the kernels read in place, over the host link, only what the
 * method needs (q(x*) of each verify row and the row at each request's first
 * rejection); pageable draft_probs is copied whole.  When the target logits are pinned
 * too (and draft_probs, if given), the batch has at least 64 requests and rows are
 * 16-byte aligned, nothing large is copied: the target rows are read in place as well,
 * only those up to each request's output row (the pass keeps device copies of those rows, and
 * of the draft row of each explicit-q rejection, in the arena's logits and draft-probability
 * regions for its residual pass and draw).  Rows are passed with the same strides as the
 * device form (0 = aliasing is not allowed here: strides must be >= V).
 * `device_arena` must hold spec_reject_host_arena_size() bytes.
 */
size_t spec_reject_host_arena_size(int32_t B, int64_t T, int32_t V, spec_dtype logits_dtype, int has_draft_probs);
spec_status spec_reject_sample_host(const void *target_logits, spec_dtype logits_dtype, int64_t T, int32_t V,
                                    const float *draft_probs, const int32_t *draft_ids, const int32_t *cu_num_draft,
                                    int32_t B, const float *uniforms, const float *temperature, int32_t *out_tokens,
                                    int32_t *out_num_accepted, void *device_arena, size_t arena_bytes,
                                    void *stream);

/*
 * spec_reject_sample_host() with top-k / top-p on the target distribution (as
 * spec_reject_sample_filtered(): "第12章 投机解码：以小博大" §12.2.3 and §12.9) and the acceptance
 * counters (as spec_reject_sample_ex(), §12.7.5):
 *   top_k, top_p  host int32 [B] / float [B], or NULL (copied into the arena)
 *   counters      host int64 [SPEC_METRIC_COUNT], or NULL: this call's counters are added to
 *                 it (copied to the arena, updated there, copied back)
 * Pinned bf16 logits of 64 or more requests with cuts are still read in place (each reached row
 * is cut from its device copy); fp32 logits with cuts are copied whole.  Same arena size.
 */
spec_status spec_reject_sample_host_ex(const void *target_logits, spec_dtype logits_dtype, int64_t T, int32_t V,
                                       const float *draft_probs, const int32_t *draft_ids,
                                       const int32_t *cu_num_draft, int32_t B, const float *uniforms,
                                       const float *temperature, int32_t *out_tokens, int32_t *out_num_accepted,
                                       void *device_arena, size_t arena_bytes, void *stream, const int32_t *top_k,
                                       const float *top_p, int64_t *counters);

/*
 * Diagnostic form: runs spec_reject_sample() and also writes, per target row,
 * the row maximum m_t, the softmax normaliser s_t = sum_v exp((l - m_t) / T_r)
 * (0 on greedy rows) and the lowest-index argmax; per draft row p_i(x*) (0 on
 * greedy rows); and per request the normalised mass Z of the distribution the
 * output token was drawn from (1 for a bonus draw, sum max(0, p - q) for an
 * explicit-q recovery, 1 - p(x*) for a one-hot recovery, 0 on greedy rows).
 * All debug outputs are device fp32 / int32 arrays; any may be NULL.  Slower
 * than spec_reject_sample (an extra argmax pass); used to check probabilities.
 */
spec_status spec_reject_debug_rowstats(const void *target_logits, spec_dtype logits_dtype, int64_t T, int32_t V,
                                       int64_t logits_row_stride, const float *draft_probs, int64_t q_row_stride,
                                       const int32_t *draft_ids, const int32_t *cu_num_draft, int32_t B,
                                       const float *uniforms, const float *temperature, int32_t *out_tokens,
                                       int32_t *out_num_accepted, void *workspace, size_t workspace_bytes,
                                       void *stream, float *row_max, float *row_sum, int32_t *row_argmax,
                                       float *p_draft, float *z_out);

/*
 * Options of spec_reject_sample_ex(); a NULL pointer switches the option off, and a NULL
 * options pointer is spec_reject_sample().
 *   top_k, top_p       device int32 [B] / fp32 [B]: top-k / top-p on the target, exactly as
 *                      spec_reject_sample_filtered() (same readings and limits)
 *   counters           device int64 [SPEC_METRIC_COUNT], 8-byte aligned: this call's acceptance
 *                      counters are added to it inside the per-request finalize pass (no extra
 *                      launch), with the definitions and the result of
 *                      spec_reject_metrics_update() on the call's outputs (vLLM's spec_decode_*
 *                      counters of "第12章 投机解码：以小博大" §12.7.5)
 *   row_sum, p_draft   diagnostics as in spec_reject_sample_filtered()
 */
typedef struct spec_reject_options {
    const int32_t *top_k;
    const float *top_p;
    int64_t *counters;
    float *row_sum;
    float *p_draft;
} spec_reject_options;

/*
 * spec_reject_sample() with options (see spec_reject_options).  Same arguments, workspace,
 * errors and asynchrony as spec_reject_sample(); a misaligned counters pointer is
 * SPEC_ERR_INVALID_ARG.
 */
spec_status spec_reject_sample_ex(const void *target_logits, spec_dtype logits_dtype, int64_t T, int32_t V,
                                  int64_t logits_row_stride, const float *draft_probs, int64_t q_row_stride,
                                  const int32_t *draft_ids, const int32_t *cu_num_draft, int32_t B,
                                  const float *uniforms, const float *temperature, int32_t *out_tokens,
                                  int32_t *out_num_accepted, void *workspace, size_t workspace_bytes, void *stream,
                                  const spec_reject_options *options);

/*
 * Measurement form of spec_reject_sample() / spec_reject_sample_filtered() (top_k and top_p
 * may be NULL): identical work, plus cudaEventRecord of caller-created events (cudaEvent_t
 * handles) on `stream`: stage_events[0] before the first kernel, then one after each kernel
 * launched, in order.  Calls on 16-byte-aligned rows without cuts (any B >= 1), or with cuts on
 * bf16 rows and at least 64 requests: the layout check, then the pass that reads rows up to
 * each first rejection and draws the outputs (2 events after the first; with events the pass
 * follows the check in plain stream order instead of as a programmatic dependent launch).
 * Otherwise: row statistics, the top-k / top-p cut (filtered calls only), the per-request
 * finalize, the residual / recovery pass (with draft_probs only).  Entries beyond num_events,
 * or NULL entries, are skipped.
 * The pages have no counterpart: this exists to time each kernel on its own stream.
 */
spec_status spec_reject_sample_profiled(const void *target_logits, spec_dtype logits_dtype, int64_t T, int32_t V,
                                        int64_t logits_row_stride, const float *draft_probs, int64_t q_row_stride,
                                        const int32_t *draft_ids, const int32_t *cu_num_draft, int32_t B,
                                        const float *uniforms, const float *temperature, int32_t *out_tokens,
                                        int32_t *out_num_accepted, void *workspace, size_t workspace_bytes,
                                        void *stream, const int32_t *top_k, const float *top_p,
                                        void *const *stage_events, int num_events);

/*
 * spec_reject_sample() for callers that cannot allocate device memory: for example a
 * plugin inside a host inference engine that is handed only its inputs and outputs, or
 * a serving loop that must not call cudaMalloc between steps (it can synchronise the
 * device and stall the other streams).  The pages have no counterpart; this is a
 * deployment convenience.
 *
 * Same arguments and results as spec_reject_sample(), without the workspace: the
 * scratch is a fixed array of SPEC_REJECT_NOALLOC_SCRATCH_BYTES in device memory that
 * every GPU loading this library holds until the process exits.  A batch whose
 * spec_reject_workspace_size() exceeds that returns SPEC_ERR_WORKSPACE and launches
 * nothing (for V = 128256 bf16 logits with draft probabilities and K = 8 that is
 * 3376 requests, 30384 target rows).  Argument errors are reported first, with the status
 * spec_reject_sample() returns for them.  The call allocates nothing.
 *
 * The first call on a device (the current device) looks up the array's device address
 * (once, safely when several host threads make it at once); make that first call before
 * any stream capture.  cudaDeviceReset() on a device invalidates that address: do not call
 * this entry on that device again in the same process.  Every call shares the one array and
 * leaves its contents behind: calls that can overlap on the GPU (different streams, or
 * different host threads on one device) race and must be serialised by the caller.
 *
 * device_error_word: optional device int32[2] that receives the device error word of
 * this call ([0] SPEC_DEVERR_* bits, [1] first bad request or INT32_MAX), copied on
 * `stream` after the kernels; NULL to skip.
 */
#define SPEC_REJECT_NOALLOC_SCRATCH_BYTES (8u << 20)
spec_status spec_reject_sample_noalloc(const void *target_logits, spec_dtype logits_dtype, int64_t T, int32_t V,
                                       int64_t logits_row_stride, const float *draft_probs, int64_t q_row_stride,
                                       const int32_t *draft_ids, const int32_t *cu_num_draft, int32_t B,
                                       const float *uniforms, const float *temperature, int32_t *out_tokens,
                                       int32_t *out_num_accepted, int32_t *device_error_word, void *stream);

/*
 * Acceptance counters, cumulative across calls (the caller zeroes `counters` once):
 * the spec_decode_num_drafts / num_draft_tokens / num_accepted_tokens /
 * num_accepted_tokens_per_pos counters of "第12章 投机解码：以小博大" §12.7.5, and the verify
 * count that "投机解码（Speculative Decoding）端到端深挖" §13 divides by:
 *   accept rate   alpha = counters[NUM_ACCEPTED_TOKENS] / counters[NUM_DRAFT_TOKENS]
 *   accept length tau   = (counters[NUM_ACCEPTED_TOKENS] + counters[NUM_VERIFIES]) / counters[NUM_VERIFIES]
 * (the bonus or recovered token counts in tau, not in alpha).  The library returns the counters
 * only; the two divisions are the caller's (the Python binding's accept_rate_and_length does them
 * as a convenience outside this interface).
 *
 *   cu_num_draft, out_num_accepted  device int32 [B + 1] and [B] of a spec_reject_sample() call
 *   counters                        device int64 [SPEC_METRIC_COUNT], 8-byte aligned
 *
 * Requests reported invalid (out_num_accepted = -1) are not counted.  Asynchronous on
 * `stream`; integer sums, so the result is independent of scheduling.
 */
#define SPEC_METRIC_NUM_DRAFTS 0          /* requests with at least one draft */
#define SPEC_METRIC_NUM_DRAFT_TOKENS 1    /* sum of k_r */
#define SPEC_METRIC_NUM_ACCEPTED_TOKENS 2 /* sum of accepted drafts */
#define SPEC_METRIC_NUM_VERIFIES 3        /* requests verified (each emits accepted + 1 tokens) */
#define SPEC_METRIC_ACCEPTED_PER_POS 4    /* [4 + i]: requests whose draft at position i was accepted */
#define SPEC_METRIC_COUNT (4 + SPEC_REJECT_MAX_SPEC_LEN)
spec_status spec_reject_metrics_update(const int32_t *cu_num_draft, const int32_t *out_num_accepted, int32_t B,
                                       int64_t *counters, void *stream);

/*
 * Greedy tree verification, "投机解码（Speculative Decoding）端到端深挖" §6.2 and §7.1 (draft
 * trees with several siblings per depth, temperature 0).  Request r's nodes are
 * cu_nodes[r] .. cu_nodes[r+1] - 1 (local index i = node - cu_nodes[r]); node 0 is the root
 * (the last verified token), every other node i has parent[node] in [0, i) and draft token
 * node_tokens[node].  target_logits row `node` holds the target's logits for the token after
 * that node's prefix.  From the root: take the lowest-index argmax of the current node's row;
 * the lowest-index child carrying that token is accepted and becomes the current node;
 * otherwise stop.  The argmax at the last accepted node is the bonus token.
 *
 *   target_logits     device [N, V] (fp32 / bf16, rows logits_row_stride apart, stride >= V or 0)
 *   parent            device int32 [N] (-1 at each root)
 *   node_tokens       device int32 [N] (ignored at roots)
 *   cu_nodes          device int32 [B + 1], cu_nodes[B] = N
 *   out_tokens        device int32 [N]: per request, the accepted tokens then the bonus, -1 after
 *   out_num_accepted  device int32 [B] (-1 for a malformed tree)
 *   out_last_node     device int32 [B]: local index of the last accepted node (0 = root)
 *   workspace         spec_tree_workspace_size(N, B, V, dtype) bytes (contents need no setup)
 * Malformed trees set SPEC_DEVERR_TREE in the error word (spec_reject_last_device_error).
 */
size_t spec_tree_workspace_size(int64_t N, int32_t B, int32_t V, spec_dtype logits_dtype);
spec_status spec_tree_verify_greedy(const void *target_logits, spec_dtype logits_dtype, int64_t N, int32_t V,
                                    int64_t logits_row_stride, const int32_t *parent, const int32_t *node_tokens,
                                    const int32_t *cu_nodes, int32_t B, int32_t *out_tokens,
                                    int32_t *out_num_accepted, int32_t *out_last_node, void *workspace,
                                    size_t workspace_bytes, void *stream);

/*
 * n-gram (prompt-lookup) draft proposer, "第12章 投机解码：以小博大" §12.4.4: for each
 * request, for n = max_n down to min_n, the last n context tokens are searched for their
 * leftmost earlier occurrence (one that ends before the final n tokens); the first n that
 * matches wins and the tokens that follow the occurrence are proposed, at most
 * min(k, max_model_len - L) of them (fewer when the context ends first).  No match, or a
 * context that already reaches max_model_len, proposes nothing.
 *
 *   tokens          device int32, all contexts back to back
 *   cu_tokens       device int64 [B + 1]: context r is tokens[cu[r] .. cu[r+1])
 *   min_n, max_n    1 <= min_n <= max_n <= SPEC_NGRAM_MAX_N
 *   k               1 <= k <= 32 (MAX_SPEC_LEN)
 *   max_model_len   <= 0 for no limit
 *   out_drafts      device int32 [B, k], -1 padded
 *   out_num_drafts  device int32 [B]
 * Asynchronous on `stream`; the page runs this search on the CPU with KMP, here every
 * candidate start is tested in parallel by one thread block per request.
 */
#define SPEC_NGRAM_MAX_N 64
spec_status spec_ngram_propose(const int32_t *tokens, const int64_t *cu_tokens, int32_t B, int32_t min_n,
                               int32_t max_n, int32_t k, int64_t max_model_len, int32_t *out_drafts,
                               int32_t *out_num_drafts, void *stream);

/* Kernels one call of B requests on 16-byte-aligned rows in device memory launches: 2 when
 * B >= 1 and the call has no top-k / top-p, or B >= 64 with top-k / top-p on bf16 rows (the
 * layout check, then the pass that reads rows up to each first rejection); otherwise row
 * statistics and the finalize (2), plus the top-k / top-p cut with filters, plus the residual
 * pass with draft probabilities. */
int spec_reject_num_kernels(spec_dtype logits_dtype, int32_t B, int has_draft_probs, int has_filters);

/* Blocks (one thread-block cluster) that work on each request in a call of B requests with
 * V-token rows on the current device that reads rows up to each first rejection without top-k /
 * top-p: 1 when the batch fills the GPU one block per request, else 2, 4 or 8 (rows split over
 * more warps); 0 for invalid sizes or when no device is usable.  The pages have no counterpart:
 * this reports the launch shape, for tests and measurements. */
int spec_reject_blocks_per_request(spec_dtype logits_dtype, int32_t B, int32_t V);

/* Kernel launches one call makes on the current device (16-byte-aligned rows in device memory):
 * spec_reject_num_kernels() stages, of which the first-rejection pass of a large batch is two
 * launches (most requests one block each, the last ones in a second launch chained by
 * programmatic dependent launch, which takes SM slots as the first launch's blocks run out of
 * requests: without top-k / top-p two blocks per request, with them a 16-warp block per
 * request).  The profiled entry records its events per stage.  The pages have no counterpart:
 * this reports the launch shape, for measurements. */
int spec_reject_launches_per_call(spec_dtype logits_dtype, int32_t B, int32_t V, int has_draft_probs,
                                  int has_filters);

/* Static description of a status code. */
const char *spec_reject_status_string(spec_status status);

/* Library version as major * 10000 + minor * 100 + patch. */
int spec_reject_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_REJECT_H */
