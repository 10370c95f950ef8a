/*
 * specdec.h — C ABI of the GB300 speculative-sampling verifier (libspecdec.so).
 *
 * The library runs the verify step of speculative decoding (Leviathan et al.,
 * "Fast Inference from Transformers via Speculative Decoding", Algorithm 1, as
 * restated on the bloss0m reading notes "Speculative Decoding：用小模型打草稿、
 * 大模型一次驗…", sections "Algorithm 1" and "Speculative sampling (Section
 * 2.3)", and on the vllbc notes "Speculative Decoding：draft 先猜，target 一次
 * 验证", Algorithm 1 steps 3-4) for a whole batch of requests in one call, on
 * one GPU, asynchronously on the caller's stream.  Per request b with gamma_b
 * drafts it
 *   1. forms p_i = softmax(target_logits_i / T) for i = 0..gamma_b;
 *   2. tests draft i with r_i < min(1, p_i(x_i) / q_i(x_i)) (strict, as in the
 *      pseudo-code of the timinsight guide "Speculative Decoding 實作指南", Step 2)
 *      and stops at the first rejection: n_b = accepted drafts;
 *   3. draws one more token t: from norm(max(0, p_n - q_n)) when n_b < gamma_b
 *      (correction), else from p_gamma (bonus);
 *   4. reports beta_i = sum_v min(p_i(v), q_i(v)) for every draft position
 *      (Theorem 3.5 / Corollary 3.6 on the same pages).
 * At T == 0 it runs the greedy reading of the vllbc page's Section 2.2 note
 * (argmax folds into the adjusted p, q): accept iff x_i equals the target argmax
 * (lowest index on ties), t = argmax of row n_b, beta_i = [x_i == argmax].
 *
 * Randomness is counter based, so a call is a pure function of its inputs and
 * `seed` (SplitMix64 of Steele, Lea and Flood, OOPSLA 2014):
 *     sm(z)  = SplitMix64 finaliser applied to z + 0x9E3779B97F4A7C15
 *     key    = sm(sm(sm(seed) ^ b) ^ ((pos << 8) | stream))
 *     h      = sm(key ^ (v >> 1))      (one hash for the pair of entries 2j, 2j + 1)
 *     U      = ((h >> 41) + 0.5) * 2^-23                 for even v
 *     U      = (((h >> 18) & (2^23 - 1)) + 0.5) * 2^-23  for odd v   (exact in float32)
 * r_i = U(seed, b, i, stream 0, v 0); the extra token is the exponential race
 * t = argmax_v w(v) / E_v with E_v = -ln U(seed, b, n_b, stream 1, v), an exact
 * sampler of norm(w) that needs no normaliser and no prefix scan.
 *
 * Batch layout (the flattened ragged batch that the vllbc page describes for
 * vLLM's rejection sampler, `cu_num_draft_tokens`):
 *   cu[0] = 0, cu[b+1] = cu[b] + gamma_b, N_d = cu[B], N_t = N_d + B.
 *   draft row / id of (b, i), i < gamma_b : cu[b] + i
 *   target row of (b, i),     i <= gamma_b: cu[b] + b + i   (i = gamma_b: bonus row)
 *   output token slot of (b, i)           : cu[b] + b + i
 * All matrices are row-major and contiguous: target_logits [N_t, V],
 * draft_probs [N_d, V].
 *
 * Ownership: the caller owns every input and output buffer (device memory).  The
 * handle owns a device workspace (per-row softmax statistics, adjusted-row
 * thresholds, status words, greedy keys and the dual kernel's halves, 80 bytes
 * per target row, plus 1036 bytes per request) and one stream-ordered error
 * word.  A handle serves one stream at a time; calls on it are asynchronous and
 * never synchronise, except the first call that needs a larger workspace than
 * specdec_reserve() provided (it reads cu[B] back to size it).  A call on a
 * handle makes the handle's device current while it runs and restores the
 * calling thread's current device before it returns; the stream must belong to
 * the handle's device.  Calls without a handle run on the current device.
 *
 * Errors: host-checked problems return a negative status before anything is
 * launched.  Problems only the device can see (a draft id outside [0, V), a
 * cu array that does not start at 0 or decreases, more rows than the reserved
 * workspace) set bits of the handle's sticky device error word, never trap, and
 * leave the affected outputs defined: a bad draft id is treated as a rejected
 * draft with p(x) = q(x) = 0; a bad cu or capacity overflow writes nothing.
 */
#ifndef SPECDEC_H
#define SPECDEC_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct specdec_ctx* specdec_handle_t;

/* dtype of target_logits (draft_probs are always float32) */
#define SPECDEC_F32 0
#define SPECDEC_BF16 1

/* status codes */
#define SPECDEC_OK 0
#define SPECDEC_ERR_INVALID_ARG (-1)
#define SPECDEC_ERR_UNSUPPORTED_DTYPE (-2)
#define SPECDEC_ERR_CUDA (-3)
#define SPECDEC_ERR_OOM (-4)
#define SPECDEC_ERR_BAD_DRAFT_ID (-5)
#define SPECDEC_ERR_CAPACITY (-6)
#define SPECDEC_ERR_TIMEOUT (-7)

/* bits of the device error word */
#define SPECDEC_DEVERR_BAD_DRAFT_ID 1u
#define SPECDEC_DEVERR_BAD_CU 2u
#define SPECDEC_DEVERR_CAPACITY 4u
#define SPECDEC_DEVERR_TIMEOUT 8u
#define SPECDEC_DEVERR_BAD_TREE 16u   /* specdec_tree_verify: a node's parent is not an earlier node */

/* execution paths (specdec_set_path); AUTO picks per call */
#define SPECDEC_PATH_AUTO 0
#define SPECDEC_PATH_FUSED 1    /* cluster-staged single HBM pass (T > 0)            */
#define SPECDEC_PATH_TWO_PASS 2 /* statistics kernel, then verify kernel (T > 0)     */
#define SPECDEC_PATH_SWEEP 3    /* one CTA per row pair, second sweep from L2 (T > 0) */
#define SPECDEC_PATH_GREEDY 4   /* reported by specdec_last_path for T == 0          */
#define SPECDEC_PATH_STREAM 5   /* the two sweeps fed by bulk copies through a shared-
                                   memory ring (T > 0; needs 16-byte aligned rows)   */
#define SPECDEC_PATH_PAIR 6     /* the two sweeps with each row split over a 2-CTA
                                   cluster (T > 0)                                    */
#define SPECDEC_PATH_DUAL 7     /* two independent CTAs per row: each sweeps the whole
                                   row for (max, sum) and half of it for the rest;
                                   the second to finish combines (T > 0)            */

/* Creates a handle bound to CUDA device `device`.  *out receives the handle.
 * Returns SPECDEC_OK, SPECDEC_ERR_INVALID_ARG (null out, bad device),
 * SPECDEC_ERR_OOM or SPECDEC_ERR_CUDA. */
int specdec_create(specdec_handle_t* out, int device);

/* Pre-sizes the workspace for calls with cu[B] <= max_draft_positions and
 * B <= max_batch, so that later calls within those bounds allocate nothing and
 * never read cu back to the host.  Optional.  Returns SPECDEC_OK,
 * SPECDEC_ERR_INVALID_ARG or SPECDEC_ERR_OOM. */
int specdec_reserve(specdec_handle_t h, int64_t max_draft_positions, int max_batch);

/* One verify step for B requests (see the top of this file for the layout).
 *   target_logits      device [N_t, V] of `dtype`; any alignment (16-byte aligned
 *                      rows, with draft rows to match, are read with 16-byte
 *                      vector loads, other rows element by element)
 *   dtype              SPECDEC_F32 or SPECDEC_BF16
 *   draft_probs        device [N_d, V] float32 rows of q (taken as given, not
 *                      renormalised); ignored when T == 0.  NULL at T > 0 means
 *                      a one-hot ("greedy") drafter, q_i = [v == x_i] (the
 *                      vllbc page's Section 2.2 note on vLLM's draft sampling):
 *                      beta_i = p_i(x_i), accept iff r_i < p_i(x_i), and the
 *                      correction is drawn from p with x removed; no draft row
 *                      is read
 *   draft_ids          device [N_d] int32 (a valid pointer even when N_d == 0)
 *   cu_num_draft_tokens device [B+1] int32, cu[0] = 0, non-decreasing
 *   B, V               requests (>= 1) and vocabulary size (1 .. 2^30)
 *   T                  temperature: > 0 samples, == 0 greedy; NaN, inf or < 0 is
 *                      SPECDEC_ERR_INVALID_ARG
 *   seed               generator seed
 *   out_tokens         device [N_t] int32: slots cu[b]+b .. cu[b]+b+n_b-1 get the
 *                      accepted drafts, slot cu[b]+b+n_b the correction / bonus
 *                      token, later slots of the request -1
 *   out_num_accepted   device [B] int32: n_b in [0, gamma_b]
 *   out_beta           device [N_d] float32 beta_i for every draft position, or NULL
 *   stream             cudaStream_t (NULL = legacy default stream)
 * Returns SPECDEC_OK once the kernels are queued, a negative status otherwise. */
int specdec_rejection_sample(specdec_handle_t h, const void* target_logits, int dtype,
                             const float* draft_probs, const int32_t* draft_ids,
                             const int32_t* cu_num_draft_tokens, int B, int V, float T,
                             uint64_t seed, int32_t* out_tokens, int32_t* out_num_accepted,
                             float* out_beta, void* stream);

/* As specdec_rejection_sample, with three more optional per-draft-position
 * outputs (device [N_d], each may be NULL):
 *   out_target_prob   p_i(x_i) (0 for an out-of-range id; [x_i == argmax] at T == 0)
 *   out_draft_prob    q_i(x_i) (0 for an out-of-range id; 1 at T == 0)
 *   out_accept        int32 result of the accept test at every position, also
 *                     after the first rejection, where it no longer matters
 * and `request_offset`: request b of this call uses generator index
 * request_offset + b, so a batch split into shards (one call per GPU, each
 * with the index of its first request) draws exactly what one call over the
 * whole batch draws.  specdec_rejection_sample uses 0. */
int specdec_rejection_sample_ex(specdec_handle_t h, const void* target_logits, int dtype,
                                const float* draft_probs, const int32_t* draft_ids,
                                const int32_t* cu_num_draft_tokens, int B, int V, float T,
                                uint64_t seed, uint64_t request_offset, int32_t* out_tokens,
                                int32_t* out_num_accepted, float* out_beta,
                                float* out_target_prob, float* out_draft_prob,
                                int32_t* out_accept, void* stream);

/* As specdec_rejection_sample_ex, with the target distribution of every row of
 * request b restricted by top-k and top-p before the test (the vllbc page's
 * Section 2.2 note folds top-k and top-p, like temperature, into the adjusted
 * p that the same rejection test then uses):
 *   top_k   device [B] int32 or NULL.  top_k[b] in [1, V) keeps the tokens with
 *           fewer than top_k[b] larger logits (every token tied with the k-th
 *           largest logit stays); other values switch top-k off for b.
 *   top_p   device [B] float32 or NULL.  top_p[b] < 1 keeps, among the tokens
 *           top-k kept, those whose larger-logit tokens hold no mass or less
 *           than top_p[b] of the top-k mass (the smallest top set reaching
 *           top_p[b], ties at its edge included); values <= 0 and NaN keep the
 *           most probable tokens only; values >= 1 switch top-p off for b.
 * p'_i is then p_i restricted to the kept tokens and renormalised; beta, the
 * accept test, the correction max(0, p' - q) and the bonus draw all use p'.
 * Draft probabilities are taken as already adjusted by the caller.  At T == 0
 * both are ignored (the argmax is always kept).  Adjusted calls run on the
 * sweep path whatever specdec_set_path asked for; each adjusted row costs a few
 * extra passes over the row while it is held in L2 (a selection of the
 * threshold: exact counts, masses as 64-bit fixed point).
 * NULL, NULL is exactly specdec_rejection_sample_ex. */
int specdec_rejection_sample_topk_topp(
    specdec_handle_t h, const void* target_logits, int dtype, const float* draft_probs,
    const int32_t* draft_ids, const int32_t* cu_num_draft_tokens, int B, int V, float T,
    const int32_t* top_k, const float* top_p, uint64_t seed, uint64_t request_offset,
    int32_t* out_tokens, int32_t* out_num_accepted, float* out_beta, float* out_target_prob,
    float* out_draft_prob, int32_t* out_accept, void* stream);

/* ---- token trees: several candidates per position --------------------------
 * Verifies B requests whose drafts form trees (the tree drafts of EAGLE that the
 * tarrragon page lists among the drafter variants; the vllbc page, Section 3.6,
 * notes that any drafter works as long as its probabilities are known at
 * verification).  The pages state the accept rule for one candidate per
 * position; this entry point applies it again after each rejection, with the
 * normalised residual as the next candidate's target (the correctness argument
 * of the vllbc page's Appendix A.1 holds at every round):
 *   request b owns nodes cu[b] .. cu[b+1]-1 (at least one); its node 0 is the
 *   context the target has seen, every other node j carries a draft token
 *   node_tokens[j] and a parent node_parent[j] (an index within the request,
 *   < j; node 0 has -1).  The children of a node, in node order, are
 *   candidates for the same next token, each drawn independently from that
 *   node's draft distribution q_u.  Target row j (target_logits, [N, V], N =
 *   cu[B]) is the target's distribution after node j, draft row j
 *   (draft_probs, [N, V] float32) the drafter's; draft rows of nodes without
 *   children are never read.
 *   At node u with target t (first p_u = softmax(target row u / T)), child r
 *   with token x is accepted when U(seed, b, u, 0, r) < min(1, t(x) / q_u(x));
 *   otherwise t <- norm(max(0, t - q_u)) (t unchanged if that is zero
 *   everywhere).  An accepted child becomes the next node; after the last
 *   rejection, or at a node without children, the extra token is drawn from t
 *   by the exponential race with U(seed, b, u, 1, v).  On a chain (node i + 1
 *   the only child of node i) this is exactly specdec_rejection_sample_ex.
 *   T == 0 is greedy: the first child whose token is the argmax of target row
 *   u (lowest index on ties) is accepted; otherwise that argmax is the extra
 *   token; draft_probs may be NULL.
 * Outputs (device; slots follow the nodes):
 *   out_tokens        [N] int32: request b's accepted tokens in slots
 *                     cu[b] .. cu[b] + n_b - 1, the extra token in slot
 *                     cu[b] + n_b, later slots -1
 *   out_num_accepted  [B] int32 n_b (the depth reached)
 *   out_path          [N] int32 or NULL: the accepted nodes (indices within the
 *                     request) in the first n_b slots of the request, then -1
 * request_offset as in specdec_rejection_sample_ex.  Host-checked errors as for
 * the other entry points (draft_probs NULL at T > 0 is SPECDEC_ERR_INVALID_ARG).
 * Device-detected: a token outside [0, V) is a rejected candidate
 * (SPECDEC_DEVERR_BAD_DRAFT_ID); a request whose tree is malformed writes
 * nothing (SPECDEC_DEVERR_BAD_TREE; SPECDEC_DEVERR_BAD_CU for cu[0] != 0 or a
 * request without nodes); a node with more than 256 children has only its
 * first 256 tested (SPECDEC_DEVERR_CAPACITY).  One CTA walks a request: per
 * visited node one pass over its target row, one over the row pair for every
 * rejection followed by another candidate, and one for the race. */
int specdec_tree_verify(specdec_handle_t h, const void* target_logits, int dtype,
                        const float* draft_probs, const int32_t* node_tokens,
                        const int32_t* node_parent, const int32_t* cu_num_nodes, int B, int V,
                        float T, uint64_t seed, uint64_t request_offset, int32_t* out_tokens,
                        int32_t* out_num_accepted, int32_t* out_path, void* stream);

/* Reads the handle's sticky device error word (SPECDEC_DEVERR_* bits) into
 * *device_error and clears it.  Queues the read on `stream` and waits for it, so
 * it reports every call queued on that stream before it.  Returns SPECDEC_OK,
 * SPECDEC_ERR_INVALID_ARG (null handle or pointer) or SPECDEC_ERR_CUDA. */
int specdec_get_error(specdec_handle_t h, int* device_error, void* stream);

/* Forces an execution path for T > 0 (SPECDEC_PATH_FUSED, _TWO_PASS, _SWEEP,
 * _STREAM, _PAIR, _DUAL or _AUTO, the default, which takes PAIR for batches of fewer
 * requests than twice the SM count and SWEEP otherwise).  A forced FUSED or STREAM
 * path falls back to SWEEP where its layout rules (16-byte aligned rows; for
 * FUSED a vocabulary that fits a cluster) do not hold. */
int specdec_set_path(specdec_handle_t h, int path);

/* Profiling hook: when set, every later call records `before_rows`
 * (cudaEvent_t) on its stream just before the row kernel(s) and `after_rows`
 * just after them, so a caller can time the dominant kernel on its own stream.
 * Pass NULL, NULL to stop.  The events stay owned by the caller. */
int specdec_set_timing_events(specdec_handle_t h, void* before_rows, void* after_rows);

/* Profiling hook for adjusted (top-k / top-p) rows (no counterpart in the pages;
 * it reports how this library's selection resolved each row): when set, every later call
 * adds to device_counters (device memory, 8 uint64 entries, owned by the
 * caller, zeroed by the caller): [0] adjusted rows, [1] rows whose sampled
 * estimate put the edge in the tail, [2] rows whose edge lay past the
 * estimated cut (both take a selection over the whole row), [3] key-refinement
 * passes, [4] rows left without a threshold (NaN logits), [5] rows resolved on
 * bins of one bf16 value each (one counting pass), [6..7] unused.
 * NULL stops. */
int specdec_set_adjust_counters(specdec_handle_t h, uint64_t* device_counters);

/* Test hook for the bounded waits (no counterpart in the pages; it exercises
 * this library's failure handling without faulting the GPU).  The kernels that
 * wait on another CTA (the cluster paths) give every wait a time limit and, when
 * it runs out, set SPECDEC_DEVERR_TIMEOUT and leave.  With
 * mode = SPECDEC_FAULT_PAIR_STALL, later calls on the pair path (forced with
 * specdec_set_path) have rank 0 of every 2-CTA cluster withhold the first work
 * slot from rank 1, whose wait then runs out after wait_limit_ns (1 ns .. 2 s;
 * the pair kernel's waits all use this limit while the hook is on); the call's
 * outputs are then undefined and the error word carries the timeout bit.
 * SPECDEC_FAULT_NONE (wait_limit_ns ignored) restores normal operation.
 * Returns SPECDEC_OK or SPECDEC_ERR_INVALID_ARG. */
#define SPECDEC_FAULT_NONE 0
#define SPECDEC_FAULT_PAIR_STALL 1
int specdec_set_fault_injection(specdec_handle_t h, int mode, uint64_t wait_limit_ns);

/* Path the last call on this handle used (SPECDEC_PATH_FUSED, _TWO_PASS, _SWEEP,
 * _STREAM, _PAIR, _DUAL or _GREEDY), and the cluster size of a cluster path (0
 * otherwise). */
int specdec_last_path(specdec_handle_t h, int* path, int* cluster_size);

/* Writes out[j] = U(seed, b, pos, stream_id, v0 + j) for j < n into device
 * memory `out` (float32, exact), from the same device code the verifier uses.
 * Returns SPECDEC_OK, SPECDEC_ERR_INVALID_ARG or SPECDEC_ERR_CUDA. */
int specdec_uniform(uint64_t seed, uint64_t b, uint64_t pos, uint32_t stream_id, uint64_t v0,
                    int64_t n, float* out, void* stream);

/* Diagnostic: writes out[j] = E(k0 + j) = -ln U for the 23-bit uniform
 * U = (k + 1/2) 2^-23, k = k0 + j < 2^23, computed by the same device code the
 * race uses (so tests can bound its error against double precision). */
int specdec_neg_log_uniform(uint32_t k0, int64_t n, float* out, void* stream);

/* Diagnostic for the top-p edge (no counterpart in the pages; it exposes this
 * library's float32 mass definition so that tests can compare it with an
 * independent implementation): for j < n, out_pow2[j] = 2^-z[j] as the
 * selection computes it (0 for z >= 64 or NaN; otherwise the degree-8 Taylor
 * series of 2^-frac(z) with float32 coefficients (-ln 2)^i / i!, Horner's rule
 * with fused multiply-adds, times 2^-floor(z)) and out_mass[j] = that value
 * times 2^F, F = 62 - ceil(log2 V), rounded to the nearest integer (ties to
 * even): the integer mass an entry at distance z (in base-2 units, z >= 0)
 * from the maximum of a row of V entries contributes to the top-p sums.  z,
 * out_mass and out_pow2 are device arrays of n entries; either output may be
 * NULL.  Asynchronous on `stream`.  SPECDEC_ERR_INVALID_ARG for n < 0,
 * V outside [1, 2^30], or n > 0 with z NULL or both outputs NULL. */
int specdec_selection_mass(const float* z, int64_t n, int V, uint64_t* out_mass, float* out_pow2,
                           void* stream);

/* ---- allocation-free variant -----------------------------------------------
 * No counterpart in the pages: this entry point exists for callers that cannot
 * allocate device memory at the point where they verify (code running inside a
 * memory pool or arena it does not own, plug-ins that are handed only
 * pre-allocated buffers, hosts that freeze device allocation after start-up).
 * It needs no handle and allocates nothing: its scratch (per-row softmax
 * statistics and status words, the deferred-request list, a few counters) is
 * one file-scope device array of about 1.5 MB, which every GPU that loads the
 * library holds until the process exits.  It runs the same kernels as
 * specdec_rejection_sample (the sweep path for T > 0, the greedy path at
 * T == 0) with the same arguments, plus:
 *   n_draft_positions  cu[B] (the host needs it to check the size limits)
 *   out_device_error   optional device word; SPECDEC_DEVERR_* bits are OR-ed
 *                      into it (the caller clears it); NULL drops them
 * Limits: cu[B] + B <= SPECDEC_NOALLOC_MAX_ROWS and B <= SPECDEC_NOALLOC_MAX_BATCH;
 * larger calls return SPECDEC_ERR_CAPACITY before anything is queued.  The
 * check trusts n_draft_positions: when it is below the device's cu[B] and the
 * real rows pass the limit, the kernels skip the rows past it and set
 * SPECDEC_DEVERR_CAPACITY, and the outputs of the requests that own them are
 * left unwritten -- with out_device_error NULL the call then reports nothing.
 * Every call made outside stream capture looks up the array's device address
 * (cudaGetSymbolAddress, a host-side query; after cudaDeviceReset the array
 * may sit elsewhere); a call made while `stream` is capturing reuses the
 * address of the last call on that device outside capture, so make the first
 * call on a device before any capture.  Every call on a device shares the one
 * array and it keeps the last call's contents; each call clears what it
 * accumulates into at its start, on its stream.  Calls whose work overlaps on
 * the GPU (two streams, two host threads) race on the array and must be
 * serialised by the caller. */
#define SPECDEC_NOALLOC_MAX_ROWS 16384
#define SPECDEC_NOALLOC_MAX_BATCH 4096
int specdec_rejection_sample_noalloc(const void* target_logits, int dtype,
                                     const float* draft_probs, const int32_t* draft_ids,
                                     const int32_t* cu_num_draft_tokens, int B, int V, float T,
                                     uint64_t seed, int64_t n_draft_positions,
                                     int32_t* out_tokens, int32_t* out_num_accepted,
                                     float* out_beta, uint32_t* out_device_error, void* stream);

/* Human-readable text of a status code (static storage). */
const char* specdec_status_string(int status);

/* Frees the handle and its workspace (waits for work queued on it). */
int specdec_destroy(specdec_handle_t h);

#ifdef __cplusplus
}
#endif

#endif /* SPECDEC_H */
