/*
 * specverify.h -- C ABI of the GB300 verify step for speculative sampling.
 *
 * What the library computes (one call = one verify round for a ragged batch):
 *
 *   "Speculative Decoding: Medusa, MTP, EAGLE, DFlash, DDTree, and DSpark",
 *   section 1 "What Speculative Decoding Actually Guarantees": with p_i the
 *   target distribution and q_i the proposal distribution at draft position
 *   i, draft token y_i is accepted with probability
 *       alpha_i(y_i) = min(1, p_i(y_i) / q_i(y_i)),
 *   positions are tested left to right and everything after the first
 *   rejection is discarded (draft A B C D with C rejected commits A B R); at
 *   the first rejection one token is drawn from the normalised positive
 *   residual [p_i - q_i]_+, and when every draft survives one extra token is
 *   drawn from the target.  Greedy rounds keep y_i while it equals the target
 *   argmax.  Temperature enters p and q alike: p_i = softmax(target_i / T),
 *   q_i = softmax(draft_i / T).  Section 2 of the same page defines A, the
 *   accepted draft-prefix length, excluding the correction or bonus token.
 *
 * Readings this library takes where the pages leave a step open:
 *   - T == 0 means greedy (target argmax, lowest index on ties; draft logits
 *     are not read); T > 0 means sampling.
 *   - The test "u < p(y)/q(y)" is evaluated as u*q(y) < p(y) (strict).
 *   - Randomness is counter-based Philox4x32-10 (Salmon et al., SC'11) with
 *     key = (seed low 32 bits, seed high 32 bits) and counter
 *       (floor(v/4), position, request low 32 bits, stream | request high << 8),
 *     taking output word v mod 4.  Stream 0, v = 0: acceptance uniform
 *     u = (word >> 8) * 2^-24.  Stream 1: race exponentials
 *     E_v = -ln((word + 1/2) * 2^-32).
 *   - Every categorical draw is one exponential race over the vocabulary:
 *       token = argmin_{v: w_v > 0} E_v / w_v   (lowest index on ties),
 *     E_v from the stream-1 word of vocab id v itself (counter floor(v/4),
 *     word v mod 4) at the draw's position and request.  The result does not
 *     depend on how the vocabulary is split across threads.  Correction:
 *     w = [p_j - q_j]_+ at position j = A (Philox position j); if that
 *     residual has no mass the draw is made from p_j with the same
 *     exponentials.  Bonus: w = p_k at position k.
 *   - "request" is the batch index r unless request ids are given.
 *
 * Data layout (row-major, one row = V logits of one position):
 *   request r has k_r = num_draft[r] draft positions;
 *   its target rows are  target_logits[tgt_off(r) + i],  i = 0..k_r,
 *       tgt_off(r) = sum_{s<r} (k_s + 1);
 *   its draft rows are   draft_logits[drf_off(r) + i],   i = 0..k_r-1,
 *   its draft tokens are draft_tokens[drf_off(r) + i],
 *       drf_off(r) = sum_{s<r} k_s.
 *
 * Outputs (caller-owned device memory):
 *   accepted_len[r]                   A_r, or -1 when request r was skipped;
 *   committed_tokens[r*(max_k+1)+i]   y_i for i < A_r, the correction or bonus
 *                                     token at i = A_r, -1 after it;
 *   accept_flags[drf_off(r)+i]        1 if i < A_r else 0 (per-position flags).
 *
 * Errors.  Entry points return SPECVERIFY_OK or a negative error code and
 * launch nothing on an error.  Problems that only the device can see (token
 * out of range, bad temperature, NaN/+inf logits, inconsistent num_draft) set
 * bits in a device status word and skip the affected request (or, for an
 * inconsistent layout, the whole batch); read it with specverify_status().
 * No kernel traps or asserts.
 *
 * Threading.  A handle may be used from one host thread and one stream at a
 * time; concurrent runs on one handle race on its scratch memory.
 */
#ifndef SPECVERIFY_H
#define SPECVERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct specverify_ctx *specverify_t;
typedef struct specverify_tree_ctx *specverify_tree_t;

typedef enum {
    SPECVERIFY_F32 = 0,   /* float32 logits */
    SPECVERIFY_BF16 = 1   /* bfloat16 logits (raw 16-bit patterns) */
} specverify_dtype;

/* Return codes. */
#define SPECVERIFY_OK 0
#define SPECVERIFY_ERR_INVALID_ARG (-1)   /* null pointer, size out of range, misalignment */
#define SPECVERIFY_ERR_DTYPE (-2)         /* unknown dtype */
#define SPECVERIFY_ERR_CUDA (-3)          /* a CUDA runtime call or launch failed */
#define SPECVERIFY_ERR_DESTROYED (-4)     /* handle already destroyed */
#define SPECVERIFY_ERR_NO_STAGING (-5)    /* host entry point on a handle made without staging */
#define SPECVERIFY_ERR_TOO_LARGE (-6)     /* above the static scratch limits (specverify_run_static) */

/* Device status bits (specverify_status). */
#define SPECVERIFY_STATUS_BAD_TOKEN 1     /* a draft token outside [0, V): request skipped */
#define SPECVERIFY_STATUS_BAD_K 2         /* a num_draft outside [0, max_k]: batch skipped */
#define SPECVERIFY_STATUS_BAD_TEMP 4      /* T NaN, negative, infinite or subnormal: request skipped */
#define SPECVERIFY_STATUS_NONFINITE 8     /* NaN/+inf logit, or no finite logit, in a read row: request skipped */
#define SPECVERIFY_STATUS_BAD_TOTAL 16    /* sum of num_draft != total_draft: batch skipped */
#define SPECVERIFY_STATUS_BAD_PARENT 32   /* tree: a parent outside [-1, node index): request skipped */
#define SPECVERIFY_STATUS_NO_DRAFT 64     /* T > 0 and k > 0 but draft_logits is NULL: request skipped */
#define SPECVERIFY_STATUS_BAD_CONF 512    /* trimmed run: a confidence NaN or outside [0, 1], or a NaN cost:
                                             request skipped */
#define SPECVERIFY_STATUS_BAD_TRUNC 1024  /* truncation: a top_p NaN or <= 0 (its rows copied) */

/* Flags for specverify_create_ex. */
#define SPECVERIFY_CREATE_HOST_STAGING 1  /* allocate device staging for specverify_run_host */

/*
 * specverify_create -- make a handle bound to CUDA device `device`.
 *   max_batch  in [1, 4096]: largest batch a run may pass;
 *   max_k      in [0, 31]: largest num_draft (committed rows are max_k+1 wide);
 *   vocab      in [1, 2^30]: V, the logits row length;
 *   dtype      SPECVERIFY_F32 or SPECVERIFY_BF16.
 * Allocates all scratch memory now (a few MB: per-row partial results,
 * counters, the residual work list); runs never allocate.
 * Returns SPECVERIFY_ERR_INVALID_ARG / _DTYPE on bad sizes, _CUDA if the
 * device cannot be used.  *out is NULL on failure.
 */
int specverify_create(specverify_t *out, int device, int max_batch, int max_k, int vocab,
                      int dtype);

/* As specverify_create; flags may add SPECVERIFY_CREATE_HOST_STAGING, which also
 * allocates device buffers for the largest inputs and outputs so that
 * specverify_run_host can copy host data in and out. */
int specverify_create_ex(specverify_t *out, int device, int max_batch, int max_k, int vocab,
                         int dtype, unsigned flags);

/*
 * specverify_run -- verify one ragged batch; asynchronous on `stream`
 * (a cudaStream_t; NULL = the legacy default stream).  All pointers are device
 * pointers owned by the caller:
 *   target_logits   [batch + total_draft, vocab] of dtype, element-aligned;
 *   draft_logits    [total_draft, vocab] of dtype, or NULL when every request
 *                   with k_r > 0 is greedy;
 *   draft_tokens    [total_draft] int32;
 *   num_draft       [batch] int32, each in [0, max_k];
 *   temperature     [batch] float32; 0 = greedy, > 0 = sampling;
 *   seed            Philox key;
 *   batch           in [0, max_batch];
 *   total_draft     host copy of sum_r num_draft[r], in [0, batch*max_k];
 *   accepted_len    [batch] int32 out;
 *   committed_tokens[batch, max_k+1] int32 out;
 *   accept_flags    [total_draft] uint8 out.
 * Enqueues the round's launches (specverify_launches_per_run) and returns
 * without waiting; nothing is allocated.
 */
int specverify_run(specverify_t h, const void *target_logits, const void *draft_logits,
                   const int32_t *draft_tokens, const int32_t *num_draft,
                   const float *temperature, uint64_t seed, int batch, int total_draft,
                   int32_t *accepted_len, int32_t *committed_tokens, uint8_t *accept_flags,
                   void *stream);

/*
 * specverify_run_ex -- specverify_run plus optional inputs/outputs (each may be NULL):
 *   request_ids  [batch] int64: the "request" word of the Philox counter (so a
 *                request draws the same numbers in any batch position);
 *   p_y, q_y, u  [total_draft] float32: p_i(y_i), q_i(y_i) and u_i of every draft
 *                position of sampling requests (NaN for greedy/skipped ones);
 *   req_status   [batch] int32: the status bits that concern each request.
 */
int specverify_run_ex(specverify_t h, const void *target_logits, const void *draft_logits,
                      const int32_t *draft_tokens, const int32_t *num_draft,
                      const float *temperature, uint64_t seed, int batch, int total_draft,
                      int32_t *accepted_len, int32_t *committed_tokens, uint8_t *accept_flags,
                      const int64_t *request_ids, float *p_y, float *q_y, float *u,
                      int32_t *req_status, void *stream);

/*
 * specverify_run_truncated -- specverify_run on top-k / top-p truncated
 * distributions, applied alike to each request's target and draft rows.
 *
 * "Speculative Decoding: Medusa, MTP, EAGLE, DFlash, DDTree, and DSpark",
 * section 1: truncation must enter the acceptance test and the residual
 * consistently.  The rules and their thresholds are those of
 * specverify_truncate (top_k [batch] int32, top_p [batch] float32, same
 * meaning), but no truncated copy is written: before each wave of the round a
 * threshold pass stores one order-key threshold for every row that wave reads
 * (in the handle's scratch), and the wave reads every logit below its row's
 * threshold as -inf as it loads it; rows the round never reads get none.
 * The outputs are those of specverify_run on the rows specverify_truncate
 * writes (draft tokens must come from the truncated draft distributions).  A
 * top_p NaN or <= 0 keeps its request's rows whole and sets
 * SPECVERIFY_STATUS_BAD_TRUNC.  The other arguments are those of
 * specverify_run; the round has one more launch per wave (its threshold pass,
 * two CTAs per SM).
 */
int specverify_run_truncated(specverify_t h, const void *target_logits,
                             const void *draft_logits, const int32_t *draft_tokens,
                             const int32_t *num_draft, const float *temperature,
                             const int32_t *top_k, const float *top_p, uint64_t seed, int batch,
                             int total_draft, int32_t *accepted_len, int32_t *committed_tokens,
                             uint8_t *accept_flags, void *stream);

/*
 * specverify_run_trimmed -- verify per-request windows chosen from draft
 * confidences, in place in a full-window layout.
 *
 * "Speculative Decoding: Medusa, MTP, EAGLE, DFlash, DDTree, and DSpark",
 * section 5 (DSpark): with conditional confidence estimates c_i the estimated
 * probability of accepting through position j is s_j = prod_{i<=j} c_i, and
 * verifying a prefix of length k has estimated progress 1 + sum_{j<=k} s_j;
 * the scheduler asks whether another verification position is worth its
 * marginal cost, and compact verification executes only the selected
 * per-request windows.  Here request r verifies the k_r in [0, K_r] that
 * maximises 1 + sum_{j<=k} s_j - cost[r] * k (the shortest on ties; fp64),
 * i.e. a verify round with num_draft = k_r on the same rows: rows past
 * position k_r are never read, the bonus after k_r acceptances comes from
 * target row k_r.
 *   window       [batch] int32: K_r, the layout of the inputs (as num_draft in
 *                specverify_run: target rows K_r + 1, draft rows and tokens K_r);
 *   confidence   [total_draft] float32: c_i of each draft position of the
 *                layout, in [0, 1] (may be NULL when total_draft == 0);
 *   cost         [batch] float32: cost of one verified position, in units of
 *                expected progress (any value but NaN; <= 0 keeps every position);
 *   verified_k   [batch] int32 out: k_r (-1 when the confidences are invalid);
 *   p_y, q_y, u, req_status: as specverify_run_ex (nullable).
 * The other arguments and outputs are those of specverify_run; flags are 0
 * (and debug values NaN) past k_r.  A request with a confidence NaN or outside
 * [0, 1], or a NaN cost, is skipped with SPECVERIFY_STATUS_BAD_CONF.
 */
int specverify_run_trimmed(specverify_t h, const void *target_logits, const void *draft_logits,
                           const int32_t *draft_tokens, const int32_t *window,
                           const float *confidence, const float *cost, const float *temperature,
                           uint64_t seed, int batch, int total_draft, int32_t *verified_k,
                           int32_t *accepted_len, int32_t *committed_tokens,
                           uint8_t *accept_flags, float *p_y, float *q_y, float *u,
                           int32_t *req_status, void *stream);

/*
 * specverify_run_host -- the same verify round on HOST buffers (same shapes as
 * specverify_run; draft_logits may be NULL as there).  When both logits
 * buffers lie in pinned host memory that the device maps (cudaHostAlloc, or
 * cudaHostRegister with mapping, on a unified-address system) and the mode
 * (specverify_set_host_reads) is AUTO, the kernels read the logits where they
 * lie: only the rows the round needs cross to the GPU (over NVLink-C2C on
 * Grace-Blackwell), and the host buffers must stay unchanged until the call
 * returns.  Otherwise the logits are copied into the handle's device staging
 * first (asynchronous DMA from pinned memory).  The small inputs are copied
 * in, the three outputs copied back, and the call waits for `stream`.  Needs a
 * handle made with SPECVERIFY_CREATE_HOST_STAGING.
 */
int specverify_run_host(specverify_t h, const void *target_logits, const void *draft_logits,
                        const int32_t *draft_tokens, const int32_t *num_draft,
                        const float *temperature, uint64_t seed, int batch, int total_draft,
                        int32_t *accepted_len, int32_t *committed_tokens,
                        uint8_t *accept_flags, void *stream);

/* Limits of specverify_run_static. */
#define SPECVERIFY_STATIC_MAX_BATCH 256
#define SPECVERIFY_STATIC_MAX_K 7

/*
 * specverify_run_static -- the verify round of specverify_run without a handle
 * and without allocating anything: no cudaMalloc/cudaFree, no allocating
 * library routine.  The pages have no counterpart of this entry point.  It is
 * for callers that may not allocate device memory: a serving process that
 * reserves all of the GPU's memory for its own pool at start-up (KV cache and
 * weights), where a cudaMalloc would fail or steal from the pool, and
 * embedding runtimes whose rules forbid allocation once they are serving,
 * because an allocation can block on device-wide synchronisation.
 *
 * Scratch is one file-scope static device array of about 0.71 MiB, sized for
 * batch <= SPECVERIFY_STATIC_MAX_BATCH (256) and max_k <=
 * SPECVERIFY_STATIC_MAX_K (7) on a grid of at most 1024 CTAs.  On its first use
 * on a device the call takes the array's address (cudaGetSymbolAddress,
 * checked), sizes the kernel grids, and clears the array on `stream` (its
 * completion counters must start at zero); later calls on that device reuse
 * them.  Because that first call does this set-up, make it before any stream
 * capture begins.  Every other piece of scratch is reset by the round itself.
 *
 * Arguments as specverify_run, plus device, max_k (width of committed_tokens
 * is max_k + 1; every num_draft must lie in [0, max_k]), vocab and dtype.
 * Returns SPECVERIFY_ERR_TOO_LARGE, launching nothing, when batch or max_k
 * exceeds the limits; the other errors as specverify_run.  Status bits are
 * not reported (there is no handle); inputs that set them still skip their
 * requests (accepted_len = -1).
 *
 * There is one arena per device: calls that overlap in time -- on different
 * streams, or from different host threads without ordering -- race on it and
 * produce garbage.  Serialise them on one stream.
 */
int specverify_run_static(int device, int max_k, int vocab, int dtype,
                          const void *target_logits, const void *draft_logits,
                          const int32_t *draft_tokens, const int32_t *num_draft,
                          const float *temperature, uint64_t seed, int batch, int total_draft,
                          int32_t *accepted_len, int32_t *committed_tokens,
                          uint8_t *accept_flags, void *stream);

/* Wait for the handle's last stream and return the status bits of its last run
 * in *status_out (host pointer). */
int specverify_status(specverify_t h, int32_t *status_out);

/*
 * Round tags (test aid).  Each round tags its completion counters with a
 * 32-bit round number; before the number would wrap past 2^32 - 1 the
 * counters are cleared on the round's stream and numbering restarts at 1, so
 * a handle (or the static arena) serves any number of rounds.  These calls let
 * a test reach the wrap quickly: they wait for the device, clear the counters
 * and set the number the last round had, so the next round is tagged
 * epoch + 1 (epoch = 0xffffffff makes the next round clear and restart).
 * specverify_static_debug_set_epoch needs a completed specverify_run_static
 * on `device` (the arena's set-up) and returns SPECVERIFY_ERR_INVALID_ARG
 * before it.  Not for use while rounds are in flight.
 */
int specverify_debug_set_epoch(specverify_t h, uint32_t epoch);
int specverify_static_debug_set_epoch(int device, uint32_t epoch);

/*
 * specverify_set_timing_events -- measurement aid.  After this call, run number
 * i (counting from 0) records start_events[i % n] on its stream just before its
 * first launch and stop_events[i % n] just after its last.  The arrays hold cudaEvent_t values created
 * by the caller, n in [1, 64]; they are copied.  n = 0 turns recording off.
 */
int specverify_set_timing_events(specverify_t h, int n, void *const *start_events,
                                 void *const *stop_events);

/*
 * specverify_set_depth -- positions verified per wave launch.  A round reads
 * the rows of positions 0..A only when it decides one position per wave
 * (depth 1, the least traffic); a larger depth reads up to depth - 1 rows past
 * a rejection but needs fewer launches, which is faster for small batches.
 * depth in [1, max_k + 1] fixes it; 0 (the default) chooses per run from the
 * bytes of every row of the batch's verify window: max_k + 1 up to 192 MiB,
 * 2 up to 1 GiB, else 1.  Results do not depend on the depth.
 */
int specverify_set_depth(specverify_t h, int depth);

/* The depth a wave-schedule run of `batch` requests on h uses (the setting, or
 * the per-run choice above) in *depth_out. */
int specverify_wave_depth(specverify_t h, int batch, int *depth_out);

/*
 * specverify_set_schedule -- how a round is laid out on the GPU.  Results do
 * not depend on it.
 *   SPECVERIFY_SCHEDULE_WAVES: a wave launch per group of `depth` positions
 *     (specverify_set_depth), every request in lockstep;
 *   SPECVERIFY_SCHEDULE_AUTO (default): waves.
 * Any other value returns SPECVERIFY_ERR_INVALID_ARG.
 */
#define SPECVERIFY_SCHEDULE_AUTO 0
#define SPECVERIFY_SCHEDULE_WAVES 1
int specverify_set_schedule(specverify_t h, int schedule);

/*
 * specverify_set_host_reads -- how specverify_run_host gets the logits to the
 * GPU.  Results do not depend on it.
 *   SPECVERIFY_HOST_READS_AUTO (default): read in place when both logits
 *     buffers are pinned and mapped host memory, else staged copies;
 *   SPECVERIFY_HOST_READS_STAGE: always copy the whole window into the
 *     device staging first.
 * Returns SPECVERIFY_ERR_INVALID_ARG for another mode.
 */
#define SPECVERIFY_HOST_READS_AUTO 0
#define SPECVERIFY_HOST_READS_STAGE 1
int specverify_set_host_reads(specverify_t h, int mode);

/* How the last specverify_run_host on h got its logits: *in_place_out = 1 read
 * in place, 0 copied into staging, -1 no host run yet (or it returned before
 * choosing). */
int specverify_last_host_reads(specverify_t h, int *in_place_out);

/* Kernel launches a run of `batch` requests makes on handle h (for launch
 * accounting): the plan launch and one launch per wave of `depth` positions
 * (plus one for the last wave's correction draws when depth > 1), or the plan
 * and one cluster launch.  Waves with nothing left to do return at once.
 * Counts assume 16-byte aligned rows. */
int specverify_launches_per_run(specverify_t h, int batch, int *launches_out);

/*
 * specverify_metrics -- acceptance statistics of verify rounds, accumulated on
 * the device ("Speculative Decoding on AMD GPUs", "Monitor acceptance
 * behavior" and the appendix tables: mean accepted length MAL, overall
 * acceptance rate, per-position acceptance rates; the printed rows satisfy
 * MAL = 1 + the sum of the per-position rates, so MAL counts the round's
 * correction or bonus token as well).  Needs no handle; runs on the current
 * device, asynchronously on `stream`, one single-CTA launch.  Device pointers:
 *   accepted_len [batch] int32  a round's output (-1: request skipped);
 *   num_draft    [batch] int32  the round's k_r;
 *   hist     [max_k + 2] uint64 in/out: hist[a] += rounds with A = a (a <= max_k;
 *                               larger A counts in hist[max_k]), hist[max_k + 1]
 *                               += skipped requests;
 *   proposed [max_k] uint64     in/out: += rounds with k_r > j (k_r counts up to max_k);
 *   accepted [max_k] uint64     in/out: += rounds with A_r > j;
 *   summary  [max_k + 4] double out, may be NULL: from the counts after this
 *                               batch: MAL = 1 + sum_a a hist[a] / rounds, the
 *                               acceptance rate sum(accepted) / sum(proposed), the
 *                               max_k per-position rates accepted[j] / proposed[j],
 *                               the number of rounds and of skipped requests
 *                               (NaN where a denominator is 0).
 * The counts are running totals owned by the caller (zero them to start);
 * they are added to with atomics.  proposed and accepted may be NULL when
 * max_k = 0.  Returns SPECVERIFY_ERR_INVALID_ARG on a bad size or pointer
 * (max_k in [0, 31]), _CUDA if the launch fails.
 */
int specverify_metrics(const int32_t *accepted_len, const int32_t *num_draft, int batch,
                       int max_k, uint64_t *hist, uint64_t *proposed, uint64_t *accepted,
                       double *summary, void *stream);

/*
 * specverify_truncate -- top-k / top-p truncation applied alike to the target
 * and draft rows of a ragged batch, before a verify round.
 *
 * "Speculative Decoding: Medusa, MTP, EAGLE, DFlash, DDTree, and DSpark",
 * section 1: temperature, truncation, penalties and grammar constraints must be
 * incorporated consistently -- the acceptance test and the residual must use
 * the distributions the target and the drafter actually sample from.  Per
 * request r (T_r > 0):
 *   top_k[r] = K (0 < K < V): keep every logit >= the K-th largest (ties kept);
 *   top_p[r] = P (0 < P < 1): on the top-k survivors renormalised
 *     (softmax(x / T)), keep a logit while the mass of the survivors with a
 *     strictly larger logit is below P;
 *   kept logits are copied to the output, the others become -inf, so softmax
 *   of an output row is the truncated, renormalised distribution and
 *   specverify_run on the outputs verifies the truncated distributions (draft
 *   tokens must have been sampled from the truncated draft distribution).
 * K <= 0 or K >= V turns top-k off, P >= 1 turns top-p off; rows of greedy
 * requests (T = 0) and rows holding NaN are copied; a P NaN or <= 0 copies the
 * rows and sets SPECVERIFY_STATUS_BAD_TRUNC in *status (nullable device int32,
 * OR-ed).  The top-k threshold is exact.  The top-p masses are fp32 weights
 * 2^(c (x - max)): for bf16 rows, one per exact logit value times its count,
 * summed in fp64 in a fixed order; otherwise summed as 2^-40 fixed-point
 * integers.  Neither depends on the order of atomics, and a top-p decision
 * within about 1e-6 of its threshold can differ from an exact computation.
 * Layout as specverify_run: target_in/_out [batch + total_draft, vocab],
 * draft_in/_out [total_draft, vocab] (both NULL, or both given), dtype F32 or
 * BF16, device pointers on the current device; asynchronous on stream, one
 * launch (two CTAs per SM, a few passes over each row through L2).
 */
int specverify_truncate(int dtype, int vocab, const void *target_in, const void *draft_in,
                        const int32_t *num_draft, const float *temperature, const int32_t *top_k,
                        const float *top_p, int batch, int total_draft, void *target_out,
                        void *draft_out, int32_t *status, void *stream);

/*
 * Greedy verification of drafted token trees.
 *
 * "Speculative Decoding: Medusa, MTP, EAGLE, DFlash, DDTree, and DSpark",
 * section 5 (DDTree): the tree uses depth-based positions and ancestor-only
 * attention; verification walks the target's selected tokens, and when no
 * child matches, that target token becomes the next bonus token; only the
 * accepted path survives.  Selection is the target argmax (lowest index on
 * ties); section 1 of the same page gives no sampling rule for trees, so none
 * is offered.
 *
 * Layout (row-major, one row = V logits; device pointers, caller-owned):
 *   request r has n_r = num_nodes[r] nodes, 0 <= n_r <= max_nodes;
 *   node_tokens[n_off(r) + i], parent[n_off(r) + i]  token and parent of node i,
 *       parent in [-1, i) (-1: child of the root, the last committed token),
 *       n_off(r) = sum_{s<r} n_s;
 *   target_logits[t_off(r) + 0]      the target's output at the root,
 *   target_logits[t_off(r) + 1 + i]  its output after node i,
 *       t_off(r) = sum_{s<r} (n_s + 1): batch + total_nodes rows in all.
 * The walk: from the root, tau = argmax of the current node's row; the
 * lowest-index child of the current node whose token is tau is accepted and
 * becomes current; when none is, tau is the bonus token.
 * Outputs:
 *   accepted_len [batch] int32       A_r, the accepted nodes (-1: skipped);
 *   path         [batch, max_nodes]  accepted node indices by depth, -1 after;
 *   committed    [batch, max_nodes+1] accepted tokens then the bonus, -1 after;
 *   req_status   [batch] int32 (nullable) status bits of each request.
 * Device-side problems set status bits (specverify_tree_status) and skip the
 * request: a parent out of range (BAD_PARENT), a token outside [0, V)
 * (BAD_TOKEN), NaN/+inf or no finite logit in a row the walk reads
 * (NONFINITE); a num_nodes outside [0, max_nodes] (BAD_K) or a sum other
 * than total_nodes (BAD_TOTAL) skips the batch.  Only the rows of the
 * accepted path are read (A_r + 1 rows of request r), by one block of threads
 * per tree walking from the root (two launches, asynchronous on stream).
 */
/* max_batch in [1, 4096], max_nodes in [0, 1024], vocab in [1, 2^30]; allocates
 * the scratch (offsets and status words) now. */
int specverify_tree_create(specverify_tree_t *out, int device, int max_batch, int max_nodes,
                           int vocab, int dtype);
/* batch in [0, max_batch], total_nodes = host copy of sum num_nodes. */
int specverify_tree_run(specverify_tree_t h, const void *target_logits, const int32_t *num_nodes,
                        const int32_t *parent, const int32_t *node_tokens, int batch,
                        int total_nodes, int32_t *accepted_len, int32_t *path,
                        int32_t *committed, int32_t *req_status, void *stream);
/* Waits for the last run's stream and returns its status bits. */
int specverify_tree_status(specverify_tree_t h, int32_t *status_out);
int specverify_tree_destroy(specverify_tree_t h);

/* Free the handle and its device memory.  Further use returns _ERR_DESTROYED
 * only while the memory of the freed handle is not reused; do not use it. */
int specverify_destroy(specverify_t h);

/* Static English text for a return code. */
const char *specverify_error_string(int code);

#ifdef __cplusplus
}
#endif

#endif /* SPECVERIFY_H */
