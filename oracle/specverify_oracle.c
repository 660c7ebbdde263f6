/*
 * specverify_oracle.c -- plain, slow, single-threaded CPU oracle for the
 * target-side verify step of speculative sampling.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check and
 * the benchmark's CPU-baseline / reference leg load this file.  The CUDA
 * library never links, includes or calls it, and it shares no code with the
 * CUDA library (its own Philox, its own softmax, its own scan and race).
 *
 * Everything is computed in double precision from logits that are read
 * exactly (fp32 -> double and bf16 -> fp32 -> double are lossless).  Each step
 * follows the passage of the pages it cites:
 *
 *   [SD]  "Speculative Decoding: Medusa, MTP, EAGLE, DFlash, DDTree, and
 *         DSpark", section 1 "What Speculative Decoding Actually Guarantees":
 *         the worked example (draft A B C D, C rejected, commit A B R), the
 *         acceptance probability alpha_i(y_i) = min(1, p_i(y_i)/q_i(y_i)),
 *         the correction drawn from the normalised positive residual
 *         [p_i - q_i]_+, the bonus token drawn from the target when every
 *         draft survives, greedy equivalence (accepted tokens follow the
 *         target argmax) and the rule that temperature enters p and q
 *         consistently.
 *   [SD2] same page, section 2 "The Cost Model Behind the Comparison": A is
 *         the accepted draft-prefix length, excluding the correction/bonus.
 *   [AMD] "Speculative Decoding on AMD GPUs" (vLLM blog), "Core idea of
 *         speculative decoding": verification runs left to right and every
 *         candidate after the first rejection is discarded.
 *
 * Randomness (not fixed by the pages; the reading this library takes):
 *   Philox4x32-10 from Salmon, Moraes, Dror and Shaw, "Parallel Random
 *   Numbers: As Easy as 1, 2, 3" (SC'11), keyed by the 64-bit seed
 *   (key = seed low word, seed high word) with the counter
 *       (floor(v/4), position, request low word, stream | request high << 8)
 *   and output word v mod 4.  Stream 0 gives the acceptance uniform of a
 *   position (v = 0); stream 1 the exponentials of the correction or bonus
 *   draw, one per vocab id v.
 *     u      = (w >> 8) * 2^-24                 in [0, 1)       (exact in fp32)
 *     E      = -ln((w + 1/2) * 2^-32)           in (1.2e-10, 22.9)
 *   A categorical draw from weights w_v >= 0 is the exponential race
 *     token  v* = argmin_{v: w_v > 0} E_v / w_v,   lowest index on ties,
 *   E_v from the stream-1 word of vocab id v at the draw's (request,
 *   position).  E_v / w_v ~ Exp(w_v), so P(v* = v) = w_v / sum_u w_u.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <float.h>

#define ORC_DTYPE_F32 0
#define ORC_DTYPE_BF16 1

/* Status bits (same meaning as the library's; defined here independently). */
#define ORC_BAD_TOKEN 1u      /* a draft token outside [0, V) */
#define ORC_BAD_K 2u          /* a num_draft outside [0, max_k] */
#define ORC_BAD_TEMP 4u       /* temperature NaN, negative, infinite or subnormal */
#define ORC_NONFINITE 8u      /* a read row holds NaN/+inf or no finite logit */
#define ORC_BAD_TOTAL 16u     /* sum of num_draft differs from total_draft */
#define ORC_NO_DRAFT 64u      /* T > 0 but no draft logits were given */

/* Race kinds reported per request. */
#define ORC_RACE_NONE 0
#define ORC_RACE_GREEDY 1     /* token = target argmax (T = 0) */
#define ORC_RACE_BONUS 2      /* every draft accepted: race on p_k */
#define ORC_RACE_RESIDUAL 3   /* race on [p_j - q_j]_+ */
#define ORC_RACE_FALLBACK 4   /* residual has no mass: race on p_j */

/* ------------------------------------------------------------------------ */
/* Philox4x32-10 (SC'11): ten rounds of two 32x32->64 multiplies; the key is  */
/* bumped by the Weyl constants between rounds.                               */
/* ------------------------------------------------------------------------ */
void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4])
{
    const uint32_t mul0 = 0xD2511F53u, mul1 = 0xCD9E8D57u;
    const uint32_t weyl0 = 0x9E3779B9u, weyl1 = 0xBB67AE85u;
    uint32_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += weyl0;
            k1 += weyl1;
        }
        uint64_t prod0 = (uint64_t)mul0 * (uint64_t)x0;
        uint64_t prod1 = (uint64_t)mul1 * (uint64_t)x2;
        uint32_t hi0 = (uint32_t)(prod0 >> 32), lo0 = (uint32_t)prod0;
        uint32_t hi1 = (uint32_t)(prod1 >> 32), lo1 = (uint32_t)prod1;
        uint32_t y0 = hi1 ^ x1 ^ k0;
        uint32_t y1 = lo1;
        uint32_t y2 = hi0 ^ x3 ^ k1;
        uint32_t y3 = lo0;
        x0 = y0; x1 = y1; x2 = y2; x3 = y3;
    }
    out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

/* One 32-bit random word for (seed, stream, request, position, v). */
uint32_t orc_random_word(uint64_t seed, uint32_t stream, uint64_t request,
                         uint32_t position, uint32_t v)
{
    uint32_t key[2] = {(uint32_t)(seed & 0xFFFFFFFFu), (uint32_t)(seed >> 32)};
    uint32_t ctr[4] = {v / 4u, position, (uint32_t)(request & 0xFFFFFFFFu),
                       (stream & 0xFFu) | ((uint32_t)(request >> 32) << 8)};
    uint32_t out[4];
    orc_philox4x32_10(ctr, key, out);
    return out[v % 4u];
}

/* Acceptance uniform: the top 24 bits of the word, scaled into [0, 1). */
double orc_uniform_accept(uint32_t w)
{
    return (double)(w >> 8) * 0x1p-24;
}

/* Race exponential: E = -ln(U) with U = (w + 1/2) * 2^-32 strictly in (0, 1). */
double orc_exponential(uint32_t w)
{
    double u = ((double)w + 0.5) * 0x1p-32;
    return -log(u);
}

/* ------------------------------------------------------------------------ */
/* Logit access: row-major [rows, V]; fp32 or bf16 (raw 16-bit patterns).     */
/* ------------------------------------------------------------------------ */
static double logit_at(const void *base, int dtype, size_t row, int vocab, int v)
{
    size_t idx = row * (size_t)vocab + (size_t)v;
    if (dtype == ORC_DTYPE_F32)
        return (double)((const float *)base)[idx];
    uint32_t bits = (uint32_t)((const uint16_t *)base)[idx] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* A row is usable when it has no NaN, no +inf and at least one finite logit. */
static int row_is_valid(const void *base, int dtype, size_t row, int vocab)
{
    int any_finite = 0;
    for (int v = 0; v < vocab; ++v) {
        double x = logit_at(base, dtype, row, vocab, v);
        if (isnan(x) || x == INFINITY)
            return 0;
        if (isfinite(x))
            any_finite = 1;
    }
    return any_finite;
}

/* p = softmax(x / T) over the row, in double ([SD] section 1: temperature  */
/* enters p and q alike).  A logit of -inf gets probability 0.              */
void orc_softmax(const void *base, int dtype, size_t row, int vocab, double temperature,
                 double *p)
{
    double m = -INFINITY;
    for (int v = 0; v < vocab; ++v) {
        double z = logit_at(base, dtype, row, vocab, v) / temperature;
        if (z > m)
            m = z;
    }
    double total = 0.0;
    for (int v = 0; v < vocab; ++v) {
        double z = logit_at(base, dtype, row, vocab, v) / temperature;
        p[v] = exp(z - m);
        total += p[v];
    }
    for (int v = 0; v < vocab; ++v)
        p[v] /= total;
}

/* Greedy choice: the first index holding the row maximum ([SD] section 1, */
/* greedy equivalence).                                                     */
int orc_argmax(const void *base, int dtype, size_t row, int vocab)
{
    int best = 0;
    double best_x = logit_at(base, dtype, row, vocab, 0);
    for (int v = 1; v < vocab; ++v) {
        double x = logit_at(base, dtype, row, vocab, v);
        if (x > best_x) {
            best_x = x;
            best = v;
        }
    }
    return best;
}

/* Exponential race over weights w (length V): the token is
 *     v* = argmin_{v: w_v > 0} E_v / w_v,
 * E_v the race exponential of the stream-1 word at (request, position, v),
 * lowest index on ties.  With E_v iid Exp(1), E_v / w_v is exponential with
 * rate w_v, so P(v* = v) = w_v / sum_u w_u: a categorical draw from w that
 * needs no normalisation and does not depend on the order the ids are
 * visited in.  keys_out [V] (nullable) receives every key (+inf where the
 * weight is not positive); *margin (nullable) gets second / best - 1.
 * Returns the winner, or -1 when no weight is positive. */
static int race(const double *w, int vocab, uint64_t seed, uint64_t request, uint32_t position,
                double *keys_out, double *margin)
{
    int winner = -1;
    double best = INFINITY, second = INFINITY;
    for (int v = 0; v < vocab; ++v) {
        double key = INFINITY;
        if (w[v] > 0.0)
            key = orc_exponential(orc_random_word(seed, 1u, request, position, (uint32_t)v)) / w[v];
        if (keys_out)
            keys_out[v] = key;
        if (!(w[v] > 0.0))
            continue;
        if (key < best) {
            second = best;
            best = key;
            winner = v;
        } else if (key < second) {
            second = key;
        }
    }
    if (margin)
        *margin = winner < 0 ? INFINITY : second / best - 1.0;
    return winner;
}

/* Temperature is usable when it is 0 (greedy) or a normal, finite positive. */
static int temperature_ok(float t)
{
    if (isnan(t) || isinf(t) || t < 0.0f)
        return 0;
    return t == 0.0f || t >= FLT_MIN;
}

/*
 * The verify step over a ragged batch.
 *
 * Layout: request r owns k_r = num_draft[r] draft positions.  Its target rows
 * are rows tgt_off(r) .. tgt_off(r)+k_r of target_logits with
 * tgt_off(r) = sum_{s<r} (k_s + 1); its draft rows are drf_off(r) ..
 * drf_off(r)+k_r-1 of draft_logits, and its draft tokens are
 * draft_tokens[drf_off(r) + i], with drf_off(r) = sum_{s<r} k_s.
 *
 * Outputs: accepted_len[r] = A_r ([SD2]); committed[r*(max_k+1) + i] holds the
 * accepted draft tokens for i < A_r, the correction or bonus token at i = A_r,
 * and -1 after it; accept_flags[drf_off(r) + i] = (i < A_r).  A request whose
 * inputs are invalid gets accepted_len -1, a committed row of -1 and flags 0.
 *
 * Debug outputs (all nullable): p_y/q_y/u per decided draft position (0..A)
 * of sampling requests, NaN elsewhere; accept_margin = (p - u q) / max(p, u q);
 * race_kind/race_pos/race_margin per request (race_margin: the relative gap
 * of the draw's decisive comparisons); req_status per request.
 * Returns the OR of all status bits.
 */
uint32_t orc_verify(int dtype, int vocab, int batch, int max_k, int total_draft,
                    const void *target_logits, const void *draft_logits,
                    const int32_t *draft_tokens, const int32_t *num_draft,
                    const float *temperature, const int64_t *request_ids, uint64_t seed,
                    int32_t *accepted_len, int32_t *committed, uint8_t *accept_flags,
                    double *p_y, double *q_y, double *u_out, double *accept_margin,
                    int32_t *race_kind, int32_t *race_pos, double *race_margin,
                    int32_t *req_status)
{
    const int width = max_k + 1;
    uint32_t status = 0;

    for (int r = 0; r < batch; ++r) {
        accepted_len[r] = -1;
        for (int i = 0; i < width; ++i)
            committed[(size_t)r * width + i] = -1;
        if (race_kind) race_kind[r] = ORC_RACE_NONE;
        if (race_pos) race_pos[r] = -1;
        if (race_margin) race_margin[r] = NAN;
        if (req_status) req_status[r] = 0;
    }
    for (int d = 0; d < total_draft; ++d) {
        accept_flags[d] = 0;
        if (p_y) p_y[d] = NAN;
        if (q_y) q_y[d] = NAN;
        if (u_out) u_out[d] = NAN;
        if (accept_margin) accept_margin[d] = NAN;
    }

    /* The layout is only trustworthy when every k_r is in range and they  */
    /* add up to total_draft; otherwise nothing is verified.               */
    long long sum_k = 0;
    for (int r = 0; r < batch; ++r) {
        if (num_draft[r] < 0 || num_draft[r] > max_k)
            status |= ORC_BAD_K;
        sum_k += num_draft[r];
    }
    if (status & ORC_BAD_K)
        return status;
    if (sum_k != total_draft)
        return status | ORC_BAD_TOTAL;

    double *p = (double *)malloc(sizeof(double) * (size_t)(vocab > 0 ? vocab : 1));
    double *q = (double *)malloc(sizeof(double) * (size_t)(vocab > 0 ? vocab : 1));
    double *w = (double *)malloc(sizeof(double) * (size_t)(vocab > 0 ? vocab : 1));

    size_t tgt_off = 0, drf_off = 0;
    for (int r = 0; r < batch; ++r) {
        const int k = num_draft[r];
        const float t = temperature[r];
        const uint64_t req = request_ids ? (uint64_t)request_ids[r] : (uint64_t)r;
        uint32_t rs = 0;

        if (!temperature_ok(t))
            rs |= ORC_BAD_TEMP;
        for (int i = 0; i < k; ++i) {
            int32_t y = draft_tokens[drf_off + i];
            if (y < 0 || y >= vocab)
                rs |= ORC_BAD_TOKEN;
        }
        const int greedy = (t == 0.0f);
        if (!rs && !greedy && k > 0 && draft_logits == NULL)
            rs |= ORC_NO_DRAFT;
        if (rs) {
            status |= rs;
            if (req_status) req_status[r] = (int32_t)rs;
            tgt_off += (size_t)k + 1;
            drf_off += (size_t)k;
            continue;
        }

        /* Positions are verified left to right and nothing after the first  */
        /* rejection is kept ([SD] section 1, [AMD]), so a round reads the     */
        /* rows of positions 0..A (and the bonus row when A = k) and no more. */
        /* A row it reads with NaN, +inf or no finite logit skips the request. */
        int accepted = 0;
        int token = -1;
        int bad_row = 0;
        if (greedy) {
            /* Greedy equivalence: keep y_i while it equals the target argmax; */
            /* the committed extra token is the target argmax at position A.   */
            for (;;) {
                if (!row_is_valid(target_logits, dtype, tgt_off + accepted, vocab)) {
                    bad_row = 1;
                    break;
                }
                const int a = orc_argmax(target_logits, dtype, tgt_off + accepted, vocab);
                if (accepted < k && draft_tokens[drf_off + accepted] == a) {
                    ++accepted;
                    continue;
                }
                token = a;
                break;
            }
            if (race_kind) race_kind[r] = ORC_RACE_GREEDY;
            if (race_pos) race_pos[r] = accepted;
        } else {
            const double temp = (double)t;
            /* Accept y_i with probability min(1, p_i(y_i)/q_i(y_i)), tested as */
            /* u_i q_i(y_i) < p_i(y_i); stop at the first rejection.             */
            int rejected = 0;
            for (int i = 0; i < k && !rejected; ++i) {
                if (!row_is_valid(target_logits, dtype, tgt_off + i, vocab) ||
                    !row_is_valid(draft_logits, dtype, drf_off + i, vocab)) {
                    bad_row = 1;
                    break;
                }
                const int32_t y = draft_tokens[drf_off + i];
                orc_softmax(target_logits, dtype, tgt_off + i, vocab, temp, p);
                orc_softmax(draft_logits, dtype, drf_off + i, vocab, temp, q);
                const double u = orc_uniform_accept(orc_random_word(seed, 0u, req, (uint32_t)i, 0u));
                const double lhs = u * q[y], rhs = p[y];
                if (p_y) p_y[drf_off + i] = rhs;
                if (q_y) q_y[drf_off + i] = q[y];
                if (u_out) u_out[drf_off + i] = u;
                if (accept_margin) {
                    double scale = lhs > rhs ? lhs : rhs;
                    accept_margin[drf_off + i] = scale > 0.0 ? (rhs - lhs) / scale : 0.0;
                }
                if (lhs < rhs)
                    ++accepted;
                else
                    rejected = 1;
            }
            double gap = NAN;
            if (!bad_row && accepted == k) {
                /* Every draft survived: one more token from the target p_k. */
                if (!row_is_valid(target_logits, dtype, tgt_off + k, vocab)) {
                    bad_row = 1;
                } else {
                    orc_softmax(target_logits, dtype, tgt_off + k, vocab, temp, p);
                    token = race(p, vocab, seed, req, (uint32_t)k, NULL, &gap);
                    if (race_kind) race_kind[r] = ORC_RACE_BONUS;
                }
            } else if (!bad_row) {
                /* First rejection at j = A: draw from [p_j - q_j]_+, normalised */
                /* (normalisation does not change the race winner).             */
                const int j = accepted;
                orc_softmax(target_logits, dtype, tgt_off + j, vocab, temp, p);
                orc_softmax(draft_logits, dtype, drf_off + j, vocab, temp, q);
                for (int v = 0; v < vocab; ++v)
                    w[v] = p[v] > q[v] ? p[v] - q[v] : 0.0;
                token = race(w, vocab, seed, req, (uint32_t)j, NULL, &gap);
                if (token >= 0) {
                    if (race_kind) race_kind[r] = ORC_RACE_RESIDUAL;
                } else {
                    /* p <= q everywhere means p == q: draw from p instead. */
                    token = race(p, vocab, seed, req, (uint32_t)j, NULL, &gap);
                    if (race_kind) race_kind[r] = ORC_RACE_FALLBACK;
                }
            }
            if (race_pos) race_pos[r] = accepted;
            if (race_margin) race_margin[r] = gap;
        }
        if (bad_row) {
            status |= ORC_NONFINITE;
            if (req_status) req_status[r] = (int32_t)ORC_NONFINITE;
            if (race_kind) race_kind[r] = ORC_RACE_NONE;
            if (race_pos) race_pos[r] = -1;
            if (race_margin) race_margin[r] = NAN;
            for (int i = 0; i < k; ++i) {
                if (p_y) p_y[drf_off + i] = NAN;
                if (q_y) q_y[drf_off + i] = NAN;
                if (u_out) u_out[drf_off + i] = NAN;
                if (accept_margin) accept_margin[drf_off + i] = NAN;
            }
            tgt_off += (size_t)k + 1;
            drf_off += (size_t)k;
            continue;
        }

        accepted_len[r] = accepted;
        for (int i = 0; i < accepted; ++i)
            committed[(size_t)r * width + i] = draft_tokens[drf_off + i];
        committed[(size_t)r * width + accepted] = token;
        for (int i = 0; i < k; ++i)
            accept_flags[drf_off + i] = (uint8_t)(i < accepted);

        tgt_off += (size_t)k + 1;
        drf_off += (size_t)k;
    }
    free(p);
    free(q);
    free(w);
    return status;
}

/*
 * Keys of one request's correction/bonus draw, so a test can check any token:
 * keys [V] as in race().  kind: ORC_RACE_BONUS or ORC_RACE_FALLBACK (weights
 * p from target_row), ORC_RACE_RESIDUAL (weights [p - q]_+ from target_row and
 * draft_row).  Rows are single rows [V].  Returns the winner.
 */
int orc_race_keys(int dtype, int vocab, const void *target_row, const void *draft_row,
                  float temperature, uint64_t seed, uint64_t request, int position, int kind,
                  double *keys)
{
    double *p = (double *)malloc(sizeof(double) * (size_t)vocab);
    double *q = (double *)malloc(sizeof(double) * (size_t)vocab);
    double *w = (double *)malloc(sizeof(double) * (size_t)vocab);
    orc_softmax(target_row, dtype, 0, vocab, (double)temperature, p);
    int winner;
    if (kind == ORC_RACE_RESIDUAL) {
        orc_softmax(draft_row, dtype, 0, vocab, (double)temperature, q);
        for (int v = 0; v < vocab; ++v)
            w[v] = p[v] > q[v] ? p[v] - q[v] : 0.0;
        winner = race(w, vocab, seed, request, (uint32_t)position, keys, NULL);
    } else {
        winner = race(p, vocab, seed, request, (uint32_t)position, keys, NULL);
    }
    free(p);
    free(q);
    free(w);
    return winner;
}

/* The race over explicit weights (for tests): returns the winner. */
int orc_race_weights(const double *w, int vocab, uint64_t seed, uint64_t request, int position,
                     double *keys)
{
    return race(w, vocab, seed, request, (uint32_t)position, keys, NULL);
}

/* ------------------------------------------------------------------------ */
/* Acceptance statistics of verify rounds.                                   */
/*                                                                          */
/* [AMD] "Monitor acceptance behavior" names the signals: mean accepted      */
/* length (draft tokens committed per round), overall acceptance rate (the   */
/* share of proposed draft tokens accepted) and per-position acceptance      */
/* rate; its appendix tables print MAL = 1 + the sum of the per-position     */
/* rates, i.e. MAL counts the target's own token of the round as well.       */
/* This adds one batch of round outputs to running counts:                   */
/*   hist[a]        rounds that accepted a draft tokens (a = 0..max_k),      */
/*   hist[max_k+1]  requests that were skipped (accepted_len = -1),          */
/*   proposed[j]    rounds with a draft at position j  (num_draft > j),      */
/*   accepted[j]    rounds that accepted position j    (accepted_len > j).   */
/* A num_draft outside [0, max_k] counts only as far as max_k.               */
/* ------------------------------------------------------------------------ */
void orc_metrics(int batch, int max_k, const int32_t *accepted_len, const int32_t *num_draft,
                 uint64_t *hist, uint64_t *proposed, uint64_t *accepted)
{
    for (int r = 0; r < batch; ++r) {
        const int a = accepted_len[r];
        if (a < 0) {
            hist[max_k + 1] += 1;
            continue;
        }
        hist[a <= max_k ? a : max_k] += 1;
        int k = num_draft[r];
        if (k > max_k) k = max_k;
        for (int j = 0; j < k; ++j) {
            proposed[j] += 1;
            if (a > j) accepted[j] += 1;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Greedy tree verification.                                                */
/*                                                                          */
/* [SD] section 5, "DDTree: Build a Tree from Parallel Marginals": the      */
/* drafted tree uses depth-based positions and ancestor-only attention;     */
/* verification walks the target's selected tokens, and when no child       */
/* matches, that target token becomes the next bonus token; only the        */
/* accepted path survives.  [SD] section 1 gives no sampling rule for trees */
/* (the single-chain formula is not a tree algorithm), so only greedy       */
/* selection (the target argmax, lowest index on ties) is defined here.     */
/*                                                                          */
/* Request r has n_r draft nodes, 0 <= n_r <= max_nodes; node i has token   */
/* tokens[i] and parent[i] in [-1, i) (-1: a child of the root, the last    */
/* committed token).  Its n_r + 1 target rows are consecutive, starting at  */
/* row sum_{s<r} (n_s + 1): row 0 is the target's output at the root, row   */
/* 1 + i its output after node i.  Node arrays start at sum_{s<r} n_s.      */
/*                                                                          */
/* The walk: at the current node (the root first) tau = argmax of its row;  */
/* the lowest-index child of the current node whose token is tau is         */
/* accepted and becomes current; when none is, tau is the bonus token and   */
/* the walk ends.  Outputs: accepted_len[r] = A (accepted nodes),           */
/* path[r * max_nodes + d] the accepted node at depth d (d < A, else -1),   */
/* committed[r * (max_nodes + 1) + d] the accepted tokens then the bonus    */
/* (d <= A, else -1).  A request whose parents or tokens are out of range,  */
/* or whose walk reads a row with NaN, +inf or no finite logit, is skipped  */
/* (accepted_len -1, outputs -1) with its status bit; a num_nodes outside   */
/* [0, max_nodes], or a total other than total_nodes, skips the batch.      */
/* ------------------------------------------------------------------------ */
#define ORC_BAD_PARENT 32u

uint32_t orc_tree_greedy(int dtype, int vocab, int batch, int max_nodes, int total_nodes,
                         const void *target, const int32_t *num_nodes, const int32_t *parent,
                         const int32_t *tokens, int32_t *accepted_len, int32_t *path,
                         int32_t *committed, int32_t *req_status)
{
    uint32_t status = 0;
    const int pw = max_nodes, cw = max_nodes + 1;
    for (int r = 0; r < batch; ++r) {
        accepted_len[r] = -1;
        for (int d = 0; d < pw; ++d) path[(size_t)r * pw + d] = -1;
        for (int d = 0; d < cw; ++d) committed[(size_t)r * cw + d] = -1;
        if (req_status) req_status[r] = 0;
    }
    long long total = 0;
    for (int r = 0; r < batch; ++r) {
        if (num_nodes[r] < 0 || num_nodes[r] > max_nodes) status |= ORC_BAD_K;
        total += num_nodes[r];
    }
    if (!status && total != total_nodes) status |= ORC_BAD_TOTAL;
    if (status) {
        for (int r = 0; r < batch; ++r)
            if (req_status) req_status[r] = (int32_t)status;
        return status;
    }
    size_t t_off = 0, n_off = 0;
    for (int r = 0; r < batch; ++r) {
        const int n = num_nodes[r];
        const int32_t *par = parent + n_off, *tok = tokens + n_off;
        uint32_t rs = 0;
        for (int i = 0; i < n; ++i) {
            if (par[i] < -1 || par[i] >= i) rs |= ORC_BAD_PARENT;
            if (tok[i] < 0 || tok[i] >= vocab) rs |= ORC_BAD_TOKEN;
        }
        int cur = -1, a = 0;
        int32_t *pth = path + (size_t)r * pw, *com = committed + (size_t)r * cw;
        while (!rs) {
            const size_t row = t_off + (size_t)(cur + 1);
            if (!row_is_valid(target, dtype, row, vocab)) {
                rs |= ORC_NONFINITE;
                break;
            }
            const int tau = orc_argmax(target, dtype, row, vocab);
            int child = -1;
            for (int i = 0; i < n; ++i)
                if (par[i] == cur && tok[i] == tau) {
                    child = i;
                    break;
                }
            com[a] = tau;
            if (child < 0)
                break;
            pth[a] = child;
            ++a;
            cur = child;
        }
        if (rs) {
            for (int d = 0; d < pw; ++d) pth[d] = -1;
            for (int d = 0; d < cw; ++d) com[d] = -1;
            status |= rs;
        } else {
            accepted_len[r] = a;
        }
        if (req_status) req_status[r] = (int32_t)rs;
        t_off += (size_t)n + 1;
        n_off += (size_t)n;
    }
    return status;
}

/* ------------------------------------------------------------------------ */
/* Confidence-based window trimming.                                        */
/*                                                                          */
/* [SD] section 5, "DSpark: Dependencies Plus a Verification Budget": with  */
/* conditional confidence estimates c_i, the estimated probability of       */
/* accepting through position j is s_j = prod_{i<=j} c_i, and verifying a   */
/* prefix of length k has estimated progress 1 + sum_{j<=k} s_j; the        */
/* scheduler asks whether another verification position is worth its       */
/* marginal cost.  Reading taken: with a cost of `cost` (units of progress) */
/* per verified position, the window is the k in [0, K] that maximises      */
/* 1 + sum_{j<=k} s_j - cost * k, the shortest on ties.  Request r's        */
/* confidences are conf[d_off(r) + i], i < K_r (the window's layout).       */
/* A confidence that is NaN or outside [0, 1], or a NaN cost, sets          */
/* ORC_BAD_CONF and gives k = -1.                                           */
/* ------------------------------------------------------------------------ */
#define ORC_BAD_CONF 512u

uint32_t orc_trim(int batch, const int32_t *window, const float *conf, const float *cost,
                  int32_t *k_out)
{
    uint32_t status = 0;
    size_t off = 0;
    for (int r = 0; r < batch; ++r) {
        const int K = window[r];
        const double lam = (double)cost[r];
        int bad = isnan(lam);
        for (int i = 0; i < K; ++i) {
            const double c = (double)conf[off + (size_t)i];
            if (!(c >= 0.0 && c <= 1.0))
                bad = 1;
        }
        if (bad) {
            k_out[r] = -1;
            status |= ORC_BAD_CONF;
        } else {
            /* the objective, evaluated for every k; the first maximum wins */
            double best = 1.0, s = 1.0, value = 1.0;
            int best_k = 0;
            for (int j = 1; j <= K; ++j) {
                s *= (double)conf[off + (size_t)(j - 1)];
                value += s - lam;
                if (value > best) {
                    best = value;
                    best_k = j;
                }
            }
            k_out[r] = best_k;
        }
        off += (size_t)(K > 0 ? K : 0);
    }
    return status;
}

/* ------------------------------------------------------------------------ */
/* Top-k / top-p truncation, applied alike to the target and draft rows.    */
/*                                                                          */
/* [SD] section 1: temperature, truncation, penalties and grammar           */
/* constraints must be incorporated consistently -- the acceptance test and */
/* the residual must use the distributions the target and the drafter       */
/* actually sample from.  Readings taken (the page names no rule):          */
/*   temperature first: p = softmax(x / T);                                 */
/*   top-k (0 < K < V): keep every logit >= the K-th largest logit (ties    */
/*     with it are kept);                                                   */
/*   top-p (0 < P < 1), on the top-k survivors renormalised: keep v when    */
/*     the mass of the survivors with a strictly larger logit is below P    */
/*     (the most probable token is always kept);                            */
/*   the kept logits are copied, the others become -inf, so softmax of the  */
/*   output row is the truncated, renormalised distribution.                */
/* K <= 0 or K >= V turns top-k off, P >= 1 turns top-p off; P NaN or <= 0  */
/* is invalid (ORC_BAD_TRUNC, row copied unchanged).  Rows of greedy        */
/* requests (T = 0) and rows holding NaN are copied unchanged (the verify   */
/* itself reads them).  margin_out[row] (nullable) gets the relative        */
/* distance of the top-p decision from its threshold, min over the last     */
/* kept and the first dropped logit of |mass_gt - P| / P (+inf without      */
/* top-p): fp32 arithmetic may decide rows within 1e-5 differently.          */
/* ------------------------------------------------------------------------ */
#define ORC_BAD_TRUNC 1024u

static int cmp_desc(const void *a, const void *b)
{
    const double x = *(const double *)a, y = *(const double *)b;
    return x < y ? 1 : (x > y ? -1 : 0);
}

static uint32_t truncate_row(int dtype, int vocab, const void *in, size_t row, float t, int k,
                             float p, void *out, double *margin)
{
    const size_t esz = dtype == ORC_DTYPE_F32 ? 4 : 2;
    memcpy((char *)out + row * (size_t)vocab * esz, (const char *)in + row * (size_t)vocab * esz,
           (size_t)vocab * esz);
    *margin = INFINITY;
    const int top_k = k > 0 && k < vocab;
    const int top_p = p < 1.0f;
    if (p != p || p <= 0.0f)
        return ORC_BAD_TRUNC;
    if (!(t > 0.0f) || (!top_k && !top_p))
        return 0;
    double *x = malloc(sizeof(double) * (size_t)vocab);
    double *srt = malloc(sizeof(double) * (size_t)vocab);
    for (int v = 0; v < vocab; ++v) {
        x[v] = logit_at(in, dtype, row, vocab, v);
        if (isnan(x[v])) {
            free(x);
            free(srt);
            return 0;
        }
        srt[v] = x[v];
    }
    qsort(srt, (size_t)vocab, sizeof(double), cmp_desc);
    double tau = -INFINITY;   /* keep x >= tau */
    if (top_k)
        tau = srt[k - 1];
    if (top_p) {
        /* masses of the survivors, renormalised, from the largest logit down;  */
        /* every logit value of a run of equal values shares mass_gt            */
        const double m = srt[0];
        double total = 0.0;
        int n_kept = 0;
        while (n_kept < vocab && srt[n_kept] >= tau) {
            total += exp((srt[n_kept] - m) / (double)t);
            ++n_kept;
        }
        double gt = 0.0;      /* mass of strictly larger survivors */
        int i = 0;
        double tau_p = srt[0], last_kept_gt = 0.0, first_drop_gt = INFINITY;
        while (i < n_kept) {
            int j = i;
            double run = 0.0;
            while (j < n_kept && srt[j] == srt[i]) {
                run += exp((srt[j] - m) / (double)t);
                ++j;
            }
            if (gt / total < (double)p) {
                tau_p = srt[i];
                last_kept_gt = gt / total;
            } else {
                first_drop_gt = gt / total;
                break;
            }
            gt += run;
            i = j;
        }
        tau = tau_p > tau ? tau_p : tau;
        const double mk = ((double)p - last_kept_gt) / (double)p;
        const double md = (first_drop_gt - (double)p) / (double)p;
        *margin = mk < md ? mk : md;
    }
    for (int v = 0; v < vocab; ++v) {
        if (x[v] >= tau)
            continue;
        if (dtype == ORC_DTYPE_F32) {
            ((float *)out)[row * (size_t)vocab + (size_t)v] = -INFINITY;
        } else {
            ((uint16_t *)out)[row * (size_t)vocab + (size_t)v] = 0xff80u;  /* bf16 -inf */
        }
    }
    free(x);
    free(srt);
    return 0;
}

/* Truncates every target and draft row of a ragged batch (layout as        */
/* orc_verify) with its request's temperature, top_k and top_p.  draft_in   */
/* may be NULL.  Returns the status bits.                                   */
uint32_t orc_truncate(int dtype, int vocab, int batch, const int32_t *num_draft,
                      const float *temperature, const int32_t *top_k, const float *top_p,
                      const void *target_in, const void *draft_in, void *target_out,
                      void *draft_out, double *margin_t, double *margin_d)
{
    uint32_t status = 0;
    size_t t_row = 0, d_row = 0;
    double scratch;
    for (int r = 0; r < batch; ++r) {
        const int k = num_draft[r];
        for (int i = 0; i <= k; ++i, ++t_row)
            status |= truncate_row(dtype, vocab, target_in, t_row, temperature[r], top_k[r],
                                   top_p[r], target_out, margin_t ? &margin_t[t_row] : &scratch);
        if (draft_in)
            for (int i = 0; i < k; ++i, ++d_row)
                status |= truncate_row(dtype, vocab, draft_in, d_row, temperature[r], top_k[r],
                                       top_p[r], draft_out, margin_d ? &margin_d[d_row] : &scratch);
    }
    return status;
}
