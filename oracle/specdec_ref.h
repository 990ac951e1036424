/*
 * specdec_ref.h -- CPU oracle for batched speculative-decoding verification.
 *
 * TEST INFRASTRUCTURE ONLY. This header and specdec_ref.c are the plain, slow,
 * fp64 definition that the GPU library is checked against. Only the test suite,
 * the smoke check and the benchmark's CPU-baseline leg may load it; the product
 * path never does. It shares no source, header, table or helper with the GPU
 * library.
 *
 * The method (what one call computes), with the passage each step follows:
 *   - target logits for every draft position plus one bonus position, upcast to
 *     a wider float, temperature applied ("vLLM tour part 2", pyshine.com/vllm-2,
 *     section "Verification: rejection sampling on the GPU");
 *   - the grammar bitmask removes the tokens the grammar cannot accept (same page,
 *     section "Grammar gates: structured output");
 *   - accept draft x when a uniform draw is below min(1, p(x)/q(x)); greedy
 *     requests accept iff x is the argmax; stop at the first rejection and draw a
 *     recovered token from max(p - q, 0) renormalised; emit a bonus token when every
 *     draft is accepted (section "Verification: rejection sampling on the GPU"; the
 *     Rejection Sampler walk-through of "Speculative decoding -- code walkthrough",
 *     vllm-learning.pages.dev);
 *   - a draft with no probabilities (n-gram / suffix) is a one-hot q: accept with
 *     probability p(x); on rejection the residual is p with x removed, renormalised
 *     ("5.2 Draft models and model-free methods", infra-guide, section 4.3);
 *   - optional top-k / top-p on the target distribution before acceptance ("vLLM tour
 *     part 2", section "Verification: rejection sampling on the GPU");
 *   - counters R (raw drafts), I (grammar-invalidated), D = R - I (eligible),
 *     A (accepted) ("Structured output speculative decoding acceptance",
 *     fanout.sh, section "Name the three counters").
 *
 * Layout: B requests, cu[B+1] exclusive prefix of draft counts (cu[0] = 0),
 * k_b = cu[b+1] - cu[b]; draft d(b,j) = cu[b] + j; logit row t(b,j) = cu[b] + b + j
 * for j in [0, k_b], row j = k_b being the bonus row; T = cu[B] + B rows.
 * All pointers are host pointers.
 */
#ifndef SPECDEC_REF_H
#define SPECDEC_REF_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { REF_LOGITS_F32 = 0, REF_LOGITS_BF16 = 1 };

/* per-request status bits (status[b]) */
enum {
    REF_ST_BAD_DRAFT_ID = 1u,     /* a draft id outside [0, V) */
    REF_ST_EMPTY_MASK_ROW = 2u,   /* a row that was read allows no token (or only -inf logits) */
    REF_ST_BAD_TEMPERATURE = 4u,  /* temperature not 0 and not a positive normal finite float */
    REF_ST_K_TOO_LARGE = 8u,      /* k_b > max_k: request skipped */
    REF_ST_BAD_OFFSETS = 16u,     /* cu not non-decreasing within [0, cu[B]]: request skipped */
    REF_ST_BAD_TOP_P = 64u        /* top_p not a number in (0, 1]: no top-p filter */
};

/* Optional fp64 diagnostics (any pointer may be NULL). */
typedef struct {
    double* alpha;        /* [N]   acceptance probability of each draft that was tested, else NaN */
    double* row_m;        /* [T]   random rows read: max_i z_i/T; greedy rows read: max_i z_i; else NaN */
    double* row_S;        /* [T]   random rows read: sum_i exp(z_i/T - m); greedy rows: NaN; unread: NaN */
    double* emit_top1;    /* [B]   best score w_i/E_i of the emitting exponential race, else NaN */
    double* emit_top2;    /* [B]   runner-up score of that race (0 when it had one candidate), else NaN */
    double* emit_scores;  /* [V]   all race scores of request score_request (0 where w_i = 0), else NaN */
    int32_t score_request;/*       request whose race scores fill emit_scores (-1: none) */
    double* top_p_margin; /* [T] or NULL: for rows a top-p filter was applied to, the distance of
                           * the boundary tie groups' mass above from top_p; else +inf */
    uint64_t* telemetry;  /* [4][33] ADDED to, or NULL: per position j, row 0 counts drafts
                           * (j < k_b), row 1 grammar-eligible drafts (j < g_b), row 2 drafts
                           * accepted through position j (j < a_b); row 3 [a] counts requests
                           * that accepted exactly a drafts. Skipped requests are not counted.
                           * ("vLLM tour part 2", section "Telemetry and tuning": per-position
                           * draft / accepted counts and the acceptance histogram; "5.2 Draft
                           * models and model-free methods", section 7.2: the per-position count
                           * is of drafts accepted all the way through that position.) */
} specdec_ref_diag;

/* Returns 0 on success, 1 on invalid arguments (nothing written). counters[4] =
 * R, I, D, A are accumulated (added to), never cleared. */
int specdec_verify_ref(
    const void* target_logits, int32_t logits_dtype,   /* [T, V] */
    const int32_t* draft_ids,                          /* [N]; NULL allowed (then every draft is invalid) */
    const float* draft_probs,                          /* [N, V] or NULL */
    const uint8_t* has_q,                              /* [B] or NULL */
    const int32_t* cu_num_draft,                       /* [B+1] */
    int32_t B, int32_t V, int32_t max_k,
    const int32_t* bitmask,                            /* [T, ceil(V/32)] or NULL */
    const float* temperature,                          /* [B] */
    const float* uniforms,                             /* [T] */
    const float* exp_noise,                            /* [T, V] */
    const int32_t* top_k,                              /* [B] or NULL: top-k per request (<= 0: off) */
    const float* top_p,                                /* [B] or NULL: top-p per request (>= 1: off) */
    int32_t* out_tokens,                               /* [T] */
    int32_t* out_num_accepted,                         /* [B] */
    uint64_t* counters,                                /* [4] */
    uint32_t* status,                                  /* [B] or NULL */
    specdec_ref_diag* diag);                           /* or NULL */

/*
 * N-gram proposer ("5.2 Draft models and model-free methods", infra-guide, sections 4.1 and 6):
 * for request b with history h = tokens[cu_hist[b] .. cu_hist[b+1]) of length L, try window
 * lengths n from min(max_n, L - 1) down to min_n; for each n scan start positions 0, 1, ...,
 * L - n - 1 (the tail itself excluded) for h[start, start + n) == h[L - n, L); the first hit
 * proposes h[start + n, start + n + k) cut at L. out_drafts[b * k + j] holds the proposal
 * (-1 after it), out_num[b] its length, out_match[b] the window length n (0 on a miss).
 * Returns 0, or 1 on invalid arguments (min_n < 1, k < 0, B < 0, a NULL pointer, or
 * decreasing offsets); nothing is written then.
 */
int specdec_ngram_ref(const int32_t* tokens, const int64_t* cu_hist, int32_t B, int32_t min_n,
                      int32_t max_n, int32_t k, int32_t* out_drafts, int32_t* out_num,
                      int32_t* out_match);

#ifdef __cplusplus
}
#endif

#endif /* SPECDEC_REF_H */
