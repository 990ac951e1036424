/*
 * specdec_ref.c -- CPU oracle for batched speculative-decoding verification.
 *
 * TEST INFRASTRUCTURE ONLY: the plain, slow, fp64 statement of what one verify
 * call computes. Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg load it. It shares nothing with the GPU library.
 *
 * Every step is written the plainest way: one request at a time, one row at a
 * time, whole vocabulary arrays in fp64, library exp(). Where the pages are
 * silent the reading taken is stated beside the step.
 *
 * Parity status of each function: pinned by the CPU test suite (worked counter
 * example, p == q invariant, greedy brute force, grammar invariants, chi-square
 * losslessness, library softmax) -- except the token that one particular
 * exponential-race draw picks, which no page fixes: that choice follows the
 * sampling identity below and is checked only in distribution.
 */
#include "specdec_ref.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    const void* logits; int32_t dtype;
    const int32_t* draft_ids; const float* q; const uint8_t* has_q;
    const int32_t* cu; int32_t B, V, max_k;
    const int32_t* bitmask; int32_t W;
    const float* temperature; const float* uniforms; const float* noise;
    const int32_t* top_k; const float* top_p;
    int32_t* out_tokens; int32_t* out_num_accepted; uint64_t* counters; uint32_t* status;
    specdec_ref_diag* diag;
    double* z; double* p; double* w;   /* per-row scratch, V doubles each */
} ref_call;

/* Target logit of token i in row t, widened exactly (bf16 and fp32 both embed in fp64).
 * "Target logits are cast to float32": section "Verification: rejection sampling on
 * the GPU" of the vLLM tour (pyshine.com/vllm-2). */
static double target_logit(const ref_call* c, int64_t t, int32_t i)
{
    int64_t at = t * (int64_t)c->V + i;
    if (c->dtype == REF_LOGITS_BF16) {
        uint16_t h = ((const uint16_t*)c->logits)[at];
        uint32_t u = (uint32_t)h << 16;
        float f;
        memcpy(&f, &u, sizeof f);
        return (double)f;
    }
    return (double)((const float*)c->logits)[at];
}

/* Grammar bitmask lookup: bit (i & 31) of word i >> 5 of row t, 1 = the FSM accepts
 * token i (one mask row per speculative position plus the bonus: section "Grammar
 * gates: structured output" of the vLLM tour). No bitmask means unconstrained. */
static int grammar_allows(const ref_call* c, int64_t t, int32_t i)
{
    if (!c->bitmask) return 1;
    uint32_t word = (uint32_t)c->bitmask[t * (int64_t)c->W + (i >> 5)];
    return (int)((word >> (i & 31)) & 1u);
}

/* a3: apply the bitmask to the row. Reading: the page's "zeroes the logits of
 * tokens the FSM cannot accept" means those tokens get probability zero, i.e.
 * logit -inf (a logit of 0 would leave them sampleable). Returns the number of
 * tokens left with a finite logit. */
static int32_t masked_row(const ref_call* c, int64_t t)
{
    int32_t live = 0;
    for (int32_t i = 0; i < c->V; ++i) {
        double zi = grammar_allows(c, t, i) ? target_logit(c, t, i) : -INFINITY;
        c->z[i] = zi;
        if (zi > -INFINITY) ++live;
    }
    return live;
}

/* a6: the greedy target token, argmax of the masked logits, lowest index on ties
 * (reading: the pages give no tie rule). "a greedy variant that skips randomness
 * entirely for temperature-zero requests": section "Verification: rejection
 * sampling on the GPU". */
static int32_t greedy_token(const ref_call* c, double* zmax)
{
    int32_t best = -1;
    double bz = -INFINITY;
    for (int32_t i = 0; i < c->V; ++i)
        if (c->z[i] > bz) { bz = c->z[i]; best = i; }
    *zmax = bz;
    return best;
}

/* a5: temperature softmax p_i = exp(z_i/T - m) / S, m = max_i z_i/T ("apply_sampling_
 * constraints applies temperature ... to the flattened tensor": section "Verification:
 * rejection sampling on the GPU"). Masked tokens (-inf) get p_i = 0. */
static void temperature_softmax(const ref_call* c, double T, double* m_out, double* S_out)
{
    double m = -INFINITY;
    for (int32_t i = 0; i < c->V; ++i) {
        double s = c->z[i] / T;
        if (s > m) m = s;
    }
    double S = 0.0;
    for (int32_t i = 0; i < c->V; ++i) {
        double e = (c->z[i] > -INFINITY) ? exp(c->z[i] / T - m) : 0.0;
        c->p[i] = e;
        S += e;
    }
    for (int32_t i = 0; i < c->V; ++i) c->p[i] /= S;
    *m_out = m;
    *S_out = S;
}

/* Top-k / top-p on the masked, temperature-scaled target distribution p of a sampled row ("vLLM
 * tour part 2", section "Verification: rejection sampling on the GPU": apply_sampling_constraints
 * applies temperature and top-k/top-p to the flattened target tensor before acceptance).
 * Readings (the page gives no more): top-k keeps every allowed id whose logit is at least the k-th
 * largest allowed logit (ties at the boundary kept), k <= 0 keeps all; top-p then works on the
 * top-k distribution renormalised and keeps every id whose mass of strictly larger logits is below
 * top_p (the smallest top set reaching top_p, ties kept), top_p >= 1 keeps all. p is renormalised
 * over the kept ids. Returns the margin min |mass above - top_p| over the two tie groups at the
 * top-p boundary (+inf when top-p keeps all), for the parity exclusion band. */
typedef struct { double z, p; } zp_pair;

static int cmp_desc(const void* a, const void* b)
{
    const double x = ((const zp_pair*)a)->z, y = ((const zp_pair*)b)->z;
    return (x < y) - (x > y);
}

static double sampling_filter(const ref_call* c, int32_t k, double tp)
{
    /* the allowed ids' (logit, probability) pairs in decreasing logit order */
    int32_t m = 0;
    for (int32_t i = 0; i < c->V; ++i) if (c->z[i] > -INFINITY) ++m;
    zp_pair* a = (zp_pair*)malloc(sizeof(zp_pair) * (size_t)(m > 0 ? m : 1));
    m = 0;
    for (int32_t i = 0; i < c->V; ++i)
        if (c->z[i] > -INFINITY) { a[m].z = c->z[i]; a[m].p = c->p[i]; ++m; }
    qsort(a, (size_t)m, sizeof(zp_pair), cmp_desc);
    double zk = -INFINITY;                                   /* top-k: keep z >= zk */
    if (k > 0 && k < m) zk = a[k - 1].z;
    double Mk = 0.0;                                         /* mass of the top-k set */
    for (int32_t i = 0; i < m && a[i].z >= zk; ++i) Mk += a[i].p;
    double zp = zk, margin = INFINITY;                       /* top-p: keep z >= zp */
    if (tp < 1.0) {
        double above = 0.0;                                  /* renormalised mass of larger logits */
        int32_t g0 = 0;
        while (g0 < m && a[g0].z >= zk) {                    /* tie groups, decreasing logit */
            int32_t g1 = g0;
            double gm = 0.0;
            while (g1 < m && a[g1].z == a[g0].z) gm += a[g1++].p;
            const double dist = fabs(above - tp);
            if (dist < margin) margin = dist;
            if (!(above < tp)) break;                        /* this group and all below are dropped */
            zp = a[g0].z;
            above += gm / Mk;
            g0 = g1;
        }
    }
    double S = 0.0;
    for (int32_t i = 0; i < c->V; ++i) {
        if (!(c->z[i] >= zp) || c->z[i] == -INFINITY) c->p[i] = 0.0;
        S += c->p[i];
    }
    for (int32_t i = 0; i < c->V; ++i) c->p[i] /= S;
    free(a);
    return margin;
}

/* a7: probability of accepting draft x at draft slot d.
 * Draft model (q given): min(1, p(x)/q(x)) -- "accepts where the target's probability
 * of the draft token exceeds the random draw" (vLLM tour) with the ratio form of the
 * Rejection Sampler walk-through (vllm-learning, "Rejection Sampler": accept_probs =
 * minimum(1, target/draft)). p(x) = 0 gives 0; q(x) <= p(x) gives 1 (this covers
 * q(x) = 0 with p(x) > 0).
 * Model-free (no q): one-hot q, so the probability is p(x) ("5.2 Draft models and
 * model-free methods", section 4.3).
 * A grammar-invalid draft (j >= g) is never accepted: it fails before target
 * verification ("Structured output speculative decoding acceptance", section
 * "Name the three counters"). */
static double accept_probability(const ref_call* c, int qmode, int64_t d, int32_t x, int grammar_valid)
{
    if (!grammar_valid) return 0.0;
    double px = c->p[x];
    if (!qmode) return px;
    double qx = (double)c->q[d * (int64_t)c->V + x];
    if (px <= 0.0) return 0.0;
    if (qx <= px) return 1.0;
    return px / qx;
}

/* a9: residual weights for the recovered token. Draft model: w = max(p - q, 0)
 * ("the target probabilities minus the draft probabilities clamped at zero": vLLM
 * tour). Model-free: p with the draft token removed ("the residual is removed then
 * renormalized": infra-guide section 4.3). Returns the number of positive weights;
 * when none is positive (p == q on its support) the weights fall back to p (reading:
 * the pages do not treat the empty residual). */
static int32_t residual_weights(const ref_call* c, int qmode, int64_t d, int32_t x)
{
    int32_t pos = 0;
    for (int32_t i = 0; i < c->V; ++i) {
        double wi;
        if (qmode) {
            double r = c->p[i] - (double)c->q[d * (int64_t)c->V + i];
            wi = r > 0.0 ? r : 0.0;
        } else {
            wi = (i == x) ? 0.0 : c->p[i];
        }
        c->w[i] = wi;
        if (wi > 0.0) ++pos;
    }
    if (pos == 0) {
        for (int32_t i = 0; i < c->V; ++i) {
            c->w[i] = c->p[i];
            if (c->p[i] > 0.0) ++pos;
        }
    }
    return pos;
}

/* a9/a10: one draw from w / sum(w) by the exponential race: with E_i ~ Exp(1)
 * independent, argmax_i w_i / E_i lands on i with probability w_i / sum(w). The
 * pages only say a token is drawn ("draws a rescue token from the residual
 * distribution"); the race with caller-supplied noise is the sampling rule of this
 * library. Ties go to the lowest index. */
static int32_t exponential_race(const ref_call* c, int64_t t, int32_t b)
{
    const float* E = c->noise + t * (int64_t)c->V;
    int32_t best = -1;
    double top1 = -INFINITY, top2 = -INFINITY;
    int want_scores = c->diag && c->diag->emit_scores && c->diag->score_request == b;
    for (int32_t i = 0; i < c->V; ++i) {
        double s = 0.0;
        if (c->w[i] > 0.0) {
            s = c->w[i] / (double)E[i];
            if (s > top1) { top2 = top1; top1 = s; best = i; }
            else if (s > top2) { top2 = s; }
        }
        if (want_scores) c->diag->emit_scores[i] = s;
    }
    if (c->diag && c->diag->emit_top1) c->diag->emit_top1[b] = top1;
    if (c->diag && c->diag->emit_top2) c->diag->emit_top2[b] = top2 > -INFINITY ? top2 : 0.0;
    return best;
}

static int temperature_is_valid(float T)
{
    /* 0 (greedy) or a positive, normal, finite float */
    return T == 0.0f || (T >= 1.17549435e-38f && T <= 3.40282347e38f);
}

static void verify_request(ref_call* c, int32_t b)
{
    const int32_t lo = c->cu[b], hi = c->cu[b + 1], n_total = c->cu[c->B];
    uint32_t st = 0;

    /* a1: ragged decode. A request whose offsets are inconsistent is skipped. */
    if (c->cu[0] != 0 || lo < 0 || hi < lo || hi > n_total) {
        if (c->status) c->status[b] = REF_ST_BAD_OFFSETS;
        c->out_num_accepted[b] = 0;
        return;
    }
    const int32_t k = hi - lo;
    const int64_t row0 = (int64_t)lo + b;   /* t(b, 0) */
    if (k > c->max_k) {
        for (int32_t j = 0; j <= k; ++j) c->out_tokens[row0 + j] = -1;
        c->out_num_accepted[b] = 0;
        if (c->status) c->status[b] = REF_ST_K_TOO_LARGE;
        return;
    }

    /* a4: grammar-valid prefix g -- the first draft the grammar forbids ends the run of
     * eligible drafts: later positions have no valid grammar state to check against
     * (grammar state "advances only with verified constrained tokens"; section
     * "Reasoning boundaries complicate the window" of the acceptance post). An id
     * outside [0, V) is treated like a forbidden draft and flagged. */
    int32_t g = k;
    for (int32_t j = 0; j < k; ++j) {
        int32_t x = c->draft_ids ? c->draft_ids[lo + j] : -1;   /* no id array: every draft invalid */
        int ok = (x >= 0 && x < c->V);
        if (!ok) st |= REF_ST_BAD_DRAFT_ID;
        if (g == k && (!ok || !grammar_allows(c, row0 + j, x))) g = j;
    }

    /* mode flags: temperature 0 is greedy; draft probabilities make a draft-model
     * request unless has_q says otherwise */
    float Tf = c->temperature[b];
    if (!temperature_is_valid(Tf)) st |= REF_ST_BAD_TEMPERATURE;
    const int greedy = !(Tf > 0.0f) || !temperature_is_valid(Tf);
    const int qmode = (c->q != NULL) && (c->has_q == NULL || c->has_q[b] != 0);
    const double T = (double)Tf;
    /* top-k / top-p of this request: k <= 0 and top_p >= 1 keep all; a top_p that is not a
     * number in (0, 1] is flagged and keeps all */
    const int32_t filter_k = c->top_k ? c->top_k[b] : 0;
    double filter_p = 1.0;
    if (c->top_p) {
        const float tpf = c->top_p[b];
        if (tpf > 0.0f && tpf < 1.0f) filter_p = (double)tpf;
        else if (!(tpf >= 1.0f)) st |= REF_ST_BAD_TOP_P;
    }

    int32_t a = k;            /* accepted length */
    int32_t emitted = -1;     /* token at position a */
    for (int32_t j = 0; j <= k; ++j) {
        const int64_t t = row0 + j;
        const int64_t d = (int64_t)lo + j;
        const int is_bonus = (j == k);
        const int32_t x = (is_bonus || !c->draft_ids) ? -1 : c->draft_ids[d];
        const int x_ok = !is_bonus && x >= 0 && x < c->V;

        int32_t live = masked_row(c, t);
        if (live == 0) {                                   /* nothing the row allows */
            st |= REF_ST_EMPTY_MASK_ROW;
            if (c->diag && c->diag->row_m) c->diag->row_m[t] = -INFINITY;
            if (c->diag && c->diag->row_S) c->diag->row_S[t] = greedy ? NAN : 0.0;
            a = j;
            emitted = -1;
            break;
        }

        if (greedy) {
            double zmax;
            int32_t ystar = greedy_token(c, &zmax);
            if (c->diag && c->diag->row_m) c->diag->row_m[t] = zmax;
            if (c->diag && c->diag->row_S) c->diag->row_S[t] = NAN;
            if (is_bonus) { emitted = ystar; break; }
            int accept = (j < g) && x_ok && (x == ystar);
            if (c->diag && c->diag->alpha) c->diag->alpha[d] = accept ? 1.0 : 0.0;
            if (accept) { c->out_tokens[t] = x; continue; }
            a = j;
            emitted = ystar;   /* the greedy recovered token is the target argmax */
            break;
        }

        double m, S;
        temperature_softmax(c, T, &m, &S);
        if (c->diag && c->diag->row_m) c->diag->row_m[t] = m;
        if (c->diag && c->diag->row_S) c->diag->row_S[t] = S;
        if (filter_k > 0 || filter_p < 1.0) {
            const double margin = sampling_filter(c, filter_k, filter_p);
            if (c->diag && c->diag->top_p_margin) c->diag->top_p_margin[t] = margin;
        }
        if (is_bonus) {
            /* a10: the bonus token is an ordinary sample from p ("the bonus position is
             * sampled ... with the request's own sampler settings") */
            for (int32_t i = 0; i < c->V; ++i) c->w[i] = c->p[i];
            emitted = exponential_race(c, t, b);
            break;
        }
        double alpha = accept_probability(c, qmode, d, x, (j < g) && x_ok);
        if (c->diag && c->diag->alpha) c->diag->alpha[d] = alpha;
        /* a8: strict comparison of the draw against the acceptance probability */
        if ((double)c->uniforms[t] < alpha) { c->out_tokens[t] = x; continue; }
        residual_weights(c, qmode, d, x_ok ? x : -1);
        a = j;
        emitted = exponential_race(c, t, b);
        break;
    }

    /* a11: emit the accepted prefix (written above), the recovered/bonus token, and
     * -1 after it; accumulate the counters of the acceptance post's section "Name the
     * three counters". */
    c->out_tokens[row0 + a] = emitted;
    for (int32_t j = a + 1; j <= k; ++j) c->out_tokens[row0 + j] = -1;
    c->out_num_accepted[b] = a;
    c->counters[0] += (uint64_t)k;          /* R: raw drafts */
    c->counters[1] += (uint64_t)(k - g);    /* I: grammar-invalidated */
    c->counters[2] += (uint64_t)g;          /* D = R - I: eligible */
    c->counters[3] += (uint64_t)a;          /* A: accepted */
    /* per-position telemetry (row layout in specdec_ref.h) */
    if (c->diag && c->diag->telemetry) {
        uint64_t* tm = c->diag->telemetry;
        for (int32_t j = 0; j < k; ++j) tm[0 * 33 + j] += 1;
        for (int32_t j = 0; j < g; ++j) tm[1 * 33 + j] += 1;
        for (int32_t j = 0; j < a; ++j) tm[2 * 33 + j] += 1;
        tm[3 * 33 + a] += 1;
    }
    if (c->status) c->status[b] = st;
}

int specdec_verify_ref(
    const void* target_logits, int32_t logits_dtype,
    const int32_t* draft_ids, const float* draft_probs, const uint8_t* has_q,
    const int32_t* cu_num_draft, int32_t B, int32_t V, int32_t max_k,
    const int32_t* bitmask, const float* temperature, const float* uniforms,
    const float* exp_noise, const int32_t* top_k, const float* top_p, int32_t* out_tokens,
    int32_t* out_num_accepted, uint64_t* counters, uint32_t* status, specdec_ref_diag* diag)
{
    if (B < 0 || V <= 0 || max_k < 0 || max_k > 32) return 1;
    if (logits_dtype != REF_LOGITS_F32 && logits_dtype != REF_LOGITS_BF16) return 1;
    if (B == 0) return 0;
    if (!target_logits || !cu_num_draft || !temperature || !uniforms ||
        !exp_noise || !out_tokens || !out_num_accepted || !counters)
        return 1;

    ref_call c;
    memset(&c, 0, sizeof c);
    c.logits = target_logits; c.dtype = logits_dtype;
    c.draft_ids = draft_ids; c.q = draft_probs; c.has_q = has_q;
    c.cu = cu_num_draft; c.B = B; c.V = V; c.max_k = max_k;
    c.bitmask = bitmask; c.W = (V + 31) / 32;
    c.temperature = temperature; c.uniforms = uniforms; c.noise = exp_noise;
    c.top_k = top_k; c.top_p = top_p;
    c.out_tokens = out_tokens; c.out_num_accepted = out_num_accepted;
    c.counters = counters; c.status = status; c.diag = diag;
    c.z = (double*)malloc(sizeof(double) * (size_t)V);
    c.p = (double*)malloc(sizeof(double) * (size_t)V);
    c.w = (double*)malloc(sizeof(double) * (size_t)V);
    if (!c.z || !c.p || !c.w) { free(c.z); free(c.p); free(c.w); return 1; }

    if (diag) {
        /* untested / unread entries read NaN */
        int64_t N = cu_num_draft[B] > 0 ? cu_num_draft[B] : 0;
        int64_t T = N + B;
        if (diag->alpha) for (int64_t i = 0; i < N; ++i) diag->alpha[i] = NAN;
        if (diag->row_m) for (int64_t i = 0; i < T; ++i) diag->row_m[i] = NAN;
        if (diag->row_S) for (int64_t i = 0; i < T; ++i) diag->row_S[i] = NAN;
        if (diag->emit_top1) for (int32_t i = 0; i < B; ++i) diag->emit_top1[i] = NAN;
        if (diag->emit_top2) for (int32_t i = 0; i < B; ++i) diag->emit_top2[i] = NAN;
        if (diag->emit_scores) for (int32_t i = 0; i < V; ++i) diag->emit_scores[i] = NAN;
        if (diag->top_p_margin) for (int64_t i = 0; i < T; ++i) diag->top_p_margin[i] = INFINITY;
    }

    for (int32_t b = 0; b < B; ++b) verify_request(&c, b);

    free(c.z); free(c.p); free(c.w);
    return 0;
}


/* ---------------------------------------------------------------------------------------------
 * N-gram proposer (see specdec_ref.h): the rule of the infra-guide's section 6 hands-on, window
 * lengths from long to short, start positions from front to back, first hit wins.
 * ------------------------------------------------------------------------------------------- */
int specdec_ngram_ref(const int32_t* tokens, const int64_t* cu_hist, int32_t B, int32_t min_n,
                      int32_t max_n, int32_t k, int32_t* out_drafts, int32_t* out_num,
                      int32_t* out_match)
{
    if (B < 0 || min_n < 1 || k < 0 || !cu_hist || !out_num || !out_match) return 1;
    if (B > 0 && (!tokens || (k > 0 && !out_drafts))) return 1;
    for (int32_t b = 0; b < B; ++b)
        if (cu_hist[b + 1] < cu_hist[b] || cu_hist[b] < 0) return 1;
    for (int32_t b = 0; b < B; ++b) {
        const int32_t* h = tokens + cu_hist[b];
        const int64_t L = cu_hist[b + 1] - cu_hist[b];
        int32_t hit_n = 0;
        int64_t hit_start = -1;
        const int64_t n_hi = (int64_t)max_n < L - 1 ? (int64_t)max_n : L - 1;
        for (int64_t n = n_hi; n >= min_n && hit_n == 0; --n) {
            const int32_t* tail = h + (L - n);
            for (int64_t start = 0; start < L - n; ++start) {
                int64_t i = 0;
                while (i < n && h[start + i] == tail[i]) ++i;
                if (i == n) { hit_n = (int32_t)n; hit_start = start; break; }
            }
        }
        int32_t num = 0;
        if (hit_n > 0) {
            const int64_t from = hit_start + hit_n;
            for (int64_t j = 0; j < k && from + j < L; ++j) out_drafts[(int64_t)b * k + j] = h[from + j];
            num = (int32_t)((L - from) < k ? (L - from) : k);
        }
        for (int64_t j = num; j < k; ++j) out_drafts[(int64_t)b * k + j] = -1;
        out_num[b] = num;
        out_match[b] = hit_n;
    }
    return 0;
}
