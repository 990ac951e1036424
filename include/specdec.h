/*
 * specdec.h -- C ABI of libspecdec.so: batched speculative-decoding verification on
 * one GB300 (sm_103a).
 *
 * One call verifies a ragged batch of draft tokens against the target model's logits:
 * it applies each position's packed grammar bitmask, takes the temperature softmax,
 * accepts each draft with probability min(1, p/q) (or by argmax equality for greedy
 * requests), stops at the first rejection, draws the recovered token there from the
 * residual distribution, emits a bonus token when every draft is accepted, and
 * accumulates the raw / grammar-invalidated / eligible / accepted counters.
 *
 * Sources for the operation:
 *   - "vLLM tour part 2" (pyshine.com/vllm-2), section "Verification: rejection sampling
 *     on the GPU": target logits for every draft position plus one bonus position, cast
 *     to float32, temperature applied; acceptance where the target probability of the
 *     draft token beats a uniform draw; recovered token from the target probabilities
 *     minus the draft probabilities clamped at zero; greedy variant for temperature 0.
 *   - same page, section "Grammar gates: structured output": one bitmask row per request
 *     and per speculative position; masked tokens cannot be produced.
 *   - "5.2 Draft models and model-free methods" (infra-guide), section 4.3: a draft with
 *     no probabilities is a one-hot q -- accept with probability p(x), residual = p with x
 *     removed, renormalised.
 *   - "Structured output speculative decoding acceptance" (fanout.sh), section "Name the
 *     three counters": R raw drafts, I grammar-invalidated, D = R - I eligible, A accepted.
 *
 * Layout conventions (all calls):
 *   B requests; cu_num_draft[B+1] is an exclusive prefix sum, cu[0] = 0, non-decreasing;
 *   request b has k_b = cu[b+1] - cu[b] drafts; N = cu[B].
 *   Draft slot d(b,j) = cu[b] + j, j in [0, k_b).
 *   Logit row t(b,j) = cu[b] + b + j, j in [0, k_b]; row j = k_b is the bonus row;
 *   T = N + B rows.  W = ceil(V / 32) mask words per row.
 *   A request is greedy iff temperature[b] == 0. It is a draft-model request iff
 *   draft_probs != NULL and (has_q == NULL or has_q[b] != 0); otherwise model-free.
 */
#ifndef SPECDEC_H
#define SPECDEC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SPECDEC_KMAX 32           /* largest supported max_k (drafts per request) */
#define SPECDEC_TELEMETRY_ROW (SPECDEC_KMAX + 1)   /* entries per telemetry row */

typedef enum {
    SPECDEC_OK = 0,
    SPECDEC_ERR_INVALID_ARG = 1,   /* a NULL required pointer, a bad size or a misaligned pointer */
    SPECDEC_ERR_UNSUPPORTED = 2,   /* dtype unknown, or a row too wide for on-chip staging */
    SPECDEC_ERR_CUDA = 3,          /* a CUDA runtime error at launch (or from specdec_wait) */
    SPECDEC_ERR_TIMEOUT = 4        /* specdec_wait gave up */
} specdec_status_t;

typedef enum { SPECDEC_F32 = 0, SPECDEC_BF16 = 1 } specdec_dtype_t;

/* Per-request status bits written to status[b] (0 = clean). The kernel never traps. */
#define SPECDEC_ST_BAD_DRAFT_ID    1u   /* a draft id outside [0, V): counted invalid, never accepted */
#define SPECDEC_ST_EMPTY_MASK_ROW  2u   /* a row read allows no finite logit: -1 emitted there, request stops */
#define SPECDEC_ST_BAD_TEMPERATURE 4u   /* not 0 and not a positive normal finite float: verified greedily */
#define SPECDEC_ST_K_TOO_LARGE     8u   /* k_b > max_k: skipped, -1 in its rows, no counters */
#define SPECDEC_ST_BAD_OFFSETS    16u   /* cu[0] != 0 or cu[b] > cu[b+1] or cu[b+1] > cu[B]: skipped */
#define SPECDEC_ST_DEVICE_TIMEOUT 32u   /* an on-chip copy did not land within its time limit */
#define SPECDEC_ST_BAD_TOP_P      64u   /* top_p not a number in (0, 1]: no top-p filter */

/*
 * specdec_verify -- verify one batch (stream-ordered, asynchronous).
 *
 * Pointers are device pointers to caller-owned memory on the current device; the
 * library allocates nothing and keeps no state between calls.
 *
 *   target_logits  [T, V] row-major, fp32 or bf16 (logits_dtype); 4- resp. 2-byte aligned.
 *   draft_ids      [N] int32; may be NULL when N = 0 (a request that does have drafts then
 *                  gets SPECDEC_ST_BAD_DRAFT_ID and all its drafts count as invalid).
 *   draft_probs    [N, V] fp32 draft distributions q, or NULL (every request model-free).
 *                  Only q(x) of each tested draft and the q row of a rejected position are read.
 *   has_q          [B] uint8 or NULL (NULL: every request is a draft-model request iff
 *                  draft_probs != NULL).
 *   cu_num_draft   [B+1] int32 exclusive prefix of draft counts.
 *   B, V, max_k    B >= 0, V >= 1, 0 <= max_k <= SPECDEC_KMAX (every k_b must be <= max_k).
 *   bitmask        [T, W] int32 or NULL (unconstrained). Bit (i & 31) of word i >> 5 is 1
 *                  when token i is allowed; bits at or above V are ignored.
 *   temperature    [B] fp32; 0 means greedy.
 *   top_k          [B] int32 or NULL: top-k per request (<= 0: off). The target distribution of a
 *                  sampled request keeps every allowed id whose logit is at least the k-th largest
 *                  allowed logit (ties at the boundary kept) before acceptance, residual and bonus
 *                  ("vLLM tour part 2", section "Verification: rejection sampling on the GPU":
 *                  temperature and top-k/top-p are applied to the target tensor). Greedy requests
 *                  ignore it (the argmax is always kept).
 *   top_p          [B] fp32 or NULL: top-p per request (>= 1: off), applied after top-k: the kept
 *                  ids are those whose (top-k renormalised) mass of strictly larger logits is
 *                  below top_p (ties kept); p is renormalised over the kept ids. A value that is
 *                  not a number in (0, 1] sets SPECDEC_ST_BAD_TOP_P and is ignored. With top_k or
 *                  top_p given, the streaming kernel runs one CTA per request. A draft that is
 *                  surely kept and whose uniform lies below e_x / (S q(x)) (S the row's whole
 *                  softmax sum, a lower bound of the filtered ratio) is accepted without a
 *                  threshold search, unless diag_accept_prob is given (every filtered row then
 *                  searches, so that the exact filtered alpha can be reported). A top-k search
 *                  (k <= 1927) first streams a filtered row once more to take its top slice of
 *                  logits (the elements carrying at least 1.0625 S / 2048 of the mass, or 16x less
 *                  on a retry); when that holds k elements the top-k search, and a top-p search
 *                  after it, run on chip. Otherwise a search streams the row to bin its logits by
 *                  mass (an accepted top-p row may be settled there) and once more to collect the
 *                  chosen bin (on chip when it holds at most 2048 elements, else one more pass per
 *                  8-bit digit of its keys: at most 2 for bf16 logits, 4 for fp32). A stop row
 *                  with few kept ids draws from those ids only. The outputs do not depend on the
 *                  route. V > 2^20, or the slice-resident cluster kernel
 *                  (specdec_set_launch_options), with either of them: SPECDEC_ERR_UNSUPPORTED.
 *   uniforms       [T] fp32 in [0, 1); draft j of request b is accepted iff
 *                  uniforms[t(b,j)] < alpha (strict). Entries at bonus rows are unused.
 *   exp_noise      [T, V] fp32 Exp(1) samples > 0; the token drawn from weights w at row t
 *                  is argmax_i w_i / exp_noise[t, i] (lowest index on ties). Read only at
 *                  the one row per random request that draws a token.
 *   out_tokens     [T] int32: the accepted drafts, then the recovered or bonus token,
 *                  then -1 for every later position of the request.
 *   out_num_accepted [B] int32: accepted drafts a_b per request.
 *   counters       [4] uint64 (R, I, D, A), ADDED to (never cleared by the library).
 *   status         [B] uint32 per-request status bits (written, not accumulated), or NULL.
 *   diag_accept_prob [N] fp32 or NULL: alpha of every draft that was tested, NaN otherwise.
 *   diag_row_stats [T, 2] fp32 or NULL: for every row read, (m, S) with m = max_i z_i / T
 *                  and S = sum_i exp(z_i / T - m) on random requests, (max_i z_i, NaN) on
 *                  greedy ones; (NaN, NaN) for rows not read. Entries of a request skipped
 *                  for SPECDEC_ST_BAD_OFFSETS are left untouched (its rows are unknown).
 *   telemetry      [4 * SPECDEC_TELEMETRY_ROW] uint64 or NULL, ADDED to (never cleared), 8-byte
 *                  aligned: per position j, row 0 counts drafts (k_b > j), row 1 grammar-eligible
 *                  drafts (g_b > j, g_b the grammar-valid prefix behind I and D), row 2 drafts
 *                  accepted all the way through position j (a_b > j); row 3 [a] counts requests
 *                  that accepted exactly a drafts. Requests skipped for K_TOO_LARGE or BAD_OFFSETS
 *                  are not counted. Rows 0..2 sum to R, D and A. ("vLLM tour part 2", section
 *                  "Telemetry and tuning": per-position draft / accepted counts and the histogram
 *                  of accepted lengths; "5.2 Draft models and model-free methods", section 7.2:
 *                  a position counts drafts accepted through it.)
 *   workspace      device scratch of at least specdec_workspace_size(B, V) bytes, 16-byte
 *                  aligned, caller-owned, or NULL. With a workspace a one-CTA kernel first orders
 *                  the requests by an estimate of their work, heaviest first, and the verify
 *                  kernel takes them in that order (list scheduling by the longest-processing-
 *                  time rule: a long request that sits late in the batch no longer runs on alone
 *                  after the rest have finished). The schedule runs only when the batch needs more
 *                  than one wave of resident CTAs (two per SM); the verify kernel then starts as a
 *                  programmatic dependent of it. A batch that exceeds that wave additionally splits
 *                  its heaviest requests (a sixth of a wave) over clusters of 2 CTAs (their chains
 *                  of row passes are what set the launch's length) and runs the others two per
 *                  cluster, one per CTA. Without a workspace, requests start in index order, one
 *                  CTA each.
 *                  Results are identical either way; only the timing differs. The workspace
 *                  needs no initialisation and holds nothing between calls; calls that share one
 *                  workspace must not overlap in time (use one per stream).
 *   workspace_bytes its size in bytes.
 *   stream         a cudaStream_t (NULL = legacy default stream).
 *
 * Rows after a request's stop row a_b (its first rejection, or the bonus row) are never used: no
 * output depends on them. At the byte level, a request whose bitmask is absent or dense may read
 * the first two ring chunks (at most 2 x 32 KB) of row a_b + 1, queued before the decision on
 * row a_b and discarded unused; a request with a sparse bitmask prefetches the mask words of all
 * its rows into L2 when it starts. Nothing else of a later row is read.
 * Returns SPECDEC_OK once the kernel is queued; data errors land in status[].
 * Errors: SPECDEC_ERR_INVALID_ARG (nothing launched, nothing written) for a NULL required
 * pointer (draft_ids may be NULL), B < 0, V < 1, max_k outside [0, SPECDEC_KMAX], or a pointer not aligned to its
 * element (telemetry: 8 bytes); SPECDEC_ERR_UNSUPPORTED for an unknown dtype, for top_k or top_p with V > 2^20
 * (or with the cluster kernel), or, with the cluster kernel that keeps each row slice on chip, a row wider than
 * 3 MiB; SPECDEC_ERR_CUDA if the launch fails.
 *
 * Kernels: by default each request is verified by a cluster of G CTAs (G = 1 for large
 * batches, up to 4 for small ones), each streaming its slice of every row through a ring of
 * 32 KB shared-memory stages filled by bulk async copies; requests whose bitmask allows few ids
 * gather only the allowed 16-byte groups instead. specdec_set_launch_options (below) selects the
 * alternative kernel that keeps a slice of every row resident in shared memory, forces G, or
 * forces the request schedule on or off. All shapes compute identical results.
 */
specdec_status_t specdec_verify(
    const void* target_logits, specdec_dtype_t logits_dtype,
    const int32_t* draft_ids,
    const float* draft_probs,
    const uint8_t* has_q,
    const int32_t* cu_num_draft,
    int32_t B, int32_t V, int32_t max_k,
    const int32_t* bitmask,
    const float* temperature,
    const int32_t* top_k,
    const float* top_p,
    const float* uniforms,
    const float* exp_noise,
    int32_t* out_tokens,
    int32_t* out_num_accepted,
    unsigned long long* counters,
    uint32_t* status,
    float* diag_accept_prob,
    float* diag_row_stats,
    unsigned long long* telemetry,
    void* workspace,
    size_t workspace_bytes,
    void* stream);

/*
 * specdec_verify_noalloc -- specdec_verify for callers that cannot hand the library scratch
 * memory. The pages have no counterpart to this: it is a calling convention of this library,
 * not a step of the method.
 *
 * Same arguments, semantics and results as specdec_verify, without workspace / workspace_bytes:
 * the request schedule's scratch (an int32 order and a cost byte per request) is a fixed array
 * inside the library, file-scope device memory of 80 KiB per device holding up to
 * SPECDEC_NOALLOC_MAX_REQUESTS requests. The call allocates nothing (no cudaMalloc, no
 * allocating library routine) and needs no memory from the caller beyond the batch itself.
 * It serves callers that have no device allocator of their own (a plain C or C++ host program
 * that links this library directly) and serving loops that must not allocate inside a decode
 * step (cudaMalloc synchronises the device; a caching allocator may have to grow its pool).
 *
 *   B > SPECDEC_NOALLOC_MAX_REQUESTS: SPECDEC_ERR_UNSUPPORTED, checked before any CUDA call;
 *   nothing is launched or written. Every other error is specdec_verify's.
 *   Zeroing: nothing in the scratch has to start at zero; each call writes every entry it reads.
 *   Set-up: the first call with B > 0 on a device looks the array's address up with
 *   cudaGetSymbolAddress (once per device, then cached; SPECDEC_ERR_CUDA if that fails). Make
 *   that first call on each device before any stream capture begins on it. The cache is keyed
 *   on the current context's unique id as well: after cudaDeviceReset, or in a context the
 *   caller created with the driver API, the next call looks the address up again (so make that
 *   call outside stream capture too).
 *   Concurrency: all calls on a device share the one array. Two calls that overlap in time (on
 *   different streams, or from host threads whose calls are not stream-ordered) race on it, and
 *   the outputs and counters of both are then undefined. Queue such calls on one stream, or use
 *   specdec_verify with one workspace per stream.
 */
#define SPECDEC_NOALLOC_MAX_REQUESTS 16384
specdec_status_t specdec_verify_noalloc(
    const void* target_logits, specdec_dtype_t logits_dtype,
    const int32_t* draft_ids,
    const float* draft_probs,
    const uint8_t* has_q,
    const int32_t* cu_num_draft,
    int32_t B, int32_t V, int32_t max_k,
    const int32_t* bitmask,
    const float* temperature,
    const int32_t* top_k,
    const float* top_p,
    const float* uniforms,
    const float* exp_noise,
    int32_t* out_tokens,
    int32_t* out_num_accepted,
    unsigned long long* counters,
    uint32_t* status,
    float* diag_accept_prob,
    float* diag_row_stats,
    unsigned long long* telemetry,
    void* stream);

/*
 * specdec_ngram_propose -- model-free drafts for a batch: the n-gram proposer of "5.2 Draft
 * models and model-free methods" (infra-guide), sections 4.1 and 6 (stream-ordered,
 * asynchronous). For request b with history h = tokens[cu_hist[b] .. cu_hist[b+1]) of length L,
 * the window length is the longest n in [min_n, min(max_n, L - 1)] such that the last n tokens of
 * h also occur earlier in h (the tail itself excluded), taking the earliest such occurrence; the
 * proposal is the (up to) k tokens that follow it, cut at the end of h. The drafts go to the
 * verify as model-free drafts (no q): accepted with probability p(x).
 *
 *   tokens         [cu_hist[B]] int32 token ids, the histories back to back (device).
 *   cu_hist        [B+1] int64 offsets; a request with cu_hist[b+1] < cu_hist[b] or a negative
 *                  offset counts as an empty history (a miss).
 *   B              requests (>= 0).
 *   min_n, max_n   window lengths tried, 1 <= min_n; max_n <= SPECDEC_NGRAM_MAX_N (64);
 *                  max_n < min_n means no window is tried.
 *   k              proposal length, 0 <= k <= SPECDEC_KMAX.
 *   out_drafts     [B, k] int32: the proposal, then -1.
 *   out_num        [B] int32 proposal lengths (0 on a miss).
 *   out_match      [B] int32 window length of the match (0 on a miss).
 * Returns SPECDEC_OK once queued; SPECDEC_ERR_INVALID_ARG for a bad size, a NULL required pointer
 * or a misaligned one (nothing launched); SPECDEC_ERR_UNSUPPORTED for max_n > 64;
 * SPECDEC_ERR_CUDA if the launch fails.
 */
#define SPECDEC_NGRAM_MAX_N 64
specdec_status_t specdec_ngram_propose(const int32_t* tokens, const int64_t* cu_hist, int32_t B,
                                       int32_t min_n, int32_t max_n, int32_t k, int32_t* out_drafts,
                                       int32_t* out_num, int32_t* out_match, void* stream);

/*
 * specdec_bitmask_scatter -- the grammar bitmask of one verify step in batch order, from the
 * compacted masks in scheduler order ("vLLM tour part 2", section "Grammar gates: structured
 * output": masks arrive compacted to the constrained requests in scheduler order, while the batch
 * has its own order and per-request speculative offsets). Stream-ordered, asynchronous.
 *
 *   compact        [compact_rows, W] int32, W = ceil(V / 32): for each constrained request in
 *                  scheduler order, its k_b + 1 rows (draft positions, then the bonus position).
 *   constrained    [n] int32: the batch index b of each constrained request, scheduler order.
 *   cu_num_draft   [B+1] int32 batch-order draft offsets (the verify's layout: row t(b, j) =
 *                  cu[b] + b + j, j in [0, k_b]).
 *   bitmask        [T, W] int32 output, T = cu[B] + B: the rows of each constrained request take
 *                  its compact rows; rows of every other request are all ones (-1: all allowed).
 * Readings for malformed input: an id outside [0, B) owns no compact rows; a request listed twice
 * takes the rows of its first listing (the second listing's rows are skipped over); a row past the
 * end of `compact` gets zeros (nothing allowed; the verify then reports an empty mask row); a
 * request with malformed offsets (as SPECDEC_ST_BAD_OFFSETS) owns no rows and its rows are not
 * written. Returns SPECDEC_OK once queued; SPECDEC_ERR_INVALID_ARG for a bad size, a NULL
 * required pointer or a misaligned one; SPECDEC_ERR_UNSUPPORTED for V > 2^26; SPECDEC_ERR_CUDA if
 * the launch fails.
 */
specdec_status_t specdec_bitmask_scatter(const int32_t* compact, int64_t compact_rows,
                                         const int32_t* constrained, int32_t n,
                                         const int32_t* cu_num_draft, int32_t B, int32_t V,
                                         int32_t* bitmask, void* stream);

/*
 * specdec_wait -- block the calling host thread until all work queued on `stream` has
 * finished, or until timeout_ms milliseconds have passed (polling; timeout_ms < 0 waits
 * without limit). Returns SPECDEC_OK, SPECDEC_ERR_TIMEOUT, or SPECDEC_ERR_CUDA when the
 * stream reports an error.
 */
specdec_status_t specdec_wait(void* stream, int32_t timeout_ms);

/*
 * specdec_set_launch_options -- for comparison and test runs: override the launch choices the
 * library otherwise makes by itself. No step of the method depends on them; every choice
 * computes identical results. Process-wide; set it between calls (a call in flight on another
 * host thread may see either setting). The initial values come once per process from the
 * environment (SPECDEC_KERNEL=cluster|stream, SPECDEC_CTAS_PER_REQUEST=G,
 * SPECDEC_SCHEDULE=1|0); no call reads the environment after that.
 *   kernel            -1: automatic (the streaming kernel); 0: streaming kernel; 1: the
 *                     slice-resident cluster kernel (a slice of every row kept in shared memory
 *                     by a cluster of CTAs per request; slower, kept as an independent
 *                     decomposition of the same computation for cross-checks).
 *   ctas_per_request  -1: automatic; 1..16: CTAs per request (the cluster size).
 *   schedule          -1: automatic (when the batch exceeds one wave of resident CTAs);
 *                     0: never; 1: always, whenever a workspace is given.
 *   wait_limit_us     -1: 2 s; 0..2000000: the limit, in microseconds, of every wait of the
 *                     streaming kernel on one of its barriers (a test sets 0 to make the waits
 *                     expire). When a wait expires the CTA issues no more copies, its other waits
 *                     give up at once, it waits (at most 1 s more) for the copies already in
 *                     flight, and the request gets SPECDEC_ST_DEVICE_TIMEOUT; its other outputs
 *                     are then undefined. Nothing traps or hangs, and later calls are unaffected.
 *   split_requests    -1: automatic; 0: none; n > 0: n. How many of the heaviest requests a
 *                     scheduled launch of one CTA per request (a workspace, no top-k / top-p)
 *                     splits over a cluster of 2 CTAs, the other requests then running two per
 *                     cluster, one per CTA. Automatic: when the batch has more requests than one
 *                     wave of resident CTAs (two per SM), the heaviest sixth of a wave of them.
 * Returns SPECDEC_ERR_INVALID_ARG (nothing changed) for a value outside those ranges.
 */
specdec_status_t specdec_set_launch_options(int32_t kernel, int32_t ctas_per_request, int32_t schedule,
                                            int32_t wait_limit_us, int32_t split_requests);

/* Bytes of workspace specdec_verify uses for B requests of vocabulary size V (0 if B or V <= 0):
 * the request order (int32 per request) and one cost byte per request. */
size_t specdec_workspace_size(int32_t B, int32_t V);

/* Human-readable name of a status code (static storage). */
const char* specdec_status_string(specdec_status_t status);

/*
 * specdec_launch_config -- the launch shape specdec_verify uses for a batch of B requests of
 * vocabulary size V (host arithmetic; the SM count comes from the current device, 152 when none
 * is visible): CTAs per request (a thread-block cluster that splits every vocabulary row into
 * contiguous slices), threads per CTA, dynamic shared memory per CTA in bytes, vocabulary ids
 * per slice, the number of kernels one call launches when given a workspace (2 when the
 * request schedule runs, else 1; without a workspace it is always 1), and how many requests a
 * call with a workspace and without top-k / top-p splits over clusters of 2 CTAs (0: none; the
 * others then run two per cluster, one per CTA, and the grid has 2 * (n + ceil((B - n) / 2))
 * CTAs). Any output pointer may be NULL. Returns SPECDEC_ERR_INVALID_ARG /
 * SPECDEC_ERR_UNSUPPORTED like specdec_verify.
 */
specdec_status_t specdec_launch_config(int32_t B, int32_t V, specdec_dtype_t logits_dtype,
                                       int32_t* ctas_per_request, int32_t* threads_per_cta,
                                       int32_t* smem_bytes, int32_t* slice_ids,
                                       int32_t* kernels_with_workspace, int32_t* split_requests);

#ifdef __cplusplus
}
#endif

#endif /* SPECDEC_H */
