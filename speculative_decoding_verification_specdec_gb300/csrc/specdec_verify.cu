/*
 * specdec_verify.cu -- fused speculative-decoding verify kernel for GB300 (sm_103a) and
 * the C-ABI launcher declared in include/specdec.h.
 *
 * What it computes (see include/specdec.h for the passages): per request, rows
 * j = 0, 1, ... of the target logits in order -- grammar bitmask, temperature softmax
 * statistics, acceptance of draft j (uniform draw below min(1, p/q), p(x) for a one-hot
 * model-free draft, argmax equality when greedy) -- until the first rejection or the
 * bonus row; there the recovered / bonus token is drawn as argmax_i w_i / E_i (exponential
 * race) with w = max(p - q, 0), p without the draft token, or p. Only w = max(p - q, 0) needs the
 * row's normaliser first and takes a second pass over the stop row; the other two fold into the
 * row's own pass. No output depends on a row after the stop row (the streaming kernel may have
 * fetched up to two chunks of the next one before the decision; they are discarded).
 *
 * GB300 mapping (the streaming kernel, used by default):
 *   - one CTA per request (a thread-block cluster of up to 4 CTAs on small batches, each owning a
 *     contiguous slice of every row); warp 0 is a producer whose lane 0 streams 32 KB chunks of
 *     the rows (logits and mask words; logits, noise, q and mask words for a draw) with bulk async
 *     copies (cp.async.bulk, the TMA engine) into a 3-stage shared-memory ring, each stage with
 *     "full" and "empty" mbarriers; 8 consumer warps fold each chunk with 128-bit shared-memory
 *     reads (online max / sum with ex2.approx, lazy argmax ids, the race score w / E);
 *   - at the end of a row the consumers reduce (redux.sync and shuffles in each warp, then the
 *     warps' partials in order; DSMEM partials across a cluster), every thread takes the same
 *     decision, and posts it to the producer, which has already queued the next row's first
 *     chunks so HBM keeps streaming across the decision;
 *   - a request whose bitmask allows few ids gathers only the allowed 16-byte groups (cp.async)
 *     after listing them from the mask words;
 *   - with a workspace, a one-CTA kernel first orders the requests heaviest first.
 * The first design, kept as an independent cross-check of the same computation
 * (specdec_verify_kernel, selected with specdec_set_launch_options): a cluster of CTAs per
 * request keeps its slices of the current row in shared memory, so the draw pass re-reads only
 * noise and q; it is about 2x slower and has no top-k / top-p.
 * No tensor cores: nothing here is a contraction. Everything is fp32 (bf16 logits are
 * widened exactly); exp uses the ex2.approx hardware instruction on pre-scaled inputs.
 *
 * Every wait on an mbarrier is bounded in time; on expiry the request gets
 * SPECDEC_ST_DEVICE_TIMEOUT and the kernel runs to completion without hanging.
 */
#include <cuda_runtime.h>
#include <stdint.h>

#include <cfloat>
#include <climits>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <ctime>
#include <atomic>
#include <mutex>
#include <type_traits>

#include "specdec.h"

// Phase tracing (diagnostic builds only: compile with -DSPECDEC_TRACE). The first consumer
// thread of each request writes (%globaltimer << 4 | tag) into trace[request * 64 + i] and the
// number of stamps into slot 63. The default build compiles every stamp away.
#ifdef SPECDEC_TRACE
__device__ unsigned long long* g_specdec_trace = nullptr;
extern "C" int specdec_trace_set(void* buffer)
{
    return (int)cudaMemcpyToSymbol(g_specdec_trace, &buffer, sizeof(buffer));
}
#define SPECDEC_TRACE_BEGIN(req, on)                                                               \
    int trace_n_ = 0;                                                                              \
    const bool trace_on_ = (on);                                                                   \
    unsigned long long* trace_ = g_specdec_trace ? g_specdec_trace + (size_t)(req) * 64 : nullptr;
// -DSPECDEC_TRACE_LIGHT keeps only the first and last stamp of each request (tags 0 and 7), so
// the timing of the phases in between is not disturbed; -DSPECDEC_TRACE_TAGS=mask keeps the tags
// whose bits are set.
#if defined(SPECDEC_TRACE_TAGS)
#define SPECDEC_TRACE_KEEP(tag) (((SPECDEC_TRACE_TAGS) >> (tag)) & 1)
#elif defined(SPECDEC_TRACE_LIGHT)
#define SPECDEC_TRACE_KEEP(tag) ((tag) == 0 || (tag) == 7)
#else
#define SPECDEC_TRACE_KEEP(tag) true
#endif
#define SPECDEC_STAMP(tag)                                                                         \
    do {                                                                                           \
        if (SPECDEC_TRACE_KEEP(tag) && trace_on_ && trace_ && trace_n_ < 62) {                    \
            unsigned long long t_;                                                                 \
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t_));                                 \
            trace_[trace_n_++] = (t_ << 4) | (unsigned long long)(tag);                            \
        }                                                                                          \
    } while (0)
#define SPECDEC_TRACE_END()                                                                        \
    do { if (trace_on_ && trace_) trace_[63] = (unsigned long long)trace_n_; } while (0)
#else
#define SPECDEC_TRACE_BEGIN(req, on)
#define SPECDEC_STAMP(tag) do { } while (0)
#define SPECDEC_TRACE_END() do { } while (0)
#endif

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kUnit = 128;                    // slice granularity in ids (4 mask words)
constexpr int kChunks = 4;                    // bulk copies / mbarriers per row slice
constexpr int kMaxCluster = 16;
constexpr int kTargetSliceBytes = 32 * 1024;
constexpr int kMaxSliceBytes = 192 * 1024;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;   // 2 s per wait
constexpr unsigned long long kDrainLimitNs = 1000000000ull;  // copies in flight after an expired wait

enum : int { kDrawP = 0, kDrawResidualQ = 1, kDrawResidualOneHot = 2 };

struct Args {
    const void* logits;
    const int32_t* draft_ids;
    const float* q;
    const uint8_t* has_q;
    const int32_t* cu;
    const int32_t* bitmask;
    const float* temperature;
    const int32_t* top_k;        // [B] or NULL: top-k per request (<= 0: off)
    const float* top_p;          // [B] or NULL: top-p per request (>= 1: off)
    const float* uniforms;
    const float* noise;
    int32_t* out_tokens;
    int32_t* out_num_accepted;
    unsigned long long* counters;
    uint32_t* status;
    float* diag_alpha;
    float* diag_row;
    unsigned long long* telemetry;   // [4][SPECDEC_KMAX + 1] or NULL (see specdec.h)
    int32_t B, V, max_k, W;
    int32_t slice_units;    // kUnit blocks per CTA slice
    int32_t G;              // CTAs per request (cluster size)
    int32_t bulk;           // 1: rows staged with bulk async copies; 0: plain loads
    int32_t vec_noise;      // 1: noise / q rows are 16-byte aligned (128-bit loads)
    // request schedule: cluster i verifies request order[i] (a permutation of [0, B), heaviest
    // expected work first), or request i when NULL
    const int32_t* order;
    // streaming kernel with clusters of 2 (G = 2): the first split_n requests of the order are split
    // over both CTAs of a cluster, every later cluster runs two requests, one per CTA; 0: off
    int32_t split_n;
    unsigned long long wait_ns;   // streaming kernel: limit of each wait on an mbarrier
};

// Partial result of one row pass, combined thread -> warp -> CTA -> cluster.
struct Part {
    float m;      // running max of the unscaled logits (random rows)
    float S;      // sum of exp2((z - m) * c)
    float zx;     // logit of the draft token (only the CTA owning it sets it)
    float best;   // argmax value (greedy: logit; draw: w / E)
    int idx;      // argmax index (lowest on ties), INT_MAX if none
    int flag;     // draw pass: some weight was positive
};

// ---------------------------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_addr(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Programmatic dependent launch: the schedule kernel lets the verify kernel's CTAs start early;
// they set up their barriers, then wait here until the schedule grid has completed and its
// writes are visible. A kernel launched without the dependency returns at once.
__device__ __forceinline__ void grid_dependency_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void allow_dependent_launch()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_id_x()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 :: "r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}

__device__ __forceinline__ unsigned long long global_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// try_wait: the thread may be suspended inside it for a system-dependent time
__device__ __forceinline__ uint32_t mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok;
}

// non-blocking test of a phase
__device__ __forceinline__ uint32_t mbar_test_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok;
}

// Limits below this poll with test_wait (no suspension inside a try, so a limit of 0 expires at
// the first probe that finds the phase pending); longer ones use try_wait.
constexpr unsigned long long kPollBelowNs = 1000000ull;

// Bounded wait for phase `parity` of an mbarrier. Returns false when `limit_ns` expired, or as
// soon as *abort is set (another thread of the CTA gave up on a wait).
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  unsigned long long limit_ns = kWaitLimitNs,
                                                  const volatile int* abort = nullptr)
{
    const bool poll = limit_ns < kPollBelowNs;
    if (poll ? mbar_test_wait(bar, parity) : mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (true) {
        if (abort && *abort) return false;
        if (global_ns() - t0 >= limit_ns) return false;
        if (poll ? mbar_test_wait(bar, parity) : mbar_try_wait(bar, parity)) return true;
    }
}

// ---------------------------------------------------------------------------------------------
// reductions
// ---------------------------------------------------------------------------------------------

__device__ __forceinline__ Part part_identity()
{
    Part p;
    p.m = -INFINITY; p.S = 0.f; p.zx = -INFINITY; p.best = -INFINITY; p.idx = INT_MAX; p.flag = 0;
    return p;
}

// Combine b into a. c = log2(e) / T scales logit differences for the softmax sum.
__device__ __forceinline__ void combine(Part& a, const Part& b, float c)
{
    if (b.m > a.m) {
        a.S = b.S + (a.m == -INFINITY ? 0.f : a.S * ex2((a.m - b.m) * c));
        a.m = b.m;
    } else if (b.m > -INFINITY) {
        a.S += b.S * ex2((b.m - a.m) * c);
    }
    a.zx = fmaxf(a.zx, b.zx);
    if (b.best > a.best || (b.best == a.best && b.idx < a.idx)) { a.best = b.best; a.idx = b.idx; }
    a.flag |= b.flag;
}

__device__ __forceinline__ Part shfl_part(const Part& p, int off)
{
    Part o;
    o.m = __shfl_xor_sync(0xffffffffu, p.m, off);
    o.S = __shfl_xor_sync(0xffffffffu, p.S, off);
    o.zx = __shfl_xor_sync(0xffffffffu, p.zx, off);
    o.best = __shfl_xor_sync(0xffffffffu, p.best, off);
    o.idx = __shfl_xor_sync(0xffffffffu, p.idx, off);
    o.flag = __shfl_xor_sync(0xffffffffu, p.flag, off);
    return o;
}

__device__ __forceinline__ Part warp_reduce(Part p, float c)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        Part o = shfl_part(p, off);
        combine(p, o, c);
    }
    return p;
}

struct Shared {
    uint64_t bars[kChunks];
    Part wpart[kWarps];
    Part red[2];
    Part res;
    int32_t xs[SPECDEC_KMAX];
    float us[SPECDEC_KMAX];
    float qxs[SPECDEC_KMAX];
    int32_t k, g, skip, greedy, qmode, timed_out;
    uint32_t st;
};

// Reduce one Part per thread over the whole cluster; every thread of every CTA gets the
// same (bitwise identical) result. `slot` alternates so one cluster barrier per reduction
// suffices: a slot is rewritten only after the next reduction's barrier, which every CTA
// reaches after it has finished reading the slot.
__device__ __forceinline__ Part cluster_reduce(Part p, float c, Shared& sh, int slot, int G)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    p = warp_reduce(p, c);
    if (lane == 0) sh.wpart[warp] = p;
    __syncthreads();
    if (warp == 0) {
        Part q = lane < kWarps ? sh.wpart[lane] : part_identity();
        q = warp_reduce(q, c);
        if (lane == 0) sh.red[slot] = q;
    }
    cluster_sync_all();
    if (warp == 0) {
        Part q = part_identity();
        if (lane < G) {
            const uint32_t base = map_to_rank(smem_addr(&sh.red[slot]), (uint32_t)lane);
            q.m = __uint_as_float(ld_cluster_u32(base + 0));
            q.S = __uint_as_float(ld_cluster_u32(base + 4));
            q.zx = __uint_as_float(ld_cluster_u32(base + 8));
            q.best = __uint_as_float(ld_cluster_u32(base + 12));
            q.idx = (int)ld_cluster_u32(base + 16);
            q.flag = (int)ld_cluster_u32(base + 20);
        }
        q = warp_reduce(q, c);
        if (lane == 0) sh.res = q;
    }
    __syncthreads();
    return sh.res;
}

// ---------------------------------------------------------------------------------------------
// element access
// ---------------------------------------------------------------------------------------------

// Per-position telemetry of one verified request, one warp (lane j = position j): drafts,
// grammar-eligible drafts and drafts accepted all the way through position j, and one count in
// the histogram of accepted lengths ("vLLM tour part 2", section "Telemetry and tuning").
__device__ __forceinline__ void add_telemetry(unsigned long long* tm, int lane, int k, int g, int acc)
{
    constexpr int kRow = SPECDEC_KMAX + 1;
    if (lane < k) atomicAdd(tm + 0 * kRow + lane, 1ull);
    if (lane < g) atomicAdd(tm + 1 * kRow + lane, 1ull);
    if (lane < acc) atomicAdd(tm + 2 * kRow + lane, 1ull);
    if (lane == 0) atomicAdd(tm + 3 * kRow + acc, 1ull);
}

// The same from one thread (the streaming kernel's writer, which holds little live state there).
__device__ __noinline__ void add_telemetry_serial(unsigned long long* tm, int k, int g, int acc)
{
    constexpr int kRow = SPECDEC_KMAX + 1;
    for (int j = 0; j < k; ++j) atomicAdd(tm + 0 * kRow + j, 1ull);
    for (int j = 0; j < g; ++j) atomicAdd(tm + 1 * kRow + j, 1ull);
    for (int j = 0; j < acc; ++j) atomicAdd(tm + 2 * kRow + j, 1ull);
    atomicAdd(tm + 3 * kRow + acc, 1ull);
}

template <typename ET> struct Elem;

template <> struct Elem<float> {
    static constexpr int VE = 4;        // elements per 16-byte vector
    __device__ static __forceinline__ void load(const unsigned char* s, int v, float z[VE])
    {
        const float4 f = reinterpret_cast<const float4*>(s)[v];
        z[0] = f.x; z[1] = f.y; z[2] = f.z; z[3] = f.w;
    }
};

template <> struct Elem<uint16_t> {       // bf16 bit patterns
    static constexpr int VE = 8;
    __device__ static __forceinline__ void load(const unsigned char* s, int v, float z[VE])
    {
        const uint4 u = reinterpret_cast<const uint4*>(s)[v];
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            z[2 * i] = __uint_as_float(w[i] << 16);
            z[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
};

// One logit from global memory, as fp32
template <typename ET> __device__ __forceinline__ float load_logit(const void* logits, int64_t i);
template <> __device__ __forceinline__ float load_logit<float>(const void* logits, int64_t i)
{
    return __ldg(reinterpret_cast<const float*>(logits) + i);
}
template <> __device__ __forceinline__ float load_logit<uint16_t>(const void* logits, int64_t i)
{
    return __uint_as_float((uint32_t)__ldg(reinterpret_cast<const unsigned short*>(logits) + i) << 16);
}

// Allowed-bits of vector v (VE ids) of the slice; all ones when there is no bitmask.
template <int VE>
__device__ __forceinline__ uint32_t vec_bits(const uint32_t* smask, bool has_mask, int v)
{
    if (!has_mask) return (1u << VE) - 1u;
    const int e0 = v * VE;
    return (smask[e0 >> 5] >> (e0 & 31)) & ((1u << VE) - 1u);
}

// Stage slice [lo, lo + n) of row t (and its mask words) into shared memory.
template <typename ET>
__device__ __forceinline__ void stage_row(const Args& a, Shared& sh, unsigned char* slice, uint32_t* smask,
                                          int64_t t, int64_t lo, int n, int nvec, int nw, uint32_t ph)
{
    constexpr int VE = Elem<ET>::VE;
    const ET* src = reinterpret_cast<const ET*>(a.logits) + t * (int64_t)a.V + lo;
    const int32_t* msrc = a.bitmask ? a.bitmask + t * (int64_t)a.W + (lo >> 5) : nullptr;
    if (a.bulk) {
        if (threadIdx.x == 0) {
            fence_proxy_async_smem();
            const int cv = (nvec + kChunks - 1) / kChunks;
            for (int c = 0; c < kChunks; ++c) {
                const int vb = min(nvec, c * cv), ve = min(nvec, (c + 1) * cv);
                const uint32_t bytes = (uint32_t)(ve - vb) * 16u;
                const uint32_t mbytes = (c == 0 && msrc) ? (uint32_t)nw * 4u : 0u;
                const uint32_t bar = smem_addr(&sh.bars[c]);
                mbar_arrive_expect_tx(bar, bytes + mbytes);
                if (bytes) bulk_copy_g2s(smem_addr(slice) + (uint32_t)vb * 16u,
                                         reinterpret_cast<const unsigned char*>(src) + (size_t)vb * 16u, bytes, bar);
                if (mbytes) bulk_copy_g2s(smem_addr(smask), msrc, mbytes, bar);
            }
        }
        (void)ph;
    } else {
        ET* dst = reinterpret_cast<ET*>(slice);
        ET pad;
        if constexpr (sizeof(ET) == 4) pad = -INFINITY;
        else pad = (ET)0xFF80u;                    // bf16 -inf
        for (int e = threadIdx.x; e < nvec * VE; e += kThreads) dst[e] = e < n ? src[e] : pad;
        if (msrc)
            for (int w = threadIdx.x; w < nw; w += kThreads) smask[w] = (uint32_t)msrc[w];
        __syncthreads();
    }
}

// Wait for piece c of the staged row (bulk path).
__device__ __forceinline__ void wait_piece(const Args& a, Shared& sh, int c, uint32_t ph)
{
    if (!a.bulk) return;
    if (!mbar_wait_bounded(smem_addr(&sh.bars[c]), ph)) sh.timed_out = 1;
}

// One pass over a staged row: greedy argmax, or the online-softmax (max, sum).
template <typename ET, bool kGreedy>
__device__ __forceinline__ Part row_pass(const Args& a, Shared& sh, const unsigned char* slice,
                                         const uint32_t* smask, int64_t lo, int nvec, float c, uint32_t ph)
{
    constexpr int VE = Elem<ET>::VE;
    const bool has_mask = a.bitmask != nullptr;
    Part p = part_identity();
    const int cv = (nvec + kChunks - 1) / kChunks;
    for (int ch = 0; ch < kChunks; ++ch) {
        wait_piece(a, sh, ch, ph);
        const int vb = min(nvec, ch * cv), ve = min(nvec, (ch + 1) * cv);
        for (int v = vb + (int)threadIdx.x; v < ve; v += kThreads) {
            const uint32_t bits = vec_bits<VE>(smask, has_mask, v);
            if (bits == 0u) continue;
            float z[VE];
            Elem<ET>::load(slice, v, z);
#pragma unroll
            for (int e = 0; e < VE; ++e) z[e] = ((bits >> e) & 1u) ? z[e] : -INFINITY;
            if (kGreedy) {
#pragma unroll
                for (int e = 0; e < VE; ++e)
                    if (z[e] > p.best) { p.best = z[e]; p.idx = (int)(lo + (int64_t)v * VE + e); }
            } else {
                float vm = z[0];
#pragma unroll
                for (int e = 1; e < VE; ++e) vm = fmaxf(vm, z[e]);
                if (vm == -INFINITY) continue;
                if (vm > p.m) {
                    p.S = (p.m == -INFINITY) ? 0.f : p.S * ex2((p.m - vm) * c);
                    p.m = vm;
                }
                float s = 0.f;
#pragma unroll
                for (int e = 0; e < VE; ++e) s += ex2((z[e] - p.m) * c);
                p.S += s;
            }
        }
    }
    return p;
}

// Draw pass on the staged stop / bonus row: argmax_i w_i / E_i.
template <typename ET>
__device__ __forceinline__ Part draw_pass(const Args& a, const unsigned char* slice, const uint32_t* smask,
                                          int64_t lo, int n, int nvec, int64_t t, int64_t d, int mode, int x,
                                          float m, float c, float invS)
{
    constexpr int VE = Elem<ET>::VE;
    const bool has_mask = a.bitmask != nullptr;
    const float* E = a.noise + t * (int64_t)a.V + lo;
    const float* Q = (mode == kDrawResidualQ) ? a.q + d * (int64_t)a.V + lo : nullptr;
    Part p = part_identity();
    for (int v = (int)threadIdx.x; v < nvec; v += kThreads) {
        const uint32_t bits = vec_bits<VE>(smask, has_mask, v);
        if (bits == 0u) continue;
        float z[VE], ev[VE], qv[VE];
        Elem<ET>::load(slice, v, z);
        const int e0 = v * VE;
        if (a.vec_noise) {
            // n is a multiple of 4 here, so each 4-id quarter is wholly inside or outside the row
#pragma unroll
            for (int h = 0; h < VE / 4; ++h) {
                float4 f = make_float4(1.f, 1.f, 1.f, 1.f), g = make_float4(0.f, 0.f, 0.f, 0.f);
                if (e0 + 4 * h < n) {
                    f = __ldcs(reinterpret_cast<const float4*>(E + e0) + h);
                    if (Q) g = __ldcs(reinterpret_cast<const float4*>(Q + e0) + h);
                }
                ev[4 * h] = f.x; ev[4 * h + 1] = f.y; ev[4 * h + 2] = f.z; ev[4 * h + 3] = f.w;
                qv[4 * h] = g.x; qv[4 * h + 1] = g.y; qv[4 * h + 2] = g.z; qv[4 * h + 3] = g.w;
            }
        } else {
#pragma unroll
            for (int e = 0; e < VE; ++e) {
                const bool in = e0 + e < n;
                ev[e] = in ? E[e0 + e] : 1.f;
                qv[e] = (in && Q) ? Q[e0 + e] : 0.f;
            }
        }
#pragma unroll
        for (int e = 0; e < VE; ++e) {
            if (!((bits >> e) & 1u) || !(z[e] > -INFINITY)) continue;
            const int i = (int)(lo + e0 + e);
            const float pe = ex2((z[e] - m) * c) * invS;
            float w = pe;
            if (mode == kDrawResidualQ) w = fmaxf(pe - qv[e], 0.f);
            else if (mode == kDrawResidualOneHot && i == x) w = 0.f;
            if (w > 0.f) {
                p.flag = 1;
                const float s = w / ev[e];
                if (s > p.best) { p.best = s; p.idx = i; }
            }
        }
    }
    return p;
}

template <typename ET>
__global__ void __launch_bounds__(kThreads) specdec_verify_kernel(const Args a)
{
    constexpr int VE = Elem<ET>::VE;
    extern __shared__ __align__(128) unsigned char dsm[];
    __shared__ Shared sh;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rank = (int)cluster_ctarank();
    const int64_t lo = (int64_t)rank * a.slice_units * kUnit;
    const int64_t hi = min((int64_t)a.V, lo + (int64_t)a.slice_units * kUnit);
    const int n = (int)max((int64_t)0, hi - lo);
    const int nvec = (n + VE - 1) / VE;
    const int nw = (n + 31) / 32;
    unsigned char* slice = dsm;
    uint32_t* smask = reinterpret_cast<uint32_t*>(dsm + (size_t)a.slice_units * kUnit * sizeof(ET));
    const bool writer = (rank == 0 && tid == 0);

    if (tid == 0) {
        for (int c = 0; c < kChunks; ++c) mbar_init(smem_addr(&sh.bars[c]), 1);
        fence_mbar_init();
        sh.timed_out = 0;
    }
    grid_dependency_wait();                                        // the request order is ready
    const int b = a.order ? a.order[cluster_id_x()] : (int)cluster_id_x();

    // ---- a1 ragged decode + a4 grammar-valid prefix (warp 0)
    const int32_t d0 = a.cu[b];
    const int64_t row0 = (int64_t)d0 + b;
    if (warp == 0) {
        const int32_t d1 = a.cu[b + 1], ntot = a.cu[a.B];
        const bool bad_off = a.cu[0] != 0 || d0 < 0 || d1 < d0 || d1 > ntot;
        const int k = d1 - d0;
        const float T = a.temperature[b];
        const bool tvalid = (T == 0.f) || (T >= FLT_MIN && T <= FLT_MAX);
        const bool greedy = !(T > 0.f) || !tvalid;
        const bool qmode = a.q != nullptr && (a.has_q == nullptr || a.has_q[b] != 0);
        int skip = 0, g = bad_off ? 0 : k;
        uint32_t st = 0;
        if (bad_off) { skip = 1; st = SPECDEC_ST_BAD_OFFSETS; }
        else if (k > a.max_k) { skip = 2; st = SPECDEC_ST_K_TOO_LARGE; }
        else {
            bool ok = true, allowed = true;
            if (lane < k) {
                const int32_t x = a.draft_ids ? a.draft_ids[d0 + lane] : -1;
                ok = x >= 0 && x < a.V;
                allowed = ok;
                if (ok && a.bitmask)
                    allowed = ((uint32_t)a.bitmask[(row0 + lane) * (int64_t)a.W + (x >> 5)] >> (x & 31)) & 1u;
                sh.xs[lane] = x;
                sh.us[lane] = a.uniforms[row0 + lane];
                sh.qxs[lane] = (qmode && ok && !greedy) ? a.q[(int64_t)(d0 + lane) * a.V + x] : 0.f;
            }
            const unsigned inval = __ballot_sync(0xffffffffu, lane < k && !allowed);
            const unsigned badid = __ballot_sync(0xffffffffu, lane < k && !ok);
            if (inval) g = __ffs(inval) - 1;
            if (badid) st |= SPECDEC_ST_BAD_DRAFT_ID;
            if (!tvalid) st |= SPECDEC_ST_BAD_TEMPERATURE;
        }
        if (lane == 0) {
            sh.k = k; sh.g = g; sh.skip = skip; sh.greedy = greedy; sh.qmode = qmode; sh.st = st;
        }
    }
    __syncthreads();

    const int k = sh.k, g = sh.g, skip = sh.skip;
    const bool greedy = sh.greedy != 0, qmode = sh.qmode != 0;
    uint32_t st = sh.st;
    const float T = a.temperature[b];
    const float c = greedy ? 0.f : (float)(1.4426950408889634 / (double)T);   // log2(e) / T

    if (writer && a.status) a.status[b] = 0u;      // bits are OR-ed in at the end
    if (writer && skip != 1) {
        if (a.diag_alpha) for (int j = 0; j < k; ++j) a.diag_alpha[d0 + j] = NAN;
        if (a.diag_row) for (int j = 0; j <= k; ++j) { a.diag_row[2 * (row0 + j)] = NAN; a.diag_row[2 * (row0 + j) + 1] = NAN; }
    }

    int acc_len = 0, emitted = -1;
    uint32_t ph = 0;
    int slot = 0;
    if (skip == 0) {
        acc_len = k;
        for (int j = 0; j <= k; ++j) {
            const int64_t t = row0 + j;
            const int64_t d = (int64_t)d0 + j;
            const bool bonus = (j == k);
            const int x = bonus ? -1 : sh.xs[j];

            // ---- a2/a3: stage the row slice (logits + mask words)
            stage_row<ET>(a, sh, slice, smask, t, lo, n, nvec, nw, ph);

            // ---- a5/a6: one pass over the slice
            Part p = greedy ? row_pass<ET, true>(a, sh, slice, smask, lo, nvec, c, ph)
                            : row_pass<ET, false>(a, sh, slice, smask, lo, nvec, c, ph);
            ph ^= 1u;
            if (!greedy && !bonus && tid == 0 && x >= lo && x < hi) {
                float z[VE];
                Elem<ET>::load(slice, (int)((x - lo) / VE), z);
                p.zx = z[(x - lo) % VE];
            }
            const Part r = cluster_reduce(p, c, sh, slot, a.G);
            slot ^= 1;

            if (greedy) {
                if (r.idx == INT_MAX) {                       // nothing allowed in this row
                    st |= SPECDEC_ST_EMPTY_MASK_ROW;
                    if (writer && a.diag_row) { a.diag_row[2 * t] = -INFINITY; a.diag_row[2 * t + 1] = NAN; }
                    acc_len = j; emitted = -1;
                    break;
                }
                if (writer && a.diag_row) { a.diag_row[2 * t] = r.best; a.diag_row[2 * t + 1] = NAN; }
                if (bonus) { emitted = r.idx; break; }
                const bool accept = (j < g) && (x == r.idx);
                if (writer && a.diag_alpha) a.diag_alpha[d] = accept ? 1.f : 0.f;
                if (accept) { if (writer) a.out_tokens[t] = x; continue; }
                acc_len = j; emitted = r.idx;                 // recovered = target argmax
                break;
            }

            if (r.m == -INFINITY) {
                st |= SPECDEC_ST_EMPTY_MASK_ROW;
                if (writer && a.diag_row) { a.diag_row[2 * t] = -INFINITY; a.diag_row[2 * t + 1] = 0.f; }
                acc_len = j; emitted = -1;
                break;
            }
            const float m = r.m, S = r.S;
            if (writer && a.diag_row) { a.diag_row[2 * t] = m / T; a.diag_row[2 * t + 1] = S; }
            int mode = kDrawP;
            if (!bonus) {
                // ---- a7: acceptance probability, a8: strict comparison with the draw
                float alpha = 0.f;
                if (j < g) {
                    const float px = (r.zx > -INFINITY) ? ex2((r.zx - m) * c) / S : 0.f;
                    if (qmode) {
                        const float qx = sh.qxs[j];
                        alpha = (px <= 0.f) ? 0.f : (qx <= px ? 1.f : px / qx);
                    } else {
                        alpha = px;
                    }
                }
                if (writer && a.diag_alpha) a.diag_alpha[d] = alpha;
                if (sh.us[j] < alpha) { if (writer) a.out_tokens[t] = x; continue; }
                mode = qmode ? kDrawResidualQ : kDrawResidualOneHot;
            }
            // ---- a9/a10: recovered or bonus token by exponential race over the staged slice
            const float invS = 1.f / S;
            Part dp = draw_pass<ET>(a, slice, smask, lo, n, nvec, t, d, mode, x, m, c, invS);
            Part dr = cluster_reduce(dp, c, sh, slot, a.G);
            slot ^= 1;
            if (mode == kDrawResidualQ && !dr.flag) {        // empty residual: fall back to p
                dp = draw_pass<ET>(a, slice, smask, lo, n, nvec, t, d, kDrawP, x, m, c, invS);
                dr = cluster_reduce(dp, c, sh, slot, a.G);
                slot ^= 1;
            }
            emitted = dr.idx == INT_MAX ? -1 : dr.idx;
            acc_len = j;
            break;
        }
    }

    // ---- a11: emit, count
    if (writer) {
        if (skip == 0) {
            a.out_tokens[row0 + acc_len] = emitted;
            for (int j = acc_len + 1; j <= k; ++j) a.out_tokens[row0 + j] = -1;
            atomicAdd(&a.counters[0], (unsigned long long)k);
            atomicAdd(&a.counters[1], (unsigned long long)(k - g));
            atomicAdd(&a.counters[2], (unsigned long long)g);
            atomicAdd(&a.counters[3], (unsigned long long)acc_len);
        } else if (skip == 2) {
            for (int j = 0; j <= k; ++j) a.out_tokens[row0 + j] = -1;
        }
        a.out_num_accepted[b] = skip == 0 ? acc_len : 0;
    }
    if (a.telemetry && skip == 0 && rank == 0 && warp == 0) add_telemetry(a.telemetry, lane, k, g, acc_len);
    __syncthreads();
    if (sh.timed_out) {
        st |= SPECDEC_ST_DEVICE_TIMEOUT;
        // copies that missed their deadline: wait once more (bounded) before the CTA exits
        if (tid == 0)
            for (int ch = 0; ch < kChunks; ++ch) (void)mbar_wait_bounded(smem_addr(&sh.bars[ch]), ph ^ 1u);
    }
    if (a.status && tid == 0) {
        if (rank == 0) atomicOr(&a.status[b], st & ~SPECDEC_ST_DEVICE_TIMEOUT);
        if (st & SPECDEC_ST_DEVICE_TIMEOUT) atomicOr(&a.status[b], SPECDEC_ST_DEVICE_TIMEOUT);
    }
    // no CTA leaves while another may still read its shared memory
    cluster_sync_all();
}

// ---------------------------------------------------------------------------------------------
// streaming kernel: one CTA per request
// ---------------------------------------------------------------------------------------------
//
// Dense requests (no bitmask, or a bitmask that allows most ids): warp 0 is a producer whose
// lane 0 issues cp.async.bulk copies of 32 KB chunks (logits + mask words of a row; logits +
// noise [+ q] + mask words of the draw row) into a ring of kStages shared-memory stages, each
// with a "full" and an "empty" mbarrier. Warps 1..8 consume chunk by chunk, reduce across the
// CTA at the end of a row and post the decision (next row / draw / done) through a shared word
// and a "decision" mbarrier. While a decision is pending the producer has already queued up to
// kSpec chunks of the next row, so HBM keeps streaming across row boundaries; if the request
// stops, the consumers drain those chunks unused.
//
// Sparse requests (a bitmask allowing few ids, judged from 32 words of the first row's mask):
// the consumers scan each row's mask words, list the 16-byte groups holding an allowed id
// (a block-wide prefix sum keeps the list in id order), and gather only those groups of
// logits -- and, for the draw, of noise and q -- with 128-bit loads. At 5 % of ids allowed
// this moves 12 % (fp32) or 21 % (bf16) of the row's bytes instead of all of it.
//
// No cross-CTA synchronisation exists on this path: every reduction is inside one CTA.

constexpr int kConsumers = 256;
constexpr int kConsumerWarps = kConsumers / 32;
constexpr int kStreamThreads = kConsumers + 32;
constexpr int kResidentPerSM = 2;              // streaming CTAs per SM (registers and shared memory)
constexpr int kStageBytes = 32 * 1024;
constexpr int kStages = 3;
constexpr int kSpec = 2;
constexpr int kRingBytes = kStages * kStageBytes;
// sparse requests reuse the ring's memory: a list of allowed 16-byte groups, then the data those
// groups gather (cp.async), in batches
constexpr int kListBytes = 32 * 1024;
constexpr int kListCap = kListBytes / 4;       // list entries
constexpr int kDataOff = kListBytes;
constexpr int kDataBytes = kRingBytes - kListBytes;
constexpr int kGatherCap = kDataBytes / 16;    // logits groups per gather batch
constexpr int kSegWords = 5120;                // mask words scanned per pass (20 per consumer thread)

constexpr int kCandCap = 2048;                 // top-k / top-p: candidate keys held on chip

enum : int { kDecNextRow = 1, kDecDrawP = 2, kDecDrawQ = 3, kDecDrawOneHot = 4, kDecDone = 5,
              kDecRescan = 6 };   // stream the same row once more (a top-k / top-p digit pass)

__host__ __device__ constexpr int ids_per_stage(int bytes_per_id)
{
    // ids (a multiple of kUnit) whose bytes plus their mask words (1/8 byte each) fit a stage
    return ((kStageBytes * 8) / (bytes_per_id * 8 + 1)) / kUnit * kUnit;
}

template <typename ET> struct Geom {
    static constexpr int ES = (int)sizeof(ET);
    static constexpr int kRowIds = ids_per_stage(ES);
    static constexpr int kRowMaskOff = kRowIds * ES;
    // draw chunks: logits, noise, [q,] mask words
    static constexpr int kDrawIdsQ = ids_per_stage(ES + 8);
    static constexpr int kDrawIdsE = ids_per_stage(ES + 4);
    __host__ __device__ static constexpr int draw_ids(bool q) { return q ? kDrawIdsQ : kDrawIdsE; }
    __host__ __device__ static constexpr int noise_off(bool q) { return draw_ids(q) * ES; }
    __host__ __device__ static constexpr int q_off(bool q) { return draw_ids(q) * (ES + 4); }
    __host__ __device__ static constexpr int dmask_off(bool q) { return draw_ids(q) * (ES + 4 + (q ? 4 : 0)); }
    static_assert(kRowMaskOff + kRowIds / 8 <= kStageBytes, "row chunk overflows a stage");
    static_assert(kDrawIdsQ * (ES + 8) + kDrawIdsQ / 8 <= kStageBytes, "draw chunk overflows a stage");
    static_assert(kDrawIdsE * (ES + 4) + kDrawIdsE / 8 <= kStageBytes, "draw chunk overflows a stage");
    static_assert(kRowMaskOff % 16 == 0 && (kDrawIdsQ * ES) % 16 == 0 && (kDrawIdsE * ES) % 16 == 0,
                  "stage sections must be 16-byte aligned");
    static constexpr int kSafeWords = kListCap / (32 / Elem<ET>::VE);   // words whose groups always fit the list
    static_assert(kSafeWords % 4 == 0 && kSafeWords <= kSegWords, "sparse segment sizes");
};

struct StreamShared {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t dec;
    uint64_t pbar[2];                      // cluster exchange: partials of the G CTAs landed
    Part wpart[2][kConsumerWarps];
    Part parts[2][kMaxCluster];            // cluster exchange: one partial per CTA of the request
    Part xres[2];                          // cluster exchange: the folded result, for every consumer
    int32_t scan[kConsumerWarps];
    int32_t xs[SPECDEC_KMAX];
    float us[SPECDEC_KMAX];
    float qxs[SPECDEC_KMAX];
    int32_t g, greedy, qmode, sparse, timed_out, dec_code;
    uint32_t st;
    float c;
    uint32_t issued;                       // chunks the producer issued (set when it is done)
    // top-k / top-p threshold search: the 256 bins of one pass. Masses are sums of 24-bit
    // integers kept as the sums of their low and high 12 bits (exact in 32 bits for V <= 2^20;
    // two 32-bit shared atomics measured far faster than one 64-bit one under contention).
    uint32_t fcnt[256];
    uint32_t flo[256], fhi[256];
    uint32_t fw_cnt[kConsumerWarps], fw_kmin[kConsumerWarps], fw_kmax[kConsumerWarps];  // per-warp partials
    float fw_a[kConsumerWarps];
    unsigned long long fw_m[kConsumerWarps], fw_m2[kConsumerWarps];
    unsigned long long ftail_m;          // first pass: tail mass in units of 2^-54
    uint32_t fsel_digit;                 // chosen digit (0xffffffff: none)
    uint32_t fsel_pad;
    unsigned long long fsel_cnt;         // count above the chosen digit (this level)
    unsigned long long fsel_mass, fsel_at;   // mass above the chosen digit / of the digit itself (2^-40)
    unsigned long long ftot_mass;        // mass of every element counted in this pass (2^-40)
    unsigned long long fsel_P;           // the top-p target mass the choice used (2^-40)
    unsigned long long fsel_n;           // elements in the chosen digit (first top-p pass: a bound)
    uint32_t fc_kmin, fc_kmax;           // collection pass: the chosen bin's smallest / largest key
    unsigned long long fc_mbin;          // collection pass: the chosen bin's mass (its units)
    unsigned long long fc_mabove;        // collection pass: mass above the bin, units of 2^-40
    uint32_t fncand;                     // candidates appended by the last collection pass
    uint32_t fcand[kCandCap];            // candidate keys (in no particular order)
    int32_t fk;
    float fp;
};

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}

__device__ __forceinline__ void consumer_sync()
{
    asm volatile("bar.sync 1, %0;" :: "n"(kConsumers) : "memory");
}

__device__ __forceinline__ void st_cluster_u32(uint32_t addr, uint32_t v)
{
    asm volatile("st.shared::cluster.u32 [%0], %1;" :: "r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr)
{
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" :: "r"(cluster_addr) : "memory");
}

__device__ __forceinline__ uint32_t mbar_try_wait_cluster(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok;
}

__device__ __forceinline__ uint32_t mbar_test_wait_cluster(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok;
}

__device__ __forceinline__ bool mbar_wait_cluster_bounded(uint32_t bar, uint32_t parity, unsigned long long limit_ns,
                                                          const volatile int* abort)
{
    const bool poll = limit_ns < kPollBelowNs;
    if (poll ? mbar_test_wait_cluster(bar, parity) : mbar_try_wait_cluster(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (true) {
        if (*abort) return false;
        if (global_ns() - t0 >= limit_ns) return false;
        if (poll ? mbar_test_wait_cluster(bar, parity) : mbar_try_wait_cluster(bar, parity)) return true;
    }
}

// Bulk prefetch of [src, src + bytes) into L2 (16-byte aligned, a multiple of 16 bytes).
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all()
{
    asm volatile("cp.async.wait_all;" ::: "memory");
}

__device__ __forceinline__ float fast_rcp(float x)
{
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// The request's offsets, checked the same way by producer and consumers.
struct ReqShape {
    int32_t d0, k, skip;   // skip: 0 ok, 1 bad offsets, 2 k > max_k
    int64_t row0;
};

__device__ __forceinline__ ReqShape request_shape(const Args& a, int b)
{
    ReqShape r;
    const int32_t d0 = a.cu[b], d1 = a.cu[b + 1], ntot = a.cu[a.B];
    r.d0 = d0;
    r.k = d1 - d0;
    r.row0 = (int64_t)d0 + b;
    r.skip = (a.cu[0] != 0 || d0 < 0 || d1 < d0 || d1 > ntot) ? 1 : (r.k > a.max_k ? 2 : 0);
    return r;
}

// Top-k / top-p of request b, read the same way by producer and consumers: k <= 0 and top_p >= 1
// are off, a top_p that is not a number in (0, 1] is off (and flagged); greedy requests ignore both
// (the argmax is always kept).
struct Filter {
    int k;
    float p;
    bool bad_p, on;
};

// What a draft row's statistics pass knows about the draft token x (the acceptance bound of the
// streaming kernel): whether fewer than k logits lie above it (cok), the mass above it (A) and its
// own mass (ex), both against the row's reference, its q and uniform. A top-p search may accept the
// row as soon as its kept mass is bounded tightly enough (on: the data is valid).
struct Settle {
    bool on, cok, qmode;
    float A, ex, qx, u;
};

__device__ __forceinline__ bool request_greedy(const Args& a, int b)
{
    const float T = a.temperature[b];
    const bool tvalid = (T == 0.f) || (T >= FLT_MIN && T <= FLT_MAX);
    return !(T > 0.f) || !tvalid;
}

__device__ __forceinline__ Filter request_filter(const Args& a, int b)
{
    Filter f;
    f.k = a.top_k ? a.top_k[b] : 0;
    f.p = 1.f;
    f.bad_p = false;
    if (a.top_p) {
        const float v = a.top_p[b];
        if (v > 0.f && v < 1.f) f.p = v;
        else if (!(v >= 1.f)) f.bad_p = true;
    }
    f.on = (f.k > 0 || f.p < 1.f) && !request_greedy(a, b);
    return f;
}

// Bit e set when z[e] is above -inf (a NaN never is)
template <int N>
__device__ __forceinline__ uint32_t finite_bits(const float* z)
{
    uint32_t b = 0u;
#pragma unroll
    for (int e = 0; e < N; ++e) b |= (z[e] > -INFINITY ? 1u : 0u) << e;
    return b;
}

// The logit whose logit_key is `key` (zero comes back as +0)
__device__ __forceinline__ float key_logit(uint32_t key)
{
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

// First-pass bin of an element by its mass e = exp2(z * c - MC) in (0, ~1]: 8 bins per halving
// (exponent and 3 mantissa bits), from bin 8 (2^-30) to 255 (1); bin 0 (the tail) holds
// everything below 2^-30. Non-decreasing in e, hence in the logit: every element of a higher bin
// has a larger logit. All elements of a bin from 8 up share e's binary exponent, so the bin's mass
// is its elements' 24-bit significands summed exactly, times 2^(exponent - 23).
__device__ __forceinline__ uint32_t mass_bin(float e)
{
    // bits 30..20 of e are its exponent and top 3 mantissa bits: 8 * exponent + those 3 bits
    const int d = (int)(__float_as_uint(e) >> 20) - (97 * 8 - 8);
    return d < 8 ? 0u : (uint32_t)min(d, 255);
}

// The 24-bit significand of e (bins 8..255) or e in units of 2^-54 (the tail, e < 2^-30): an
// integer below 2^24 whose sum over a bin, times bin_scale, is the bin's mass.
__device__ __forceinline__ uint32_t mass_units(float e, bool tail)
{
    return tail ? __float2uint_rn(e * 0x1p54f) : ((__float_as_uint(e) & 0x7fffffu) | 0x800000u);
}

// The exponent of mass bin mb's unit: its elements' masses are mass_units times 2^bin_exp
// (2^(exponent - 23) for bins 8..255, 2^-54 for the tail)
__device__ __forceinline__ int bin_exp(uint32_t mb)
{
    return mb == 0u ? -54 : (int)(mb >> 3) - 54;
}

// units * 2^e as a fixed-point mass in units of 2^-40 (bits below 2^-40 dropped). Masses are at
// most 1 each (relative to the row maximum), so sums over up to 2^20 elements stay below 2^60.
__device__ __forceinline__ unsigned long long fx40(unsigned long long units, int e)
{
    const int s = e + 40;
    return s >= 0 ? (units << s) : (s > -64 ? (units >> -s) : 0ull);
}

// Order-preserving 32-bit key of a logit (its fp32 bits): a larger logit has a larger key, and
// equal logits have equal keys (-0 and +0 both map to the key of +0).
__device__ __forceinline__ uint32_t logit_key(float z)
{
    const uint32_t u = z == 0.f ? 0u : __float_as_uint(z);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Sparse or dense: a warp reads up to 32 mask words of the request's first row; the request
// runs the sparse path when fewer than half of those bits are set. Producer and consumers
// evaluate the same words, so they agree without communicating. Only aligned layouts qualify.
__device__ __forceinline__ bool request_is_sparse(const Args& a, int64_t row0, int lane)
{
    if (a.bitmask == nullptr || !a.bulk) return false;
    const int nw = min(a.W, 32);
    const uint32_t w = lane < nw ? (uint32_t)a.bitmask[row0 * (int64_t)a.W + lane] : 0u;
    const int ones = __reduce_add_sync(0xffffffffu, (unsigned)__popc(w));
    return 2 * ones < nw * 32;
}

// exp2 of logit z against the running reference mc = round(m * c): fused as z*c - mc so that
// the rounding of mc is one common factor of every term (it cancels in p = e / S).
__device__ __forceinline__ float ex2_scaled(float z, float c, float mc)
{
    return ex2(fmaf(z, c, -mc));
}

// ---- batched per-thread processing: NB 16-byte groups at once, so that loads, exponentials and
// the max / sum trees of different groups are independent (ILP instead of one long chain)

template <int N>
__device__ __forceinline__ float tree_max(const float* v)
{
    float t[N];
#pragma unroll
    for (int i = 0; i < N; ++i) t[i] = v[i];
#pragma unroll
    for (int w = N / 2; w >= 1; w /= 2)
#pragma unroll
        for (int i = 0; i < w; ++i) t[i] = fmaxf(t[i], t[i + w]);
    return t[0];
}

template <int N>
__device__ __forceinline__ float tree_sum(const float* v)
{
    float t[N];
#pragma unroll
    for (int i = 0; i < N; ++i) t[i] = v[i];
#pragma unroll
    for (int w = N / 2; w >= 1; w /= 2)
#pragma unroll
        for (int i = 0; i < w; ++i) t[i] += t[i + w];
    return t[0];
}

// Greedy fold of N values with ids ids[i] (in any order): max, lowest id on ties.
template <int N>
__device__ __forceinline__ void argmax_batch(Part& p, const float* z, const int* ids)
{
    const float bm = tree_max<N>(z);
    if (bm > -INFINITY && bm >= p.best) {
        int id = INT_MAX;
#pragma unroll
        for (int i = 0; i < N; ++i) id = (z[i] == bm) ? min(id, ids[i]) : id;
        if (bm > p.best || id < p.idx) { p.best = bm; p.idx = id; }
    }
}

// Online-softmax fold of N masked logits against the running reference mc = round(m * c).
template <int N>
__device__ __forceinline__ void softmax_batch(Part& p, float& mc, const float* z, float c)
{
    const float bm = tree_max<N>(z);
    if (!(bm > -INFINITY)) return;
    if (bm > p.m) {
        const float nmc = bm * c;
        p.S = (p.m == -INFINITY) ? 0.f : p.S * ex2(mc - nmc);
        p.m = bm;
        mc = nmc;
    }
    float e[N];
#pragma unroll
    for (int i = 0; i < N; ++i) e[i] = ex2_scaled(z[i], c, mc);
    p.S += tree_sum<N>(e);
}

// Draw fold of N candidates with ids ids[i] (in any order): w from p (and q), score w / E;
// -1 marks "no candidate".
template <int N>
__device__ __forceinline__ void draw_batch(Part& p, const float* z, const float* E, const float* qv, const int* ids,
                                           int code, int x, float c, float MC, float invS)
{
    float sc[N];
    int any = 0;
#pragma unroll
    for (int i = 0; i < N; ++i) {
        const float pe = ex2_scaled(z[i], c, MC) * invS;        // z = -inf gives 0
        float w = pe;
        if (code == kDecDrawQ) w = fmaxf(pe - qv[i], 0.f);
        else if (code == kDecDrawOneHot) w = (ids[i] == x) ? 0.f : pe;
        const bool cand = w > 0.f && z[i] > -INFINITY;      // a forbidden / absent id never qualifies
        any |= cand ? 1 : 0;
        sc[i] = cand ? w * fast_rcp(E[i]) : -1.f;
    }
    p.flag |= any;
    const float bm = tree_max<N>(sc);
    if (bm > 0.f && bm >= p.best) {            // ids in any order: lowest id on ties
        int id = INT_MAX;
#pragma unroll
        for (int i = 0; i < N; ++i) id = (sc[i] == bm) ? min(id, ids[i]) : id;
        if (bm > p.best || id < p.idx) { p.best = bm; p.idx = id; }
    }
}


// ---- raw 16-byte groups and their max

template <typename ET> struct Raw;
template <> struct Raw<float> {
    static constexpr uint32_t kNegInf = 0xff800000u;                  // fp32 -inf
};
template <> struct Raw<uint16_t> {
    static constexpr uint32_t kNegInf = 0xff80ff80u;                  // two bf16 -inf
};

template <typename ET>
__device__ __forceinline__ void unpack_raw(const uint4 u, float* z)
{
    if constexpr (sizeof(ET) == 4) {
        z[0] = __uint_as_float(u.x); z[1] = __uint_as_float(u.y); z[2] = __uint_as_float(u.z); z[3] = __uint_as_float(u.w);
    } else {
        z[0] = __uint_as_float(u.x << 16); z[1] = __uint_as_float(u.x & 0xffff0000u);
        z[2] = __uint_as_float(u.y << 16); z[3] = __uint_as_float(u.y & 0xffff0000u);
        z[4] = __uint_as_float(u.z << 16); z[5] = __uint_as_float(u.z & 0xffff0000u);
        z[6] = __uint_as_float(u.w << 16); z[7] = __uint_as_float(u.w & 0xffff0000u);
    }
}

__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// Max of NB raw groups: exact either way (bf16 values compare exactly in bf16x2).
template <typename ET, int NB>
__device__ __forceinline__ float raw_max(const uint4* raw, const float* z)
{
    if constexpr (sizeof(ET) == 2) {
        uint32_t t[NB * 4];
#pragma unroll
        for (int u = 0; u < NB; ++u) { t[4 * u] = raw[u].x; t[4 * u + 1] = raw[u].y; t[4 * u + 2] = raw[u].z; t[4 * u + 3] = raw[u].w; }
#pragma unroll
        for (int w = NB * 2; w >= 1; w /= 2)
#pragma unroll
            for (int i = 0; i < w; ++i) t[i] = bf16x2_max(t[i], t[i + w]);
        return fmaxf(__uint_as_float(t[0] << 16), __uint_as_float(t[0] & 0xffff0000u));
    } else {
        return tree_max<NB * 4>(z);
    }
}

// Greedy fold with ids base + u * stride + e (increasing): max, lowest id on ties.
template <int NB, int VE>
__device__ __forceinline__ void argmax_lazy(Part& p, const float* z, float bm, int base, int stride)
{
    if (bm > p.best) {                         // strict: an equal earlier best keeps its lower id
        int id = INT_MAX;
#pragma unroll
        for (int u = NB - 1; u >= 0; --u)
#pragma unroll
            for (int e = VE - 1; e >= 0; --e) id = (z[u * VE + e] == bm) ? base + u * stride + e : id;
        p.best = bm;
        p.idx = id;
    }
}

// Online-softmax fold of N masked logits whose max is bm.
template <int N>
__device__ __forceinline__ void softmax_fold_max(Part& p, float& mc, const float* z, float bm, float c)
{
    if (!(bm > -INFINITY)) return;
    if (bm > p.m) {
        const float nmc = bm * c;
        p.S = (p.m == -INFINITY) ? 0.f : p.S * ex2(mc - nmc);
        p.m = bm;
        mc = nmc;
    }
    float e[N];
#pragma unroll
    for (int i = 0; i < N; ++i) e[i] = ex2_scaled(z[i], c, mc);
    p.S += tree_sum<N>(e);
}

// softmax_fold_max, and besides the count (cnt) and the mass (A, same reference as p.S) of the
// elements whose logit is above zx: on a top-k / top-p row these bound the draft token's filtered
// probability without the threshold search (the acceptance bound in the streaming kernel)
template <int N>
__device__ __forceinline__ void softmax_fold_max_above(Part& p, float& mc, float& A, uint32_t& cnt, const float* z,
                                                       float bm, float c, float zx)
{
    if (!(bm > -INFINITY)) return;
    if (bm > p.m) {
        const float nmc = bm * c;
        const float f = (p.m == -INFINITY) ? 0.f : ex2(mc - nmc);
        p.S = (p.m == -INFINITY) ? 0.f : p.S * f;
        A = (p.m == -INFINITY) ? 0.f : A * f;
        p.m = bm;
        mc = nmc;
    }
    float e[N], ea[N];
#pragma unroll
    for (int i = 0; i < N; ++i) {
        e[i] = ex2_scaled(z[i], c, mc);
        const bool above = z[i] > zx;
        ea[i] = above ? e[i] : 0.f;
        cnt += above ? 1u : 0u;
    }
    p.S += tree_sum<N>(e);
    A += tree_sum<N>(ea);
}

// Draw fold of NB groups (ids base + u * stride + e); xslot = position of the one-hot draft or -1.
template <int NB, int VE>
__device__ __forceinline__ void draw_lazy(Part& p, const float* z, const float* E, const float* qv, int base, int stride,
                                          int xslot, int code, float c, float MC, float invS)
{
    constexpr int N = NB * VE;
    float sc[N];
    int any = 0;
#pragma unroll
    for (int i = 0; i < N; ++i) {
        const float pe = ex2_scaled(z[i], c, MC) * invS;        // z = -inf gives 0
        float w = pe;
        if (code == kDecDrawQ) w = fmaxf(pe - qv[i], 0.f);
        else if (code == kDecDrawOneHot && i == xslot) w = 0.f;
        const bool cand = w > 0.f && z[i] > -INFINITY;      // a forbidden / absent id never qualifies
        any |= cand ? 1 : 0;
        sc[i] = cand ? w * fast_rcp(E[i]) : -1.f;
    }
    p.flag |= any;
    const float bm = tree_max<N>(sc);
    if (bm > 0.f && bm > p.best) {
        int id = INT_MAX;
#pragma unroll
        for (int u = NB - 1; u >= 0; --u)
#pragma unroll
            for (int e = VE - 1; e >= 0; --e) id = (sc[u * VE + e] == bm) ? base + u * stride + e : id;
        p.best = bm;
        p.idx = id;
    }
}

// ---- one-pass race over a row that needs no acceptance ratio first: the bonus row of a sampled
// request, or a row of a sampled model-free request. The bonus token is argmax_i p_i / E_i and
// a model-free recovered token argmax_{i != x} p_i / E_i; both only compare ratios of
// exp2(z * c) terms, so they need no normaliser and fold in the same pass as the softmax
// statistics (which still give p(x) for the acceptance test). The terms are kept against a
// running reference mc that is a whole number, so raising it rescales the sum and the best score
// by an exact power of two (Part.flag carries mc's bits through the reductions).

// 2^d for a whole number d <= 0 (0 below 2^-126)
__device__ __forceinline__ float pow2_int(float d)
{
    return d < -126.f ? 0.f : __int_as_float(((int)d + 127) << 23);
}

// Raise a race partial's reference to cover a new maximum bm (finite, above p.m).
__device__ __forceinline__ void race_raise(Part& p, float& mc, float bm, float c)
{
    const float nmc = ceilf(bm * c);
    if (p.m == -INFINITY) {
        mc = nmc;
    } else if (nmc > mc) {
        const float f = pow2_int(mc - nmc);
        p.S *= f;
        if (p.best > 0.f) {
            p.best *= f;
            if (!(p.best > 0.f)) { p.best = -INFINITY; p.idx = INT_MAX; }
        }
        mc = nmc;
    }
    p.m = bm;
}

// Race fold of NB groups (ids base + u * stride + e, increasing) whose max is bm; xslot = the
// excluded draft token's position or -1.
template <int NB, int VE>
__device__ __forceinline__ void race_lazy(Part& p, float& mc, const float* z, const float* E, float bm, int base,
                                          int stride, int xslot, float c)
{
    constexpr int N = NB * VE;
    if (!(bm > -INFINITY)) return;
    if (bm > p.m) race_raise(p, mc, bm, c);
    float e[N], sc[N];
#pragma unroll
    for (int i = 0; i < N; ++i) e[i] = ex2(fmaf(z[i], c, -mc));             // z = -inf gives 0
    p.S += tree_sum<N>(e);
#pragma unroll
    for (int i = 0; i < N; ++i) sc[i] = (e[i] > 0.f && i != xslot) ? e[i] * fast_rcp(E[i]) : -1.f;
    const float bs = tree_max<N>(sc);
    if (bs > 0.f && bs > p.best) {               // strict: an equal earlier best keeps its lower id
        int id = INT_MAX;
#pragma unroll
        for (int u = NB - 1; u >= 0; --u)
#pragma unroll
            for (int e2 = VE - 1; e2 >= 0; --e2) id = (sc[u * VE + e2] == bs) ? base + u * stride + e2 : id;
        p.best = bs;
        p.idx = id;
    }
}

// Race fold of N candidates with ids ids[i] (in any order, -1 = unused slot); id x is excluded.
template <int N>
__device__ __forceinline__ void race_batch(Part& p, float& mc, const float* z, const float* E, const int* ids, int x,
                                           float c)
{
    const float bm = tree_max<N>(z);
    if (!(bm > -INFINITY)) return;
    if (bm > p.m) race_raise(p, mc, bm, c);
    float e[N], sc[N];
#pragma unroll
    for (int i = 0; i < N; ++i) e[i] = ex2(fmaf(z[i], c, -mc));
    p.S += tree_sum<N>(e);
#pragma unroll
    for (int i = 0; i < N; ++i) sc[i] = (e[i] > 0.f && ids[i] != x) ? e[i] * fast_rcp(E[i]) : -1.f;
    const float bs = tree_max<N>(sc);
    if (bs > 0.f && bs >= p.best) {
        int id = INT_MAX;
#pragma unroll
        for (int i = 0; i < N; ++i) id = (sc[i] == bs) ? min(id, ids[i]) : id;
        if (bs > p.best || id < p.idx) { p.best = bs; p.idx = id; }
    }
}

// Combine race partial b into a: both rescaled to the larger reference (exact powers of two).
__device__ __forceinline__ void combine_race(Part& a, const Part& b)
{
    a.zx = fmaxf(a.zx, b.zx);
    if (!(b.m > -INFINITY)) return;
    if (!(a.m > -INFINITY)) { a.m = b.m; a.S = b.S; a.best = b.best; a.idx = b.idx; a.flag = b.flag; return; }
    const float ma = __int_as_float(a.flag), mb = __int_as_float(b.flag), M = fmaxf(ma, mb);
    const float fa = pow2_int(ma - M), fb = pow2_int(mb - M);
    a.S = a.S * fa + b.S * fb;
    float ba = a.best > 0.f ? a.best * fa : -INFINITY, bb = b.best > 0.f ? b.best * fb : -INFINITY;
    int ia = a.idx, ib = b.idx;
    if (!(ba > 0.f)) { ba = -INFINITY; ia = INT_MAX; }
    if (!(bb > 0.f)) { bb = -INFINITY; ib = INT_MAX; }
    if (bb > ba || (bb == ba && ib < ia)) { ba = bb; ia = ib; }
    a.best = ba;
    a.idx = ia;
    a.m = fmaxf(a.m, b.m);
    a.flag = __float_as_int(M);
}

template <bool kRace>
__device__ __forceinline__ void combine_any(Part& a, const Part& b, float c)
{
    if constexpr (kRace) combine_race(a, b);
    else combine(a, b, c);
}

// ---- the end-of-row reduction of the streaming kernel, shallow: a warp takes its maxima (and
// the lowest index of its best score) with redux.sync on order-preserving images, rescales each
// lane's sum once to the warp's maximum and adds the sums by shuffles; then every consumer thread
// folds the warps' partials in warp order, each rescaled once to the CTA's maximum.

// Order-preserving 32-bit image of a float that is not NaN (a < b iff ordered(a) < ordered(b));
// the map is its own inverse.
__device__ __forceinline__ int ordered(float f)
{
    const int i = __float_as_int(f);
    return i ^ ((i >> 31) & 0x7fffffff);
}

__device__ __forceinline__ float unordered(int i)
{
    return __int_as_float(i ^ ((i >> 31) & 0x7fffffff));
}

// A race partial's best score rescaled by the power of two f; a score that underflows drops out.
__device__ __forceinline__ void race_scale_best(float& best, int& idx, float f)
{
    best = best > 0.f ? best * f : -INFINITY;
    if (!(best > 0.f)) { best = -INFINITY; idx = INT_MAX; }
}

// Every lane of the warp gets the fold of the lanes' partials (bitwise the same in every lane:
// the butterfly adds commute).
template <bool kRace>
__device__ __forceinline__ Part warp_fold(const Part& p, float c)
{
    constexpr unsigned kAll = 0xffffffffu;
    Part r;
    r.m = unordered(__reduce_max_sync(kAll, ordered(p.m)));
    r.zx = unordered(__reduce_max_sync(kAll, ordered(p.zx)));
    float S, best = p.best;
    int idx = p.idx;
    if constexpr (kRace) {
        const bool has = p.m > -INFINITY;
        const float mc = __int_as_float(p.flag);
        const float M = unordered(__reduce_max_sync(kAll, ordered(has ? mc : -INFINITY)));
        const float f = has ? pow2_int(mc - M) : 0.f;
        S = p.S * f;
        race_scale_best(best, idx, f);
        r.flag = __float_as_int(M);
    } else {
        S = p.m > -INFINITY ? p.S * ex2((p.m - r.m) * c) : 0.f;
        r.flag = (int)__reduce_or_sync(kAll, (unsigned)p.flag);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) S += __shfl_xor_sync(kAll, S, off);
    r.S = S;
    const int bi = __reduce_max_sync(kAll, ordered(best));
    r.best = unordered(bi);
    r.idx = __reduce_min_sync(kAll, ordered(best) == bi ? idx : INT_MAX);
    return r;
}

// Fold of N partials in order (the same result in every thread that calls it).
template <bool kRace, int N>
__device__ __forceinline__ Part fold_partials(const Part* wp, float c)
{
    Part r;
    float m = -INFINITY, zx = -INFINITY, M = -INFINITY;
#pragma unroll
    for (int w = 0; w < N; ++w) {
        m = fmaxf(m, wp[w].m);
        zx = fmaxf(zx, wp[w].zx);
        if constexpr (kRace)
            if (wp[w].m > -INFINITY) M = fmaxf(M, __int_as_float(wp[w].flag));
    }
    float S = 0.f, best = -INFINITY;
    int idx = INT_MAX, flag = 0;
#pragma unroll
    for (int w = 0; w < N; ++w) {
        const bool has = wp[w].m > -INFINITY;
        float b = wp[w].best;
        int i = wp[w].idx;
        if constexpr (kRace) {
            const float f = has ? pow2_int(__int_as_float(wp[w].flag) - M) : 0.f;
            S += wp[w].S * f;
            race_scale_best(b, i, f);
        } else {
            S += has ? wp[w].S * ex2((wp[w].m - m) * c) : 0.f;
            flag |= wp[w].flag;
        }
        if (b > best || (b == best && i < idx)) { best = b; idx = i; }
    }
    r.m = m; r.S = S; r.zx = zx; r.best = best; r.idx = idx;
    r.flag = kRace ? __float_as_int(M) : flag;
    return r;
}

template <typename ET>
struct Producer {
    const Args& a;
    StreamShared& sh;
    unsigned char* ring;
    uint32_t it = 0;
    int lane, lo, hi;        // this CTA's slice [lo, hi) of every row

    __device__ Producer(const Args& a_, StreamShared& s_, unsigned char* r_, int lane_, int lo_, int hi_)
        : a(a_), sh(s_), ring(r_), lane(lane_), lo(lo_), hi(hi_) {}

    // The next stage, once its consumers released it; -1 (for the whole warp) when a wait of the
    // CTA has expired: from then on nothing more is issued, so no copy can land in a stage whose
    // previous copy is still in flight.
    __device__ __forceinline__ int acquire()
    {
        const int s = (int)(it % kStages);
        const uint32_t par = ((it / kStages) & 1u) ^ 1u;
        volatile int* flag = &sh.timed_out;
        bool ok = !*flag && mbar_wait_bounded(smem_addr(&sh.empty[s]), par, a.wait_ns, flag);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) *flag = 1;
        return ok ? s : -1;
    }

    // chunk c of the slice of logits row t (+ its mask words)
    __device__ __forceinline__ void row_chunk(int64_t t, int c)
    {
        using G = Geom<ET>;
        const int s = acquire();
        if (s < 0) return;
        unsigned char* st = ring + (size_t)s * kStageBytes;
        const int i0 = lo + c * G::kRowIds;
        const int n = min(G::kRowIds, hi - i0);
        const ET* src = reinterpret_cast<const ET*>(a.logits) + t * (int64_t)a.V + i0;
        const int32_t* msrc = a.bitmask ? a.bitmask + t * (int64_t)a.W + (i0 >> 5) : nullptr;
        const int nw = (n + 31) / 32;
        if (a.bulk) {
            if (lane == 0) {
                fence_proxy_async_smem();
                const uint32_t bar = smem_addr(&sh.full[s]);
                const uint32_t lb = (uint32_t)n * G::ES, mb = msrc ? (uint32_t)nw * 4u : 0u;
                mbar_arrive_expect_tx(bar, lb + mb);
                bulk_copy_g2s(smem_addr(st), src, lb, bar);
                if (mb) bulk_copy_g2s(smem_addr(st + G::kRowMaskOff), msrc, mb, bar);
            }
        } else {
            constexpr int VE = Elem<ET>::VE;
            const int npad = (n + VE - 1) / VE * VE;
            ET* d = reinterpret_cast<ET*>(st);
            ET pad;
            if constexpr (sizeof(ET) == 4) pad = -INFINITY; else pad = (ET)0xFF80u;
            for (int e = lane; e < npad; e += 32) d[e] = e < n ? src[e] : pad;
            if (msrc) {
                uint32_t* dm = reinterpret_cast<uint32_t*>(st + G::kRowMaskOff);
                for (int w = lane; w < nw; w += 32) dm[w] = (uint32_t)msrc[w];
            }
            mbar_arrive(smem_addr(&sh.full[s]));     // every lane arrives after its own stores
        }
        ++it;
    }

    // chunk c of the slice of draw row t (draft slot d): logits, noise, q (with_q), mask words
    __device__ __forceinline__ void draw_chunk(int64_t t, int64_t d, int c, bool with_q)
    {
        using G = Geom<ET>;
        const int s = acquire();
        if (s < 0) return;
        unsigned char* st = ring + (size_t)s * kStageBytes;
        const int ids = G::draw_ids(with_q);
        const int i0 = lo + c * ids;
        const int n = min(ids, hi - i0);
        const ET* src = reinterpret_cast<const ET*>(a.logits) + t * (int64_t)a.V + i0;
        const float* esrc = a.noise + t * (int64_t)a.V + i0;
        const float* qsrc = with_q ? a.q + d * (int64_t)a.V + i0 : nullptr;
        const int32_t* msrc = a.bitmask ? a.bitmask + t * (int64_t)a.W + (i0 >> 5) : nullptr;
        const int nw = (n + 31) / 32;
        if (a.bulk) {
            if (lane == 0) {
                fence_proxy_async_smem();
                const uint32_t bar = smem_addr(&sh.full[s]);
                const uint32_t lb = (uint32_t)n * G::ES, eb = (uint32_t)n * 4u;
                const uint32_t qb = qsrc ? eb : 0u, mb = msrc ? (uint32_t)nw * 4u : 0u;
                mbar_arrive_expect_tx(bar, lb + eb + qb + mb);
                bulk_copy_g2s(smem_addr(st), src, lb, bar);
                bulk_copy_g2s(smem_addr(st + G::noise_off(with_q)), esrc, eb, bar);
                if (qb) bulk_copy_g2s(smem_addr(st + G::q_off(with_q)), qsrc, qb, bar);
                if (mb) bulk_copy_g2s(smem_addr(st + G::dmask_off(with_q)), msrc, mb, bar);
            }
        } else {
            constexpr int VE = Elem<ET>::VE;
            const int npad = (n + VE - 1) / VE * VE;
            ET* dl = reinterpret_cast<ET*>(st);
            float* de = reinterpret_cast<float*>(st + G::noise_off(with_q));
            float* dq = reinterpret_cast<float*>(st + G::q_off(with_q));
            ET pad;
            if constexpr (sizeof(ET) == 4) pad = -INFINITY; else pad = (ET)0xFF80u;
            for (int e = lane; e < npad; e += 32) {
                const bool in = e < n;
                dl[e] = in ? src[e] : pad;
                de[e] = in ? esrc[e] : 1.f;
                if (with_q) dq[e] = (in && qsrc) ? qsrc[e] : 0.f;
            }
            if (msrc) {
                uint32_t* dm = reinterpret_cast<uint32_t*>(st + G::dmask_off(with_q));
                for (int w = lane; w < nw; w += 32) dm[w] = (uint32_t)msrc[w];
            }
            mbar_arrive(smem_addr(&sh.full[s]));
        }
        ++it;
    }
};

// kFilt: the variant with the top-k / top-p threshold search (compiled separately so that the
// search's code does not take registers from the variant every other batch runs)
template <typename ET, bool kFilt>
__global__ void __launch_bounds__(kStreamThreads, 2) specdec_verify_stream_kernel(const Args a)
{
    using G = Geom<ET>;
    constexpr int VE = Elem<ET>::VE;
    constexpr int GPW = 32 / VE;                                  // 16-byte groups per mask word
    extern __shared__ __align__(128) unsigned char ring[];
    __shared__ StreamShared sh;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int NCL = a.G;                                          // CTAs per cluster (launch)
    const int rank_hw = (int)cluster_ctarank();

    if (tid == 0) {
        const uint32_t full_count = a.bulk ? 1u : 32u;
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_addr(&sh.full[s]), full_count);
            mbar_init(smem_addr(&sh.empty[s]), kConsumerWarps);
        }
        mbar_init(smem_addr(&sh.dec), 1);
        mbar_init(smem_addr(&sh.pbar[0]), (uint32_t)NCL);
        mbar_init(smem_addr(&sh.pbar[1]), (uint32_t)NCL);
        fence_mbar_init();
        sh.timed_out = 0;
        sh.issued = 0;
    }
    // every CTA of the cluster has initialised its barriers before any partial is sent
    if (NCL > 1) cluster_sync_all(); else __syncthreads();
    grid_dependency_wait();                                        // the request order is ready
    // The request and the CTAs that verify it. Normally the cluster's NCL CTAs split request
    // order[i] (or i). A launch with split_n > 0 (clusters of 2) splits only the first split_n
    // requests of the order (the heaviest expected chains); every later cluster runs two requests,
    // one per CTA, independently.
    const int ci = (int)cluster_id_x();
    int b, NC, rank;
    if (a.split_n > 0 && ci >= a.split_n) {
        const int pos = a.split_n + 2 * (ci - a.split_n) + rank_hw;
        b = pos < a.B ? a.order[pos] : -1;
        NC = 1;
        rank = 0;
    } else {
        b = a.order ? a.order[ci] : ci;
        NC = NCL;
        rank = rank_hw;
    }
    if (b < 0) return;                    // the second CTA of the last pair when B - split_n is odd
    const int lo = rank * a.slice_units * kUnit;
    const int hi = NC > 1 ? min(a.V, lo + a.slice_units * kUnit) : a.V;
    const int nrow_chunks = (hi - lo + G::kRowIds - 1) / G::kRowIds;
    // at least one chunk of the next row is issued only after the pending decision was read,
    // so consumers can never post two decisions ahead of the producer
    const int spec = min(kSpec, nrow_chunks - 1);

    const ReqShape rs = request_shape(a, b);

    if (warp == 0) {
        // ------------------------------------------------------------------ producer
        const bool sp = rs.skip == 0 && request_is_sparse(a, rs.row0, lane);
        if (sp && lane == 0) {
            // sparse request: the consumers read every row's mask words first; start them into L2
            const int wlo = lo >> 5, whi = (hi + 31) >> 5;
            for (int j = 0; j <= rs.k; ++j)
                prefetch_l2(a.bitmask + (rs.row0 + j) * (int64_t)a.W + wlo, (uint32_t)(whi - wlo) * 4u);
        }
        if (rs.skip == 0 && !sp) {
            Producer<ET> pr(a, sh, ring, lane, lo, hi);
            // a filtered request streams its rows again for the threshold search, so nothing of
            // the next row may sit in the ring before a row's decisions are all taken
            const bool filt_on = kFilt && request_filter(a, b).on;
            const int spec_r = filt_on ? 0 : spec;
            // race rows (one pass over logits + noise, the consumers' test): the bonus row of an
            // unfiltered sampled request and every row of an unfiltered sampled model-free one
            const bool race_req = !request_greedy(a, b) && !filt_on;
            const bool qm = a.q != nullptr && (a.has_q == nullptr || a.has_q[b] != 0);
            const int nrace_chunks = (hi - lo + G::draw_ids(false) - 1) / G::draw_ids(false);
            auto race_row = [&](int j) { return race_req && (j == rs.k || !qm); };
            auto issue = [&](int j, int c) {
                if (race_row(j)) pr.draw_chunk(rs.row0 + j, (int64_t)rs.d0 + j, c, false);
                else pr.row_chunk(rs.row0 + j, c);
            };
            uint32_t dec_round = 0;
            int issued_next = 0;
            for (int j = 0; j <= rs.k; ++j) {
                const int64_t t = rs.row0 + j;
                const int nch = race_row(j) ? nrace_chunks : nrow_chunks;
                for (int c = issued_next; c < nch; ++c) issue(j, c);
                issued_next = 0;
                if (j < rs.k) {
                    // (a race row has at least as many chunks as a plain one: spec_r < either)
                    for (int c = 0; c < spec_r; ++c) issue(j + 1, c);
                    issued_next = spec_r;
                }
                // the consumers' next decision (kDecDone once any wait of the CTA has expired)
                auto next_code = [&]() -> int {
                    volatile int* flag = &sh.timed_out;
                    bool ok = !*flag && mbar_wait_bounded(smem_addr(&sh.dec), dec_round & 1u, a.wait_ns, flag);
                    ok = __all_sync(0xffffffffu, ok);
                    ++dec_round;
                    if (!ok) { *flag = 1; return kDecDone; }
                    return *reinterpret_cast<volatile int*>(&sh.dec_code);
                };
                int code = next_code();
                if constexpr (kFilt) {
                    while (code == kDecRescan) {             // one more pass of a threshold search
                        for (int c = 0; c < nrow_chunks; ++c) pr.row_chunk(t, c);
                        code = next_code();
                    }
                }
                if (code == kDecNextRow) continue;
                while (code == kDecDrawP || code == kDecDrawQ || code == kDecDrawOneHot) {
                    const bool wq = (code == kDecDrawQ);
                    const int nd = (hi - lo + G::draw_ids(wq) - 1) / G::draw_ids(wq);
                    for (int c = 0; c < nd; ++c) pr.draw_chunk(t, (int64_t)rs.d0 + j, c, wq);
                    code = next_code();
                }
                break;
            }
            if (lane == 0) sh.issued = pr.it;       // chunks issued, for the drain after an expired wait
        }
    } else {
        // ------------------------------------------------------------------ consumers
        const int ct = tid - 32, cw = warp - 1;
        const bool leader = (ct == 0);
        const bool writer = leader && rank == 0;
        SPECDEC_TRACE_BEGIN(b, writer);
        SPECDEC_STAMP(0);
        if (cw == 0) {
            // a1 ragged decode + a4 grammar-valid prefix (one consumer warp)
            const float T = a.temperature[b];
            const bool tvalid = (T == 0.f) || (T >= FLT_MIN && T <= FLT_MAX);
            const bool greedy = !(T > 0.f) || !tvalid;
            const bool qmode = a.q != nullptr && (a.has_q == nullptr || a.has_q[b] != 0);
            int g = rs.skip == 1 ? 0 : rs.k;
            uint32_t st = rs.skip == 1 ? SPECDEC_ST_BAD_OFFSETS : (rs.skip == 2 ? SPECDEC_ST_K_TOO_LARGE : 0u);
            bool sparse = false;
            if (rs.skip == 0) {
                sparse = request_is_sparse(a, rs.row0, lane);
                bool ok = true, allowed = true;
                if (lane < rs.k) {
                    const int32_t x = a.draft_ids ? a.draft_ids[rs.d0 + lane] : -1;
                    ok = x >= 0 && x < a.V;
                    allowed = ok;
                    if (ok && a.bitmask)
                        allowed = ((uint32_t)a.bitmask[(rs.row0 + lane) * (int64_t)a.W + (x >> 5)] >> (x & 31)) & 1u;
                    sh.xs[lane] = x;
                    sh.us[lane] = a.uniforms[rs.row0 + lane];
                    sh.qxs[lane] = (qmode && ok && !greedy) ? a.q[(int64_t)(rs.d0 + lane) * a.V + x] : 0.f;
                }
                const unsigned inval = __ballot_sync(0xffffffffu, lane < rs.k && !allowed);
                const unsigned badid = __ballot_sync(0xffffffffu, lane < rs.k && !ok);
                if (inval) g = __ffs(inval) - 1;
                if (badid) st |= SPECDEC_ST_BAD_DRAFT_ID;
                if (!tvalid) st |= SPECDEC_ST_BAD_TEMPERATURE;
            }
            if (lane == 0) {
                const Filter f = request_filter(a, b);
                if (f.bad_p && rs.skip == 0) st |= SPECDEC_ST_BAD_TOP_P;
                sh.fk = f.on ? f.k : 0;
                sh.fp = f.on ? f.p : 1.f;
                sh.g = g; sh.greedy = greedy; sh.qmode = qmode; sh.st = st; sh.sparse = sparse;
                sh.c = greedy ? 0.f : (float)(1.4426950408889634 / (double)T);   // log2(e) / T, once
            }
        }
        consumer_sync();
        SPECDEC_STAMP(sh.sparse ? 15 : 1);
        const int k = rs.k, g = sh.g;
        const bool greedy = sh.greedy != 0, qmode = sh.qmode != 0, sparse = sh.sparse != 0;
        const float c = sh.c;
        const float T = a.temperature[b];
        const int fk = sh.fk;
        const float fp = sh.fp;
        const bool filt = kFilt && (fk > 0 || fp < 1.f);          // a top-k / top-p request (sampled)
        uint32_t st = sh.st;
        const bool has_mask = a.bitmask != nullptr;
        uint32_t* list = reinterpret_cast<uint32_t*>(ring);
        const int wlo = lo >> 5, whi = (hi + 31) >> 5;             // this slice's mask words

        if (writer && rs.skip != 1) {
            if (a.diag_alpha) for (int j = 0; j < k; ++j) a.diag_alpha[rs.d0 + j] = NAN;
            if (a.diag_row)
                for (int j = 0; j <= k; ++j) { a.diag_row[2 * (rs.row0 + j)] = NAN; a.diag_row[2 * (rs.row0 + j) + 1] = NAN; }
        }

        uint32_t it = 0, xround = 0;
        int par = 0;
        // (an expired wait marks the CTA before the stage is released: the producer, which acquires
        // that release, then issues nothing more; the stage's contents are then not used for any
        // output that counts, the request being reported as timed out)
        auto wait_full = [&]() -> int {
            const int s = (int)(it % kStages);
            volatile int* flag = &sh.timed_out;
            if (!mbar_wait_bounded(smem_addr(&sh.full[s]), (it / kStages) & 1u, a.wait_ns, flag)) *flag = 1;
            return s;
        };
        auto release = [&](int s) {
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&sh.empty[s]));
            ++it;
        };
        // CTA-wide reduction of the consumers' partials, then (NC > 1) a point-to-point exchange
        // with the other CTAs of the request: consumer thread i stores this CTA's partial into
        // CTA i's slot and arrives on CTA i's barrier; every CTA folds the NC partials in rank
        // order, so all of them hold bit-identical results.
        // (race partials -- see race_raise -- combine by their own rule: `race` is a
        // std::integral_constant<bool, ...>)
        auto reduce_cta = [&](Part p, auto race) -> Part {
            constexpr bool kR = decltype(race)::value;
            const Part w = warp_fold<kR>(p, c);
            if (lane == 0) sh.wpart[par][cw] = w;
            consumer_sync();
            const Part r = fold_partials<kR, kConsumerWarps>(sh.wpart[par], c);
            par ^= 1;
            return r;
        };
        auto reduce_any = [&](Part p, auto race) -> Part {
            constexpr bool kR = decltype(race)::value;
            const Part r = reduce_cta(p, race);
            if (NC == 1) return r;
            const int slot = (int)(xround & 1u);
            if (ct < NC) {
                const uint32_t base = map_to_rank(smem_addr(&sh.parts[slot][rank]), (uint32_t)ct);
                st_cluster_u32(base + 0, __float_as_uint(r.m));
                st_cluster_u32(base + 4, __float_as_uint(r.S));
                st_cluster_u32(base + 8, __float_as_uint(r.zx));
                st_cluster_u32(base + 12, __float_as_uint(r.best));
                st_cluster_u32(base + 16, (uint32_t)r.idx);
                st_cluster_u32(base + 20, (uint32_t)r.flag);
                mbar_arrive_remote(map_to_rank(smem_addr(&sh.pbar[slot]), (uint32_t)ct));
            }
            if (!mbar_wait_cluster_bounded(smem_addr(&sh.pbar[slot]), (xround >> 1) & 1u, a.wait_ns, &sh.timed_out))
                *reinterpret_cast<volatile int*>(&sh.timed_out) = 1;
            ++xround;
            // one thread folds the partials in rank order and every consumer reads its result after a
            // barrier: all of them take the same decision even when a wait expired while partials
            // were still landing (threads reading them one by one could then disagree, and a
            // disagreement would split them across the consumers' named barriers)
            if (ct == 0) {
                Part q = part_identity();
                for (int i = 0; i < NC; ++i) combine_any<kR>(q, sh.parts[slot][i], c);
                sh.xres[slot] = q;
            }
            consumer_sync();
            return sh.xres[slot];
        };
        auto reduce = [&](Part p) -> Part { return reduce_any(p, std::false_type{}); };
        auto post = [&](int code) {
            if (leader && !sparse) {
                *reinterpret_cast<volatile int*>(&sh.dec_code) = code;
                mbar_arrive(smem_addr(&sh.dec));
            }
        };
        // Sparse path: list the 16-byte groups of mask words [w0, w1) of row t that hold an
        // allowed id, in id order (block-wide exclusive scan). Returns the count.
        auto build_list = [&](int64_t t, int w0, int w1) -> int {
            constexpr int kPer = kSegWords / kConsumers;                // 20 words per thread
            static_assert(kPer % 4 == 0, "words are loaded 4 at a time");
            const uint4* mrow = reinterpret_cast<const uint4*>(a.bitmask + t * (int64_t)a.W);
            // each thread owns a contiguous run of words so that list order is id order
            const int my0 = w0 + ct * kPer;
            uint32_t words[kPer];
            SPECDEC_STAMP(10);
            // (loaded twice: for the count, and again after the scan for the list, from L1, so
            // that the words are not held in registers across the scan's barriers)
            auto load_words = [&] {
#pragma unroll
                for (int q4 = 0; q4 < kPer / 4; ++q4) {
                    const int w = my0 + 4 * q4;           // W and the slice bounds are multiples of 4 words
                    const uint4 u = (w < w1) ? __ldg(mrow + (w >> 2)) : make_uint4(0u, 0u, 0u, 0u);
                    words[4 * q4] = u.x; words[4 * q4 + 1] = u.y; words[4 * q4 + 2] = u.z; words[4 * q4 + 3] = u.w;
                }
            };
            load_words();
            // one bit per 16-byte group (its lowest id's position) when any id of the group is allowed;
            // bits at or above V in the row's last word are dropped first
            const int vtail = a.V & 31;
            auto presence = [&](uint32_t w, int wi) -> uint32_t {
                if (vtail && wi == a.W - 1) w &= (1u << vtail) - 1u;
                uint32_t t2 = w | (w >> 1);
                t2 |= t2 >> 2;
                if constexpr (VE == 8) { t2 |= t2 >> 4; return t2 & 0x01010101u; }
                else return t2 & 0x11111111u;
            };
            int cnt = 0;
#pragma unroll
            for (int q = 0; q < kPer; ++q) cnt += __popc(presence(words[q], my0 + q));
            SPECDEC_STAMP(11);
            // exclusive scan of cnt over the consumers
            int incl = cnt;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += y;
            }
            consumer_sync();                              // the list / scan slots are free
            if (lane == 31) sh.scan[cw] = incl;
            consumer_sync();
            int base = incl - cnt, total = 0;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) {
                const int v = sh.scan[w];
                if (w < cw) base += v;
                total += v;
            }
            SPECDEC_STAMP(12);
            if (total > kListCap) {                       // caller re-scans in smaller pieces
                consumer_sync();
                return -1;
            }
            // fixed trip count (no loop over set bits): allowed ids come in runs, and a loop over
            // set bits would serialise each warp on its densest word (slots from per-word popcount
            // prefixes instead of the running count measured slower still)
            load_words();
#pragma unroll
            for (int q = 0; q < kPer; ++q) {
                const uint32_t pres = presence(words[q], my0 + q);
#pragma unroll
                for (int h = 0; h < GPW; ++h) {
                    if ((pres >> (h * VE)) & 1u)
                        list[base++] = ((uint32_t)((my0 + q) * GPW + h) << 8) | ((words[q] >> (h * VE)) & ((1u << VE) - 1u));
                }
            }
            SPECDEC_STAMP(13);
            consumer_sync();
            return total;
        };

        // Sparse statistics pass over list[0, n) of row t: the listed groups' logits are gathered
        // with cp.async in batches of kGatherCap (all in flight at once), then folded from shared memory.
        auto sparse_stats = [&](int64_t t, int x, int n, Part& p, float& mc) {
            const unsigned char* lrow = reinterpret_cast<const unsigned char*>(a.logits) + t * (int64_t)a.V * G::ES;
            const uint32_t dbase = smem_addr(ring + kDataOff);
            const uint4* data = reinterpret_cast<const uint4*>(ring + kDataOff);
            const uint32_t ni = Raw<ET>::kNegInf;
            for (int b0 = 0; b0 < n; b0 += kGatherCap) {
                const int nb = min(kGatherCap, n - b0);
                for (int e = ct; e < nb; e += kConsumers)
                    cp_async16(dbase + (uint32_t)e * 16u, lrow + (size_t)(list[b0 + e] >> 8) * 16u);
                cp_async_wait_all();
                consumer_sync();
                SPECDEC_STAMP(14);
                constexpr int U = 4;
                for (int e0 = ct; e0 < nb; e0 += kConsumers * U) {
                    float z[U * VE];
                    int ids[U * VE];
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        const int e = e0 + u * kConsumers;
                        const bool in = e < nb;
                        const uint32_t ent = in ? list[b0 + e] : 0u;
                        const uint4 raw = in ? data[e] : make_uint4(ni, ni, ni, ni);
                        const uint32_t bits = ent & 0xffu;
                        const int grp = (int)(ent >> 8);
                        unpack_raw<ET>(raw, z + u * VE);
#pragma unroll
                        for (int q = 0; q < VE; ++q) {
                            z[u * VE + q] = ((bits >> q) & 1u) ? z[u * VE + q] : -INFINITY;
                            ids[u * VE + q] = in ? grp * VE + q : -1;   // an unused slot matches no draft
                        }
                    }
                    if (greedy) {
                        argmax_batch<U * VE>(p, z, ids);
                    } else {
                        if (x >= 0) {
#pragma unroll
                            for (int q = 0; q < U * VE; ++q)
                                if (ids[q] == x) p.zx = z[q];
                        }
                        softmax_batch<U * VE>(p, mc, z, c);
                    }
                }
                // the data region is free again before the next batch's copies (after the last
                // batch, the reduction's or the next list's barrier comes before any new copy)
                if (b0 + kGatherCap < n) consumer_sync();
            }
        };
        // Sparse draw pass over list[0, n) of row t: logits, noise and (q-mode) q of the listed
        // groups, gathered with cp.async in batches sized to the data region.
        auto sparse_draw = [&](int64_t t, int64_t d, int x, int n, int code, Part& dp, float MC, float invS, uint32_t kt) {
            const bool wq = (code == kDecDrawQ);
            const int per = 16 + 4 * VE + (wq ? 4 * VE : 0);
            const int cap = kDataBytes / per;
            unsigned char* dl = ring + kDataOff;
            unsigned char* dn = dl + cap * 16;
            unsigned char* dqp = dn + cap * 4 * VE;
            const unsigned char* lrow = reinterpret_cast<const unsigned char*>(a.logits) + t * (int64_t)a.V * G::ES;
            const unsigned char* erow = reinterpret_cast<const unsigned char*>(a.noise + t * (int64_t)a.V);
            const unsigned char* qrow = wq ? reinterpret_cast<const unsigned char*>(a.q + d * (int64_t)a.V) : nullptr;
            for (int b0 = 0; b0 < n; b0 += cap) {
                const int nb = min(cap, n - b0);
                for (int e = ct; e < nb; e += kConsumers) {
                    const size_t grp = list[b0 + e] >> 8;
                    cp_async16(smem_addr(dl + e * 16), lrow + grp * 16u);
#pragma unroll
                    for (int h = 0; h < VE / 4; ++h) {
                        cp_async16(smem_addr(dn + e * 4 * VE + 16 * h), erow + grp * (4u * VE) + 16u * h);
                        if (wq) cp_async16(smem_addr(dqp + e * 4 * VE + 16 * h), qrow + grp * (4u * VE) + 16u * h);
                    }
                }
                cp_async_wait_all();
                consumer_sync();
                constexpr int U = (VE == 8) ? 1 : 2;
                for (int e0 = ct; e0 < nb; e0 += kConsumers * U) {
                    float z[U * VE], ev[U * VE], qv[U * VE];
                    int ids[U * VE];
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        const int e = e0 + u * kConsumers;
                        const bool in = e < nb;
                        const uint32_t ent = in ? list[b0 + e] : 0u;
                        const uint32_t bits = ent & 0xffu;
                        const int grp = (int)(ent >> 8);
                        const uint32_t ni = Raw<ET>::kNegInf;
                        unpack_raw<ET>(in ? reinterpret_cast<const uint4*>(dl)[e] : make_uint4(ni, ni, ni, ni), z + u * VE);
#pragma unroll
                        for (int h = 0; h < VE / 4; ++h) {
                            const float4 f = in ? reinterpret_cast<const float4*>(dn + e * 4 * VE)[h] : make_float4(1.f, 1.f, 1.f, 1.f);
                            const float4 g4 = (in && wq) ? reinterpret_cast<const float4*>(dqp + e * 4 * VE)[h] : make_float4(0.f, 0.f, 0.f, 0.f);
                            ev[u * VE + 4 * h] = f.x; ev[u * VE + 4 * h + 1] = f.y; ev[u * VE + 4 * h + 2] = f.z; ev[u * VE + 4 * h + 3] = f.w;
                            qv[u * VE + 4 * h] = g4.x; qv[u * VE + 4 * h + 1] = g4.y; qv[u * VE + 4 * h + 2] = g4.z; qv[u * VE + 4 * h + 3] = g4.w;
                        }
#pragma unroll
                        for (int q = 0; q < VE; ++q) {
                            z[u * VE + q] = ((bits >> q) & 1u) ? z[u * VE + q] : -INFINITY;
                            if (kt != 0u && logit_key(z[u * VE + q]) < kt) z[u * VE + q] = -INFINITY;
                            ids[u * VE + q] = in ? grp * VE + q : -1;
                        }
                    }
                    draw_batch<U * VE>(dp, z, ev, qv, ids, code, x, c, MC, invS);
                }
                if (b0 + cap < n) consumer_sync();       // (as in sparse_stats)
            }
        };
        // Sparse race pass over list[0, n) of row t (race rows, see race_raise): logits and noise of
        // the listed groups, gathered with cp.async in batches sized to the data region, folded into
        // the softmax statistics and the race that excludes id x (x < 0: none).
        auto sparse_race = [&](int64_t t, int x, int n, Part& p, float& mc) {
            constexpr int per = 16 + 4 * VE;
            constexpr int cap = kDataBytes / per;
            unsigned char* dl = ring + kDataOff;
            unsigned char* dn = dl + cap * 16;
            const unsigned char* lrow = reinterpret_cast<const unsigned char*>(a.logits) + t * (int64_t)a.V * G::ES;
            const unsigned char* erow = reinterpret_cast<const unsigned char*>(a.noise + t * (int64_t)a.V);
            for (int b0 = 0; b0 < n; b0 += cap) {
                const int nb = min(cap, n - b0);
                for (int e = ct; e < nb; e += kConsumers) {
                    const size_t grp = list[b0 + e] >> 8;
                    cp_async16(smem_addr(dl + e * 16), lrow + grp * 16u);
#pragma unroll
                    for (int h = 0; h < VE / 4; ++h)
                        cp_async16(smem_addr(dn + e * 4 * VE + 16 * h), erow + grp * (4u * VE) + 16u * h);
                }
                cp_async_wait_all();
                consumer_sync();
                constexpr int U = (VE == 8) ? 1 : 2;
                for (int e0 = ct; e0 < nb; e0 += kConsumers * U) {
                    float z[U * VE], ev[U * VE];
                    int ids[U * VE];
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        const int e = e0 + u * kConsumers;
                        const bool in = e < nb;
                        const uint32_t ent = in ? list[b0 + e] : 0u;
                        const uint32_t bits = ent & 0xffu;
                        const int grp = (int)(ent >> 8);
                        const uint32_t ni = Raw<ET>::kNegInf;
                        unpack_raw<ET>(in ? reinterpret_cast<const uint4*>(dl)[e] : make_uint4(ni, ni, ni, ni), z + u * VE);
#pragma unroll
                        for (int h = 0; h < VE / 4; ++h) {
                            const float4 f = in ? reinterpret_cast<const float4*>(dn + e * 4 * VE)[h] : make_float4(1.f, 1.f, 1.f, 1.f);
                            ev[u * VE + 4 * h] = f.x; ev[u * VE + 4 * h + 1] = f.y; ev[u * VE + 4 * h + 2] = f.z; ev[u * VE + 4 * h + 3] = f.w;
                        }
#pragma unroll
                        for (int q = 0; q < VE; ++q) {
                            z[u * VE + q] = ((bits >> q) & 1u) ? z[u * VE + q] : -INFINITY;
                            ids[u * VE + q] = in ? grp * VE + q : -1;
                        }
                    }
                    if (x >= 0) {
#pragma unroll
                        for (int q = 0; q < U * VE; ++q)
                            if (ids[q] == x) p.zx = z[q];
                    }
                    race_batch<U * VE>(p, mc, z, ev, ids, x, c);
                }
                if (b0 + cap < n) consumer_sync();       // (as in sparse_stats)
            }
        };

        int acc_len = 0, emitted = -1;
        int slice_oct = 0;              // top-k: octaves of the top slice below its base level (-1: off)
        if (rs.skip == 0) {
            acc_len = k;
            int listed_row = -1, listed_n = 0;            // row whose whole slice list is in `list`

            // ---- top-k / top-p (sampled requests that ask for them): the threshold key kt of row t
            // (kept ids: key >= kt) and the kept mass relative to MC, by an exact radix select:
            // a first pass bins the allowed logits by their mass exp2(z * c - MC), then passes over
            // the elements of the chosen bin resolve their order-preserving keys 8 bits at a time
            // (bf16 keys have 16 significant bits). Counts for top-k; masses for top-p as exact
            // integer sums (the result does not depend on the order of the additions). Dense rows
            // are streamed again through the ring; sparse rows reuse their gathered groups when the
            // row's list fit one gather batch, else gather again.
            // The visitors call f(z, valid, id0) for every vector of element slots of the row (z: VE
            // logits of ids id0 .. id0 + VE - 1; bit e of valid: slot e holds an allowed id with a
            // finite logit).
            auto gather_and_visit = [&](int64_t t, int n, auto&& f) {
                const unsigned char* lrow = reinterpret_cast<const unsigned char*>(a.logits) + t * (int64_t)a.V * G::ES;
                const uint32_t dbase = smem_addr(ring + kDataOff);
                const uint4* data = reinterpret_cast<const uint4*>(ring + kDataOff);
                for (int b0 = 0; b0 < n; b0 += kGatherCap) {
                    const int nb = min(kGatherCap, n - b0);
                    for (int e = ct; e < nb; e += kConsumers)
                        cp_async16(dbase + (uint32_t)e * 16u, lrow + (size_t)(list[b0 + e] >> 8) * 16u);
                    cp_async_wait_all();
                    consumer_sync();
                    for (int e0 = ct - lane; e0 < nb; e0 += kConsumers) {      // warp-uniform trip count
                        const int e = e0 + lane;
                        const bool in = e < nb;
                        float z[VE];
                        unpack_raw<ET>(in ? data[e] : make_uint4(0u, 0u, 0u, 0u), z);
                        const uint32_t bits = in ? (list[b0 + e] & 0xffu) : 0u;
                        f(z, bits & finite_bits<VE>(z), in ? (int)(list[b0 + e] >> 8) * VE : 0);
                    }
                    consumer_sync();
                }
            };
            auto visit_row = [&](int64_t t, int j, auto&& f) {
                if (!sparse) {
                    post(kDecRescan);
                    constexpr int NB = 4;                       // vectors loaded together (latency)
                    for (int ch = 0; ch < nrow_chunks; ++ch) {
                        const int s = wait_full();
                        const unsigned char* stg = ring + (size_t)s * kStageBytes;
                        const uint32_t* sm = reinterpret_cast<const uint32_t*>(stg + G::kRowMaskOff);
                        const int i0 = lo + ch * G::kRowIds;
                        const int n = min(G::kRowIds, hi - i0);
                        const int nvec = (n + VE - 1) / VE;
                        for (int vb = ct - lane; vb < nvec; vb += kConsumers * NB) {   // warp-uniform trip count
                            uint4 raw[NB];
                            uint32_t bits[NB];
#pragma unroll
                            for (int u = 0; u < NB; ++u) {
                                const int v = vb + lane + u * kConsumers;
                                const bool in = v < nvec;
                                const uint32_t ni = Raw<ET>::kNegInf;
                                raw[u] = in ? reinterpret_cast<const uint4*>(stg)[v] : make_uint4(ni, ni, ni, ni);
                                bits[u] = in ? vec_bits<VE>(sm, has_mask, v) : 0u;
                            }
#pragma unroll
                            for (int u = 0; u < NB; ++u) {
                                float z[VE];
                                unpack_raw<ET>(raw[u], z);
                                f(z, bits[u] & finite_bits<VE>(z), i0 + (vb + lane + u * kConsumers) * VE);
                            }
                        }
                        release(s);
                    }
                } else if (listed_row == j && listed_n <= kGatherCap) {
                    // the row's groups are still in the data region, in list order
                    const uint4* data = reinterpret_cast<const uint4*>(ring + kDataOff);
                    for (int e0 = ct - lane; e0 < listed_n; e0 += kConsumers) {
                        const int e = e0 + lane;
                        const bool in = e < listed_n;
                        float z[VE];
                        unpack_raw<ET>(in ? data[e] : make_uint4(0u, 0u, 0u, 0u), z);
                        const uint32_t bits = in ? (list[e] & 0xffu) : 0u;
                        f(z, bits & finite_bits<VE>(z), in ? (int)(list[e] >> 8) * VE : 0);
                    }
                } else if (listed_row == j) {
                    gather_and_visit(t, listed_n, f);
                } else {
                    for (int w0 = wlo; w0 < whi; w0 += kSegWords) {
                        const int w1 = min(whi, w0 + kSegWords);
                        const int n = build_list(t, w0, w1);
                        if (n >= 0) {
                            gather_and_visit(t, n, f);
                        } else {
                            for (int s0 = w0; s0 < w1; s0 += G::kSafeWords)
                                gather_and_visit(t, build_list(t, s0, min(w1, s0 + G::kSafeWords)), f);
                        }
                    }
                }
            };
            // Sum of v over the consumer threads, in a fixed order (shuffles, then the warps in
            // order): every consumer thread gets the same value.
            auto fold_u64 = [&](unsigned long long v, unsigned long long* slots) -> unsigned long long {
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
                if (lane == 0) slots[cw] = v;
                consumer_sync();
                unsigned long long r = 0ull;
#pragma unroll
                for (int w = 0; w < kConsumerWarps; ++w) r += slots[w];
                return r;
            };
            // One pass into the 256 bins. First pass (bin0 < 0): every element at or above floor_key,
            // by mass_bin, counting elements (want & 1: top-k) or summing masses (want & 2: top-p);
            // the tail (bin 0), where most elements of a peaked row fall, is counted and summed in
            // registers and folded afterwards, so the shared-memory additions spread over the other
            // bins. Later passes: the elements of mass bin bin0 whose key lies in [klo, khi] and
            // matches pval on the bits of pmask, counted and summed by the key's bits [shift, shift
            // + 8) (width). Integer sums only: the result does not depend on the order of the
            // additions. The elements come from the row (ncand < 0) or the first ncand candidates.
            auto hist_pass = [&](int64_t t, int j, int bin0, uint32_t pmask, uint32_t pval, int shift, uint32_t width,
                                 uint32_t floor_key, float MC, uint32_t klo, uint32_t khi, int ncand, int want) {
                for (int i = ct; i < 256; i += kConsumers) { sh.fcnt[i] = 0u; sh.flo[i] = 0u; sh.fhi[i] = 0u; }
                consumer_sync();
                SPECDEC_STAMP(13);
                const bool wcnt = bin0 >= 0 || (want & 1), wmass = bin0 >= 0 || (want & 2);
                uint32_t tcnt = 0u;
                unsigned long long tm = 0ull;
                const uint32_t kfloor = max(floor_key, klo);
                // (a first pass with no floor tests no key: every allowed element counts)
                const bool plain = bin0 < 0 && kfloor == 0u;
                auto bin = [&](const auto& z, uint32_t valid, int) {
                    constexpr int N = (int)(sizeof(z) / sizeof(z[0]));
                    uint32_t in = valid;
                    if (!plain) {
#pragma unroll
                        for (int i = 0; i < N; ++i) {
                            const uint32_t kk = logit_key(z[i]);
                            if (!(kk >= kfloor && kk <= khi && (kk & pmask) == pval)) in &= ~(1u << i);
                        }
                    }
                    if (in == 0u) return;
                    float e[N];
                    uint32_t mb[N];
#pragma unroll
                    for (int i = 0; i < N; ++i) {
                        e[i] = ex2(fmaf(z[i], c, -MC));
                        mb[i] = mass_bin(e[i]);
                    }
#pragma unroll
                    for (int i = 0; i < N; ++i) {
                        if (!((in >> i) & 1u)) continue;
                        uint32_t dg;
                        if (bin0 < 0) {
                            if (mb[i] == 0u) { tcnt += 1u; tm += mass_units(e[i], true); continue; }
                            dg = mb[i];
                        } else {
                            if ((int)mb[i] != bin0) continue;
                            dg = (logit_key(z[i]) >> shift) & width;
                        }
                        if (wcnt) atomicAdd(&sh.fcnt[dg], 1u);
                        if (wmass) {
                            const uint32_t m = mass_units(e[i], bin0 == 0);
                            atomicAdd(&sh.flo[dg], m & 0xfffu);
                            atomicAdd(&sh.fhi[dg], m >> 12);
                        }
                    }
                };
                if (ncand < 0) visit_row(t, j, bin);
                else
                    for (int i = ct; i < ncand; i += kConsumers) {
                        const float z1[1] = {key_logit(sh.fcand[i])};
                        bin(z1, 1u, 0);
                    }
                SPECDEC_STAMP(14);
                if (bin0 < 0) {
                    const unsigned long long c0 = fold_u64(tcnt, sh.fw_m);
                    const unsigned long long m0 = fold_u64(tm, sh.fw_m2);
                    if (ct == 0) { sh.fcnt[0] = (uint32_t)c0; sh.ftail_m = m0; }
                }
                consumer_sync();
            };
            // digit choice by consumer warp 0: lane l holds digits 255 - 8l .. 248 - 8l (highest
            // first); per-lane sums, an exclusive scan over lanes, then each lane walks its digits.
            // Bin masses are fixed-point integers in units of 2^-40 (fx40 of the exact unit sums:
            // each bin's own unit in the first pass (bin0 < 0), the unit of mass bin bin0 in the
            // later ones), so the choice is integer arithmetic throughout.
            // mode 0 (top-k): the digit where the count from the top reaches `need`;
            // mode 1 (top-p): the lowest non-empty digit whose mass above (plus `above`) is below P
            // (P = p_frac of this pass's total when p_frac >= 0).
            // Everything the caller needs is copied to the fsel_ fields before the closing barrier:
            // the next pass clears the bins as soon as a thread reaches it.
            auto select_digit = [&](int mode, unsigned long long need, unsigned long long P, unsigned long long above,
                                    int bin0, float p_frac) {
                if (cw == 0) {
                    const int pexp = bin0 < 0 ? 0 : bin_exp((uint32_t)bin0);
                    // digit dg's count and mass (read again from the bins where needed: fewer live registers)
                    auto dmass = [&](int dg) -> unsigned long long {
                        const unsigned long long u = ((unsigned long long)sh.fhi[dg] << 12) + sh.flo[dg];
                        if (bin0 >= 0) return fx40(u, pexp);
                        return dg == 0 ? fx40(sh.ftail_m, -54) : (dg >= 8 ? fx40(u, bin_exp((uint32_t)dg)) : 0ull);
                    };
                    unsigned long long lc = 0ull, lm = 0ull;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int dg = 255 - 8 * lane - i;
                        lc += sh.fcnt[dg];
                        lm += dmass(dg);
                    }
                    unsigned long long ic = lc, im = lm;
#pragma unroll
                    for (int off = 1; off < 32; off <<= 1) {
                        const unsigned long long yc = __shfl_up_sync(0xffffffffu, ic, off);
                        const unsigned long long ym = __shfl_up_sync(0xffffffffu, im, off);
                        if (lane >= off) { ic += yc; im += ym; }
                    }
                    const unsigned long long tot_m = __shfl_sync(0xffffffffu, im, 31);
                    if (p_frac >= 0.f) P = (unsigned long long)((double)p_frac * (double)tot_m);
                    unsigned long long c0 = __shfl_up_sync(0xffffffffu, ic, 1);
                    unsigned long long m0 = __shfl_up_sync(0xffffffffu, im, 1);
                    if (lane == 0) { c0 = 0ull; m0 = 0ull; }
                    unsigned long long fc = 0ull, fn = 0ull, fm = 0ull, fa = 0ull;
                    int found = -1;
#pragma unroll 1
                    for (int i = 0; i < 8; ++i) {
                        const int dg = 255 - 8 * lane - i;
                        const unsigned long long bc = sh.fcnt[dg], bm = dmass(dg);
                        // elements in the digit: counted, or (first top-p pass, bins from 8 up) at
                        // most the mass units over 2^23, the smallest significand
                        const unsigned long long n = (bin0 < 0 && mode == 1 && dg >= 8)
                            ? (((unsigned long long)sh.fhi[dg] << 12) + sh.flo[dg]) >> 23 : bc;
                        // (a tail too light for 2^-40 is never the choice: its mass above is the total)
                        const bool nonempty = bc != 0ull || bm != 0ull;
                        if (mode == 0) {
                            if (found < 0 && c0 + bc >= need) { found = dg; fc = c0; fm = m0; fa = bm; fn = n; }
                        } else if (nonempty && above + m0 < P) {
                            found = dg; fc = c0; fm = m0; fa = bm; fn = n;
                        }
                        c0 += bc;
                        m0 += bm;
                    }
                    const unsigned who = __ballot_sync(0xffffffffu, found >= 0);
                    // top-k: the first lane that reaches `need`; top-p: the last lane with a candidate
                    const int src = who == 0u ? -1 : (mode == 0 ? __ffs(who) - 1 : 31 - __clz(who));
                    if (lane == 0) { sh.fsel_digit = 0xffffffffu; sh.ftot_mass = tot_m; sh.fsel_P = P; }
                    __syncwarp();
                    if (lane == src) {
                        sh.fsel_digit = (uint32_t)found; sh.fsel_cnt = fc; sh.fsel_mass = fm; sh.fsel_at = fa;
                        sh.fsel_n = fn;
                    }
                }
                consumer_sync();
            };
            // One more pass for mass bin bc: the smallest and largest key and the mass of its
            // elements (at or above floor_key), the mass above it (units of 2^-40; only when
            // sum_above), and, over the row (ncand < 0), the keys of its elements (all = false) or of
            // every element from bin bc up (all = true) appended to the candidates. Returns the
            // number of such elements (above kCandCap: only the first kCandCap kept). Over the first
            // ncand candidates (ncand >= 0) nothing is appended and ncand comes back.
            // The exponent argument z*c - MC of an element decides its bin, so a compare of that
            // argument against the bin's bounds (widened by 1e-3, far more than the error of ex2)
            // skips, before any other work, the elements that cannot fall in the bin (below it, and
            // above it when neither their mass nor their keys are wanted).
            auto collect_pass = [&](int64_t t, int j, uint32_t bc, bool all, bool sum_above, uint32_t floor_key,
                                    float MC, int ncand) -> int {
                if (ct == 0 && ncand < 0) sh.fncand = 0u;
                consumer_sync();
                SPECDEC_STAMP(10);
                uint32_t kmn = 0xffffffffu, kmx = 0u;
                unsigned long long mbin = 0ull, mab = 0ull;
                const float bexp = (float)((int)(bc >> 3) - 31);           // log2 of the bin's octave
                const float alo = bc == 0u ? -INFINITY : log2f((float)(8u + (bc & 7u)) * 0.125f) + bexp - 1e-3f;
                const float ahi = (sum_above || all) ? INFINITY
                                : (bc == 0u ? -30.f : log2f((float)(9u + (bc & 7u)) * 0.125f) + bexp) + 1e-3f;
                auto take = [&](const auto& z, uint32_t valid, int) {
                    constexpr int N = (int)(sizeof(z) / sizeof(z[0]));
                    float arg[N];
                    uint32_t in = 0u;
#pragma unroll
                    for (int i = 0; i < N; ++i) {
                        arg[i] = fmaf(z[i], c, -MC);
                        in |= (((valid >> i) & 1u) && arg[i] >= alo && arg[i] <= ahi ? 1u : 0u) << i;
                    }
                    if (in == 0u) return;
                    uint32_t key[N];
                    float e[N];
                    uint32_t mb[N];
#pragma unroll
                    for (int i = 0; i < N; ++i) {
                        key[i] = logit_key(z[i]);
                        e[i] = ex2(arg[i]);
                        mb[i] = mass_bin(e[i]);
                    }
#pragma unroll
                    for (int i = 0; i < N; ++i) {
                        if (!((in >> i) & 1u) || key[i] < floor_key || mb[i] < bc) continue;
                        if (mb[i] == bc) {
                            kmn = min(kmn, key[i]);
                            kmx = max(kmx, key[i]);
                            mbin += mass_units(e[i], bc == 0u);
                        } else if (sum_above) {
                            mab += __float2ull_rn(e[i] * 0x1p40f);
                        }
                        if (ncand < 0 && (all || mb[i] == bc)) {
                            const uint32_t pos = atomicAdd(&sh.fncand, 1u);
                            if (pos < (uint32_t)kCandCap) sh.fcand[pos] = key[i];
                        }
                    }
                };
                if (ncand < 0) visit_row(t, j, take);
                else
                    for (int i = ct; i < ncand; i += kConsumers) {
                        const float z1[1] = {key_logit(sh.fcand[i])};
                        take(z1, 1u, 0);
                    }
                SPECDEC_STAMP(11);
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1) {
                    kmn = min(kmn, __shfl_xor_sync(0xffffffffu, kmn, off));
                    kmx = max(kmx, __shfl_xor_sync(0xffffffffu, kmx, off));
                }
                if (lane == 0) { sh.fw_kmin[cw] = kmn; sh.fw_kmax[cw] = kmx; }
                const unsigned long long m_bin = fold_u64(mbin, sh.fw_m);       // (its barrier covers the keys)
                const unsigned long long m_above = fold_u64(mab, sh.fw_m2);
                if (ct == 0) {
                    uint32_t k0 = 0xffffffffu, k1 = 0u;
                    for (int w = 0; w < kConsumerWarps; ++w) { k0 = min(k0, sh.fw_kmin[w]); k1 = max(k1, sh.fw_kmax[w]); }
                    sh.fc_kmin = k0; sh.fc_kmax = k1; sh.fc_mbin = m_bin; sh.fc_mabove = m_above;
                }
                consumer_sync();
                return ncand < 0 ? (int)sh.fncand : ncand;
            };
            // One pass over the row appending the key of every allowed element whose logit is at least
            // zt (a top slice of the row). Returns their number (above kCandCap: only the first
            // kCandCap kept).
            auto slice_pass = [&](int64_t t, int j, float zt) -> int {
                if (ct == 0) sh.fncand = 0u;
                consumer_sync();
                SPECDEC_STAMP(10);
                visit_row(t, j, [&](const auto& z, uint32_t valid, int) {
                    constexpr int N = (int)(sizeof(z) / sizeof(z[0]));
                    uint32_t take = 0u;
#pragma unroll
                    for (int i = 0; i < N; ++i) take |= (((valid >> i) & 1u) && z[i] >= zt ? 1u : 0u) << i;
                    if (take == 0u) return;
#pragma unroll
                    for (int i = 0; i < N; ++i)
                        if ((take >> i) & 1u) {
                            const uint32_t pos = atomicAdd(&sh.fncand, 1u);
                            if (pos < (uint32_t)kCandCap) sh.fcand[pos] = logit_key(z[i]);
                        }
                });
                SPECDEC_STAMP(11);
                consumer_sync();
                return (int)sh.fncand;
            };
            // the threshold key for one search: mode 0 (top-k: the `need`-th largest element) or
            // mode 1 (top-p: the smallest key whose mass above is below P = p_frac of the mass at or
            // above floor_key). Returns the key, the mass above it (`mass_above`) and the mass of its
            // own ties (`mass_at`); false when the search keeps every element (top-k with k >= the
            // elements). The digit passes stop at bit 16 for bf16 logits: below it a key's bits
            // follow from its sign bit (all zero for z >= 0, all one below).
            // After the first pass chooses a mass bin, a collection pass takes its key range and
            // mass and, when they fit on chip, the keys of its elements (of every element from that
            // bin up when `keep_above` and they fit, for a search that follows); the digit passes
            // then run over those candidates instead of the row. `ncand` >= 0 on entry means the
            // candidates already hold every element at or above floor_key, so the whole search
            // runs on chip; on return it is >= 0 when that holds for this search's kept elements.
            auto search = [&](int64_t t, int j, int mode, unsigned long long need, float p_frac, uint32_t floor_key,
                              float MC, float S, bool keep_above, int& slice_oct, int& ncand, uint32_t& key_out,
                              unsigned long long& mass_above, unsigned long long& mass_at, const Settle& st) -> bool {
                constexpr int kLowBit = (sizeof(ET) == 2) ? 16 : 0;
                int src0 = ncand;
                // Top-k: first try the top slice of logits whose mass exp2(z*c - MC) is at least
                // 1.0625 S / kCandCap (at most about kCandCap of them, S the row's softmax sum), lowered
                // by slice_oct octaves: when it holds k elements (and no more than fit) it holds the
                // k-th largest and everything above it, and the whole search (and a top-p search after
                // it) runs on chip. A slice with too few elements is tried once more 16x lower, one with
                // too many 4x higher; the level that worked is where the request's next row starts.
                // After two misses the row is searched as below, and the request stops trying.
                bool top_slice = false;
                if (src0 < 0 && mode == 0 && slice_oct >= 0 && need * 17 <= (unsigned long long)kCandCap * 16) {
                    for (int attempt = 0; attempt < 2 && !top_slice; ++attempt) {
                        const float zt = (__log2f(S * (1.0625f / (float)kCandCap)) - (float)slice_oct + MC) / c;
                        const int n = slice_pass(t, j, zt);
                        if (n <= kCandCap && (unsigned long long)n >= need) { src0 = n; top_slice = true; }
                        else if (n > kCandCap) slice_oct = max(0, slice_oct - 2);
                        else slice_oct += 4;
                    }
                    if (!top_slice) slice_oct = -1;
                }
                // on chip, the first pass takes counts and masses (the candidates are few)
                hist_pass(t, j, -1, 0u, 0u, 0, 0u, floor_key, MC, 0u, 0xffffffffu, src0,
                          src0 >= 0 ? 3 : (mode == 0 ? 1 : 2));
                select_digit(mode, need, 0ull, 0ull, -1, mode == 1 ? p_frac : -1.f);
                const unsigned long long P = sh.fsel_P;
                const uint32_t b0 = sh.fsel_digit;
                if (b0 == 0xffffffffu) {                             // top-k covers every element
                    mass_above = sh.ftot_mass;
                    mass_at = 0ull;
                    return false;
                }
                if (mode == 1 && st.on) {
                    // The threshold lies in mass bin b0, so the kept mass is at most the mass of b0 and
                    // everything above it: an accepted row of a surely kept draft whose uniform lies
                    // below the ratio that bound gives needs no more passes. It returns no threshold
                    // (key 0) and that bound as the kept mass, with which the acceptance test passes.
                    constexpr float kLo = 1.f - 1e-4f, kHi = 1.f + 1e-4f;
                    const unsigned long long hi = sh.fsel_mass + sh.fsel_at + 256ull;   // (+ the fx40 truncations)
                    const float S_hi = (float)hi * 0x1p-40f;
                    const bool kept = st.cok && st.A * kHi < (float)P * 0x1p-40f * kLo;
                    const float px_lo = st.ex / S_hi * kLo;
                    const float alpha_lo = !st.qmode ? px_lo : (px_lo >= st.qx ? 1.f : px_lo / st.qx * kLo);
                    if (kept && px_lo > 0.f && st.u < alpha_lo) {
                        key_out = 0u;
                        mass_above = hi;
                        mass_at = 0ull;
                        return true;
                    }
                }
                const unsigned long long n_above = sh.fsel_cnt, n_bin = sh.fsel_n;
                unsigned long long above = sh.fsel_mass;          // (first top-k pass: not summed)
                need -= n_above;
                int src = src0;
                if (top_slice) ncand = src0;             // every element at or above this search's key
                else if (src0 < 0) ncand = -1;
                const bool all = src0 < 0 && keep_above && n_above + n_bin <= (unsigned long long)kCandCap;
                const int n = collect_pass(t, j, b0, all, mode == 0, floor_key, MC, src0);
                if (src0 < 0 && n <= kCandCap) {
                    src = n;
                    if (all) ncand = n;
                }
                if (mode == 0) above = sh.fc_mabove;
                unsigned long long at = fx40(sh.fc_mbin, bin_exp(b0));
                uint32_t kmin = sh.fc_kmin;
                const uint32_t kmax = sh.fc_kmax;
                // resolve the keys of bin b0 from the highest bit where they differ, 8 bits a pass
                if (kmin != kmax) {
                    const int hb = 31 - __clz(kmin ^ kmax);
                    uint32_t pmask = hb == 31 ? 0u : (0xffffffffu << (hb + 1));
                    uint32_t pval = kmin & pmask;
                    for (int top = hb; top >= kLowBit; top -= 8) {
                        const int shift = max(kLowBit, top - 7);
                        const uint32_t width = (1u << (top - shift + 1)) - 1u;
                        hist_pass(t, j, (int)b0, pmask, pval, shift, width, floor_key, MC, kmin, kmax, src, 3);
                        select_digit(mode, need, P, above, (int)b0, -1.f);
                        const uint32_t dg = sh.fsel_digit;           // always found inside the bin
                        above += sh.fsel_mass;
                        at = sh.fsel_at;
                        need -= sh.fsel_cnt;
                        pval |= dg << shift;
                        pmask |= width << shift;
                    }
                    if (kLowBit > 0) pval |= (pval & 0x80000000u) ? 0u : ((1u << kLowBit) - 1u);
                    kmin = pval;
                }
                key_out = kmin;
                mass_above = above;
                mass_at = at;
                return true;
            };
            auto filter_row = [&](int64_t t, int j, float MC, float S, uint32_t& kt, float& S_keep, const Settle& st) -> bool {
                uint32_t floor_key = 0u;
                unsigned long long keep = 0ull, above = 0ull, at = 0ull;      // masses in units of 2^-40
                int ncand = -1;                                  // candidates hold every kept element
                bool cut_k = false;
                if (fk > 0) {
                    uint32_t key;
                    cut_k = search(t, j, 0, (unsigned long long)fk, 0.f, 0u, MC, S, fp < 1.f, slice_oct, ncand, key,
                                   above, at, Settle{});
                    if (cut_k) { floor_key = key; keep = above + at; }
                }
                bool cut_p = false;
                if (fp < 1.f) {
                    uint32_t key;
                    int no_slice = -1;
                    cut_p = search(t, j, 1, 0ull, fp, floor_key, MC, S, false, no_slice, ncand, key, above,
                                   at, st);
                    if (cut_p) { floor_key = key; keep = above + at; }
                }
                kt = floor_key;
                SPECDEC_STAMP(12);
                S_keep = (float)keep * 0x1p-40f;
                return cut_k || cut_p;
            };

            // ---- decision on row j from its reduced partial r (identical in every consumer thread
            // of every CTA of the request); returns the next code (a draw kind, next row, done)
            auto decide = [&](int j, const Part& r, bool& stop, float& MC, float& S_mc, bool cut, uint32_t kt,
                              float S_keep) -> int {
                const int64_t t = rs.row0 + j;
                const int64_t d = (int64_t)rs.d0 + j;
                const bool bonus = (j == k);
                const int x = bonus ? -1 : sh.xs[j];
                (void)d;
                int code = kDecDone;
                stop = true;
                MC = 0.f;
                S_mc = 1.f;
                if (greedy) {
                    if (r.idx == INT_MAX) {
                        st |= SPECDEC_ST_EMPTY_MASK_ROW;
                        if (writer && a.diag_row) { a.diag_row[2 * t] = -INFINITY; a.diag_row[2 * t + 1] = NAN; }
                        acc_len = j; emitted = -1;
                    } else {
                        if (writer && a.diag_row) { a.diag_row[2 * t] = r.best; a.diag_row[2 * t + 1] = NAN; }
                        if (bonus) {
                            emitted = r.idx;
                        } else {
                            const bool accept = (j < g) && (x == r.idx);
                            if (writer && a.diag_alpha) a.diag_alpha[d] = accept ? 1.f : 0.f;
                            if (accept) { if (writer) a.out_tokens[t] = x; stop = false; code = kDecNextRow; }
                            else { acc_len = j; emitted = r.idx; }
                        }
                    }
                } else if (r.m == -INFINITY) {
                    st |= SPECDEC_ST_EMPTY_MASK_ROW;
                    if (writer && a.diag_row) { a.diag_row[2 * t] = -INFINITY; a.diag_row[2 * t + 1] = 0.f; }
                    acc_len = j; emitted = -1;
                } else {
                    MC = r.m * c;
                    // S against MC = round(M*c), the reference the draw terms use
                    S_mc = fmaf(r.S, fmaf(r.m, c, -MC) * 0.69314718f, r.S);
                    if (writer && a.diag_row) { a.diag_row[2 * t] = r.m / T; a.diag_row[2 * t + 1] = r.S; }
                    if (cut) S_mc = S_keep;                        // top-k / top-p: the kept ids' mass
                    code = kDecDrawP;
                    if (!bonus) {
                        float alpha = 0.f;
                        if (j < g) {
                            const bool kept = r.zx > -INFINITY && (!cut || logit_key(r.zx) >= kt);
                            const float px = kept ? ex2_scaled(r.zx, c, MC) / S_mc : 0.f;
                            if (qmode) {
                                const float qx = sh.qxs[j];
                                alpha = (px <= 0.f) ? 0.f : (qx <= px ? 1.f : px / qx);
                            } else {
                                alpha = px;
                            }
                        }
                        if (writer && a.diag_alpha) a.diag_alpha[d] = alpha;
                        if (sh.us[j] < alpha) { if (writer) a.out_tokens[t] = x; stop = false; code = kDecNextRow; }
                        else code = qmode ? kDecDrawQ : kDecDrawOneHot;
                    }
                }
                return code;
            };

            // ---- decision on race row j (see race_raise): the bonus token, or the acceptance test
            // of model-free draft j with p(x) from the same pass and, on a rejection, the race's
            // winner (p without the draft token) as the recovered token
            auto decide_race = [&](int j, const Part& r, bool& stop) -> int {
                const int64_t t = rs.row0 + j;
                const int64_t d = (int64_t)rs.d0 + j;
                const bool bonus = (j == k);
                stop = true;
                if (!(r.m > -INFINITY)) {
                    st |= SPECDEC_ST_EMPTY_MASK_ROW;
                    if (writer && a.diag_row) { a.diag_row[2 * t] = -INFINITY; a.diag_row[2 * t + 1] = 0.f; }
                    acc_len = j; emitted = -1;
                    return kDecDone;
                }
                const float mcr = __int_as_float(r.flag);      // the reference of r.S and r.best
                if (writer && a.diag_row) {
                    a.diag_row[2 * t] = r.m / T;
                    a.diag_row[2 * t + 1] = r.S * ex2(fmaf(-r.m, c, mcr));   // S against exp2(m * c)
                }
                const int tok = r.idx == INT_MAX ? -1 : r.idx;
                if (bonus) { emitted = tok; return kDecDone; }
                const float alpha = (j < g && r.zx > -INFINITY) ? ex2(fmaf(r.zx, c, -mcr)) / r.S : 0.f;
                if (writer && a.diag_alpha) a.diag_alpha[d] = alpha;
                if (sh.us[j] < alpha) { if (writer) a.out_tokens[t] = sh.xs[j]; stop = false; return kDecNextRow; }
                acc_len = j; emitted = tok;
                return kDecDone;
            };

            // ---- a9/a10: draw pass(es) over the stop / bonus row j
            auto draw_row = [&](int j, int code, float MC, float S_mc, uint32_t kt) {
                const int64_t t = rs.row0 + j;
                const int64_t d = (int64_t)rs.d0 + j;
                const int x = (j == k) ? -1 : sh.xs[j];
                while (code == kDecDrawP || code == kDecDrawQ || code == kDecDrawOneHot) {
                    SPECDEC_STAMP(5);
                    const float invS = 1.f / S_mc;
                    Part dp = part_identity();
                    if (!sparse) {
                        const bool wq = (code == kDecDrawQ);
                        const int ids = G::draw_ids(wq);
                        const int nd = (hi - lo + ids - 1) / ids;
                        for (int ch = 0; ch < nd; ++ch) {
                            const int s = wait_full();
                            const unsigned char* stg = ring + (size_t)s * kStageBytes;
                            const uint32_t* sm = reinterpret_cast<const uint32_t*>(stg + G::dmask_off(wq));
                            const float* se = reinterpret_cast<const float*>(stg + G::noise_off(wq));
                            const float* sq = reinterpret_cast<const float*>(stg + G::q_off(wq));
                            const int i0 = lo + ch * ids;
                            const int n = min(ids, hi - i0);
                            const int nvec = (n + VE - 1) / VE;
                            constexpr int NB = (VE == 4) ? 2 : 1;
                            const int vxd = (code == kDecDrawOneHot && x >= i0 && x < i0 + n) ? (x - i0) / VE : -1;
                            for (int vb = ct; vb < nvec; vb += kConsumers * NB) {
                                float z[NB * VE], ev[NB * VE], qv[NB * VE];
                                int xslot = -1;
#pragma unroll
                                for (int u = 0; u < NB; ++u) {
                                    const int v = vb + u * kConsumers;
                                    const int e0 = v * VE;
                                    if (v < nvec) {
                                        Elem<ET>::load(stg, v, z + u * VE);
                                        const uint32_t bits = vec_bits<VE>(sm, has_mask, v);
                                        if (bits != (1u << VE) - 1u) {
#pragma unroll
                                            for (int e = 0; e < VE; ++e) z[u * VE + e] = ((bits >> e) & 1u) ? z[u * VE + e] : -INFINITY;
                                        }
                                        if (kt != 0u) {                  // top-k / top-p: ids below the threshold
#pragma unroll
                                            for (int e = 0; e < VE; ++e)
                                                if (logit_key(z[u * VE + e]) < kt) z[u * VE + e] = -INFINITY;
                                        }
#pragma unroll
                                        for (int h = 0; h < VE / 4; ++h) {
                                            const float4 f = reinterpret_cast<const float4*>(se + e0)[h];
                                            ev[u * VE + 4 * h] = f.x; ev[u * VE + 4 * h + 1] = f.y; ev[u * VE + 4 * h + 2] = f.z; ev[u * VE + 4 * h + 3] = f.w;
                                            if (wq) {
                                                const float4 g4 = reinterpret_cast<const float4*>(sq + e0)[h];
                                                qv[u * VE + 4 * h] = g4.x; qv[u * VE + 4 * h + 1] = g4.y; qv[u * VE + 4 * h + 2] = g4.z; qv[u * VE + 4 * h + 3] = g4.w;
                                            } else {
                                                qv[u * VE + 4 * h] = qv[u * VE + 4 * h + 1] = qv[u * VE + 4 * h + 2] = qv[u * VE + 4 * h + 3] = 0.f;
                                            }
                                        }
                                        if (v == vxd) xslot = u * VE + (x - i0) % VE;
                                    } else {
#pragma unroll
                                        for (int e = 0; e < VE; ++e) { z[u * VE + e] = -INFINITY; ev[u * VE + e] = 1.f; qv[u * VE + e] = 0.f; }
                                    }
                                }
                                draw_lazy<NB, VE>(dp, z, ev, qv, i0 + vb * VE, kConsumers * VE, xslot, code, c, MC, invS);
                            }
                            release(s);
                        }
                    } else {
                        if (listed_row == j) {
                            sparse_draw(t, d, x, listed_n, code, dp, MC, invS, kt);
                        } else {
                            for (int w0 = wlo; w0 < whi; w0 += kSegWords) {
                                const int w1 = min(whi, w0 + kSegWords);
                                const int n = build_list(t, w0, w1);
                                if (n >= 0) {
                                    sparse_draw(t, d, x, n, code, dp, MC, invS, kt);
                                } else {
                                    for (int s0 = w0; s0 < w1; s0 += G::kSafeWords)
                                        sparse_draw(t, d, x, build_list(t, s0, min(w1, s0 + G::kSafeWords)), code, dp, MC, invS, kt);
                                }
                            }
                        }
                    }
                    SPECDEC_STAMP(6);
                    const Part dr = reduce(dp);
                    if (code == kDecDrawQ && !dr.flag) { code = kDecDrawP; post(code); continue; }   // empty residual
                    emitted = dr.idx == INT_MAX ? -1 : dr.idx;
                    post(kDecDone);
                    break;
                }
            };

            // ---- draw over the kept ids only (top-k requests): one more pass over the row's logits
            // lists the ids at or above the threshold key kt (at most k plus ties) in the candidate
            // slots; each is then drawn from its own logit, noise and q, loaded one by one, instead of
            // streaming the noise and q rows as draw_row does. The per-id terms and the tie rule
            // (the lowest id on equal scores) are draw_lazy's, so the token is the one draw_row
            // would emit. Returns false, with the draw code posted, when the ids do not fit (the
            // caller then runs draw_row).
            auto draw_kept = [&](int j, int code, float MC, float S_mc, uint32_t kt) -> bool {
                const int64_t t = rs.row0 + j;
                const int64_t d = (int64_t)rs.d0 + j;
                const int x = (j == k) ? -1 : sh.xs[j];
                if (ct == 0) sh.fncand = 0u;
                consumer_sync();
                SPECDEC_STAMP(10);
                visit_row(t, j, [&](const auto& z, uint32_t valid, int id0) {
                    constexpr int N = (int)(sizeof(z) / sizeof(z[0]));
#pragma unroll
                    for (int i = 0; i < N; ++i)
                        if (((valid >> i) & 1u) && logit_key(z[i]) >= kt) {
                            const uint32_t pos = atomicAdd(&sh.fncand, 1u);
                            if (pos < (uint32_t)kCandCap) sh.fcand[pos] = (uint32_t)(id0 + i);
                        }
                });
                consumer_sync();
                SPECDEC_STAMP(11);
                const int n = (int)sh.fncand;
                if (n > kCandCap) { post(code); return false; }
                while (true) {
                    SPECDEC_STAMP(5);
                    const float invS = 1.f / S_mc;
                    const bool wq = (code == kDecDrawQ);
                    Part dp = part_identity();
                    for (int i = ct; i < n; i += kConsumers) {
                        const int id = (int)sh.fcand[i];
                        const float z = load_logit<ET>(a.logits, t * (int64_t)a.V + id);
                        const float E = __ldg(a.noise + t * (int64_t)a.V + id);
                        const float q = wq ? __ldg(a.q + d * (int64_t)a.V + id) : 0.f;
                        const float pe = ex2_scaled(z, c, MC) * invS;
                        float w = pe;
                        if (wq) w = fmaxf(pe - q, 0.f);
                        else if (code == kDecDrawOneHot && id == x) w = 0.f;
                        if (w > 0.f && z > -INFINITY) {
                            dp.flag = 1;
                            const float sc = w * fast_rcp(E);
                            if (sc > 0.f && (sc > dp.best || (sc == dp.best && id < dp.idx))) { dp.best = sc; dp.idx = id; }
                        }
                    }
                    SPECDEC_STAMP(6);
                    const Part dr = reduce(dp);
                    if (code == kDecDrawQ && !dr.flag) { code = kDecDrawP; continue; }   // empty residual
                    emitted = dr.idx == INT_MAX ? -1 : dr.idx;
                    break;
                }
                post(kDecDone);
                return true;
            };

            // race rows (see race_raise; the producer applies the same test): the bonus row of an
            // unfiltered sampled request and every row of an unfiltered sampled model-free one
            const bool race_req = !greedy && !filt;
            for (int j = 0; j <= k; ++j) {
                const int64_t t = rs.row0 + j;
                const bool bonus = (j == k);
                const int x = bonus ? -1 : sh.xs[j];
                const bool race = race_req && (bonus || !qmode);
                Part p = part_identity();
                float mc = 0.f;                            // running round(m * c) (race rows: a whole number)
                // acceptance bound of a filtered draft row (dense, one CTA, no per-draft diagnostics):
                // the count and mass of the logits above the draft token's, from the statistics pass
                const bool bound_on = kFilt && filt && !sparse && !bonus && j < g && NC == 1 && a.diag_alpha == nullptr;
                float zxb = INFINITY, mass_above = 0.f;
                uint32_t cnt_above = 0u;
                if (bound_on) zxb = load_logit<ET>(a.logits, t * (int64_t)a.V + x);

                if (!sparse && race) {
                    // ---- a2/a3/a5 + a9/a10 dense, one pass: logits, noise and mask words of the slice
                    const int ids = G::draw_ids(false);
                    const int nd = (hi - lo + ids - 1) / ids;
                    for (int ch = 0; ch < nd; ++ch) {
                        const int s = wait_full();
                        if (ch == 0) SPECDEC_STAMP(2);
                        const unsigned char* stg = ring + (size_t)s * kStageBytes;
                        const uint32_t* sm = reinterpret_cast<const uint32_t*>(stg + G::dmask_off(false));
                        const float* se = reinterpret_cast<const float*>(stg + G::noise_off(false));
                        const int i0 = lo + ch * ids;
                        const int n = min(ids, hi - i0);
                        const int nvec = (n + VE - 1) / VE;
                        const int vx = (x >= i0 && x < i0 + n) ? (x - i0) / VE : -1;
                        constexpr int NB = (VE == 4) ? 4 : 2;
                        constexpr uint32_t kFull = (1u << VE) - 1u;
                        for (int vb = ct; vb < nvec; vb += kConsumers * NB) {
                            uint4 raw[NB];
                            uint32_t bits[NB];
                            float ev[NB * VE];
                            bool full = true;
                            int xslot = -1;
#pragma unroll
                            for (int u = 0; u < NB; ++u) {
                                const int v = vb + u * kConsumers;
                                const bool in = v < nvec;
                                const uint32_t ni = Raw<ET>::kNegInf;
                                raw[u] = in ? reinterpret_cast<const uint4*>(stg)[v] : make_uint4(ni, ni, ni, ni);
                                bits[u] = (in && has_mask) ? vec_bits<VE>(sm, true, v) : kFull;
                                full = full && (bits[u] == kFull);
#pragma unroll
                                for (int h = 0; h < VE / 4; ++h) {
                                    const float4 f = in ? reinterpret_cast<const float4*>(se + v * VE)[h] : make_float4(1.f, 1.f, 1.f, 1.f);
                                    ev[u * VE + 4 * h] = f.x; ev[u * VE + 4 * h + 1] = f.y; ev[u * VE + 4 * h + 2] = f.z; ev[u * VE + 4 * h + 3] = f.w;
                                }
                                if (v == vx) xslot = u * VE + (x - i0) % VE;
                            }
                            float z[NB * VE];
#pragma unroll
                            for (int u = 0; u < NB; ++u) unpack_raw<ET>(raw[u], z + u * VE);
                            float bm;
                            if (full) {
                                bm = raw_max<ET, NB>(raw, z);
                            } else {
#pragma unroll
                                for (int u = 0; u < NB; ++u)
#pragma unroll
                                    for (int e = 0; e < VE; ++e)
                                        z[u * VE + e] = ((bits[u] >> e) & 1u) ? z[u * VE + e] : -INFINITY;
                                bm = tree_max<NB * VE>(z);
                            }
                            race_lazy<NB, VE>(p, mc, z, ev, bm, i0 + vb * VE, kConsumers * VE, xslot, c);
                        }
                        // the draft token's logit, read once by the thread that owns its group
                        if (vx >= 0 && ct == vx % kConsumers) {
                            float zz[VE];
                            Elem<ET>::load(stg, vx, zz);
#pragma unroll
                            for (int e = 0; e < VE; ++e)
                                if (e == (x - i0) % VE) p.zx = zz[e];
                        }
                        release(s);
                    }
                } else if (!sparse) {
                    // ---- a2/a3/a5/a6 dense: stream the slice chunk by chunk
                    for (int ch = 0; ch < nrow_chunks; ++ch) {
                        const int s = wait_full();
                        if (ch == 0) SPECDEC_STAMP(2);
                        if (j == 0 && ch > 0) SPECDEC_STAMP(8);
                        const unsigned char* stg = ring + (size_t)s * kStageBytes;
                        const uint32_t* sm = reinterpret_cast<const uint32_t*>(stg + G::kRowMaskOff);
                        const int i0 = lo + ch * G::kRowIds;
                        const int n = min(G::kRowIds, hi - i0);
                        const int nvec = (n + VE - 1) / VE;
                        constexpr int NB = 4;
                        constexpr uint32_t kFull = (1u << VE) - 1u;
                        for (int vb = ct; vb < nvec; vb += kConsumers * NB) {
                            uint4 raw[NB];
                            uint32_t bits[NB];
                            bool full = true;
#pragma unroll
                            for (int u = 0; u < NB; ++u) {
                                const int v = vb + u * kConsumers;
                                const bool in = v < nvec;
                                const uint32_t ni = Raw<ET>::kNegInf;
                                raw[u] = in ? reinterpret_cast<const uint4*>(stg)[v] : make_uint4(ni, ni, ni, ni);
                                bits[u] = (in && has_mask) ? vec_bits<VE>(sm, true, v) : kFull;
                                full = full && (bits[u] == kFull);
                            }
                            float z[NB * VE];
#pragma unroll
                            for (int u = 0; u < NB; ++u) unpack_raw<ET>(raw[u], z + u * VE);
                            float bm;
                            if (full) {
                                bm = raw_max<ET, NB>(raw, z);
                            } else {
#pragma unroll
                                for (int u = 0; u < NB; ++u)
#pragma unroll
                                    for (int e = 0; e < VE; ++e)
                                        z[u * VE + e] = ((bits[u] >> e) & 1u) ? z[u * VE + e] : -INFINITY;
                                bm = tree_max<NB * VE>(z);
                            }
                            if (greedy) argmax_lazy<NB, VE>(p, z, bm, i0 + vb * VE, kConsumers * VE);
                            else if (bound_on) softmax_fold_max_above<NB * VE>(p, mc, mass_above, cnt_above, z, bm, c, zxb);
                            else softmax_fold_max<NB * VE>(p, mc, z, bm, c);
                        }
                        // the draft token's logit, read once by the thread that owns its group
                        if (!greedy && x >= i0 && x < i0 + n && ct == ((x - i0) / VE) % kConsumers) {
                            float zz[VE];
                            Elem<ET>::load(stg, (x - i0) / VE, zz);
#pragma unroll
                            for (int e = 0; e < VE; ++e)
                                if (e == (x - i0) % VE) p.zx = zz[e];
                        }
                        if (j == 0) SPECDEC_STAMP(9);
                        release(s);
                    }
                } else {
                    // ---- sparse: gather only the allowed 16-byte groups of the slice
                    listed_row = -1;
                    for (int w0 = wlo; w0 < whi; w0 += kSegWords) {
                        const int w1 = min(whi, w0 + kSegWords);
                        const int n = build_list(t, w0, w1);
                        if (w0 == wlo) SPECDEC_STAMP(2);
                        if (n >= 0) {
                            if (race) sparse_race(t, x, n, p, mc);
                            else sparse_stats(t, greedy ? -1 : x, n, p, mc);
                            if (!race && w1 - w0 == whi - wlo) { listed_row = j; listed_n = n; }   // the whole slice in one list
                        } else {
                            for (int s0 = w0; s0 < w1; s0 += G::kSafeWords) {
                                const int n2 = build_list(t, s0, min(w1, s0 + G::kSafeWords));
                                if (race) sparse_race(t, x, n2, p, mc);
                                else sparse_stats(t, greedy ? -1 : x, n2, p, mc);
                            }
                        }
                    }
                }
                SPECDEC_STAMP(3);
                if (race) {
                    p.flag = __float_as_int(p.m > -INFINITY ? mc : -INFINITY);
                    const Part r = reduce_any(p, std::true_type{});
                    SPECDEC_STAMP(4);
                    bool stop;
                    post(decide_race(j, r, stop));
                    if (!stop) continue;
                    // drain the chunks of row j+1 the producer queued before this decision
                    if (!sparse && j < k)
                        for (int ch = 0; ch < spec; ++ch) release(wait_full());
                    acc_len = j;
                    break;
                }
                // each thread's terms were taken against mc = round(m*c); rebase its sum on the
                // exact m*c (combine() rescales partials by exp2((m_a - m_b) * c))
                if (!greedy && p.m > -INFINITY) {
                    const float dlt = fmaf(p.m, c, -mc);           // exact: m*c - round(m*c)
                    p.S = fmaf(p.S, -dlt * 0.69314718f, p.S);     // * 2^-dlt, |dlt| tiny
                }
                const Part r = reduce(p);
                SPECDEC_STAMP(4);

                uint32_t kt = 0u;
                float S_keep = 0.f;
                bool cut = false;
                if constexpr (kFilt) {
                    // Acceptance without the threshold search. Filtering only removes mass, so the kept
                    // mass is at most the row's S and the filtered p'(x) at least e_x / S: a draft that is
                    // surely kept and whose uniform lies below that bound's acceptance ratio is accepted
                    // whatever the threshold is. Kept for sure: fewer than k logits above x (top-k),
                    // and the mass above x below p of the total (top-p) or, after a top-k cut, below p
                    // of the mass of x and everything above it (a lower bound of the top-k mass).
                    // The fp32 sums here differ from the search's exact integer sums by far less than
                    // the 1e-4 margins; a row the bound does not settle takes the search as before.
                    bool sure = false;
                    Settle st{};
                    if (bound_on && r.m > -INFINITY && r.zx > -INFINITY) {
                        const float MCb = r.m * c;
                        float av = (p.m > -INFINITY) ? mass_above * ex2(mc - MCb) : 0.f;
                        uint32_t cv = cnt_above;
#pragma unroll
                        for (int off = 16; off >= 1; off >>= 1) {
                            av += __shfl_xor_sync(0xffffffffu, av, off);
                            cv += __shfl_xor_sync(0xffffffffu, cv, off);
                        }
                        if (lane == 0) { sh.fw_a[cw] = av; sh.fw_cnt[cw] = cv; }
                        consumer_sync();
                        float A = 0.f;
                        unsigned long long C = 0ull;
#pragma unroll
                        for (int w = 0; w < kConsumerWarps; ++w) { A += sh.fw_a[w]; C += sh.fw_cnt[w]; }
                        const float Smc = fmaf(r.S, fmaf(r.m, c, -MCb) * 0.69314718f, r.S);
                        const float ex = ex2_scaled(r.zx, c, MCb);
                        constexpr float kLo = 1.f - 1e-4f, kHi = 1.f + 1e-4f;
                        bool kept = fk <= 0 || C < (unsigned long long)fk;
                        if (fp < 1.f) kept = kept && A * kHi < fp * (fk > 0 ? A + ex : Smc) * kLo;
                        const float px_lo = ex / Smc * kLo;
                        const float alpha_lo = !qmode ? px_lo : (px_lo >= sh.qxs[j] ? 1.f : px_lo / sh.qxs[j] * kLo);
                        sure = kept && px_lo > 0.f && sh.us[j] < alpha_lo;
                        st = Settle{true, fk <= 0 || C < (unsigned long long)fk, qmode, A, ex, sh.qxs[j], sh.us[j]};
                    }
                    cut = filt && !sure && r.m > -INFINITY && filter_row(t, j, r.m * c, r.S, kt, S_keep, st);
                }
                bool stop;
                float MC, S_mc;
                const int code = decide(j, r, stop, MC, S_mc, cut, kt, S_keep);
                // a filtered stop row with few kept ids draws over those ids only: at most k of them
                // for top-k without ties, and at most S_keep / e(kt) in any case (each kept id has
                // mass at least e(kt), the threshold logit's)
                bool kept_draw = false;
                if constexpr (kFilt) {
                    if (stop && cut && kt != 0u && (code == kDecDrawP || code == kDecDrawQ || code == kDecDrawOneHot)) {
                        const float ekt = ex2_scaled(key_logit(kt), c, MC);
                        const float nmax = ekt > 0.f ? S_keep / ekt : INFINITY;
                        kept_draw = (fk > 0 && fk <= kCandCap - 64) || nmax <= (float)(kCandCap - 64);
                    }
                }
                if (!kept_draw) post(code);
                if (!stop) continue;

                // drain the chunks of row j+1 the producer queued before this decision
                if (!sparse && j < k && !filt)
                    for (int ch = 0; ch < spec; ++ch) release(wait_full());
                if (!kept_draw || !draw_kept(j, code, MC, S_mc, kt))
                    draw_row(j, code, MC, S_mc, cut ? kt : 0u);
                acc_len = j;
                break;
            }
        }

        SPECDEC_STAMP(7);
        SPECDEC_TRACE_END();
        // ---- a11: emit, count
        if (writer) {
            if (rs.skip == 0) {
                a.out_tokens[rs.row0 + acc_len] = emitted;
                for (int j = acc_len + 1; j <= k; ++j) a.out_tokens[rs.row0 + j] = -1;
                atomicAdd(&a.counters[0], (unsigned long long)k);
                atomicAdd(&a.counters[1], (unsigned long long)(k - g));
                atomicAdd(&a.counters[2], (unsigned long long)g);
                atomicAdd(&a.counters[3], (unsigned long long)acc_len);
                if (a.telemetry) add_telemetry_serial(a.telemetry, k, g, acc_len);
            } else if (rs.skip == 2) {
                for (int j = 0; j <= k; ++j) a.out_tokens[rs.row0 + j] = -1;
            }
            a.out_num_accepted[b] = rs.skip == 0 ? acc_len : 0;
            if (a.status) a.status[b] = st;
        }
    }
    __syncthreads();
    // after an expired wait, bulk copies may still be in flight: wait (bounded, a separate limit)
    // for the last copy issued into each stage before the CTA leaves, so that none lands in shared
    // memory the CTA no longer owns
    if (tid == 0 && sh.timed_out && a.bulk) {
        const uint32_t issued = sh.issued;
        for (uint32_t s = 0; s < (uint32_t)kStages && s < issued; ++s) {
            const uint32_t last = s + ((issued - 1u - s) / kStages) * kStages;
            (void)mbar_wait_bounded(smem_addr(&sh.full[s]), (last / kStages) & 1u, kDrainLimitNs);
        }
    }
    // a copy that missed its deadline marks the request (any CTA of it) after rank 0 wrote status
    if (NC > 1) cluster_sync_all();
    if (tid == 0 && sh.timed_out && a.status) atomicOr(&a.status[b], SPECDEC_ST_DEVICE_TIMEOUT);
}

// ---------------------------------------------------------------------------------------------
// request schedule (longest-processing-time first)
// ---------------------------------------------------------------------------------------------
//
// The requests of a batch are independent chains of row passes whose lengths differ by more
// than 10x: a greedy request streams logits rows only, a sampled one adds a draw pass over the
// stop row's logits, noise and (draft model) q, and a request with a sparse bitmask gathers a
// fraction of every row. The block scheduler starts clusters in index order as slots free up,
// so a heavy request that sits late in the batch runs on alone after the others have finished.
// Ordering the requests heaviest first (the longest-processing-time rule of list scheduling)
// lets the light ones fill in behind. The order only affects timing: every request's outputs
// are the same under any order.
//
// One CTA computes an integer cost key per request and a stable counting sort of the keys,
// descending, into order[B]. The key estimates the request's duration in units of 1/16 of a
// dense logits row pass, without knowing where it will stop:
//   rows: 1 + 0.6 k for a draft-model request (its drafts are mostly accepted), 1 + 0.3 k for a
//   greedy one, one race row over logits + noise for a sampled model-free one (accepted with
//   probability p(x), usually small); a sparse row (the same test the verify kernel applies)
//   counts 0.65 of a dense one;
//   a draft-model request's draw over logits, noise and q: 0.85 * (bytes per id of the three) /
//   (bytes per id of logits) when dense, 0.7 when sparse.

constexpr int kSchedThreads = 1024;
constexpr int kSchedWarps = kSchedThreads / 32;
constexpr int kSchedKeys = 256;

template <typename ET>
__device__ __forceinline__ int request_cost_key(const Args& a, int b)
{
    // the loads that depend on nothing are issued together; only the mask words wait for cu[b]
    const float T = __ldg(a.temperature + b);
    const bool hq = a.has_q == nullptr || __ldg(a.has_q + b) != 0;
    const ReqShape rs = request_shape(a, b);
    if (rs.skip != 0) return 0;
    const bool tvalid = (T == 0.f) || (T >= FLT_MIN && T <= FLT_MAX);
    const bool greedy = !(T > 0.f) || !tvalid;
    const bool qmode = a.q != nullptr && hq;
    bool sparse = false;
    if (a.bitmask != nullptr && a.bulk) {
        // the verify kernel's test, one thread instead of one warp: fewer than half of the
        // first min(W, 32) mask words' bits set (rows are 16-byte aligned on this path)
        // (W % 4 == 0 on this path; the eight 16-byte loads are all in flight at once)
        const int nw = min(a.W, 32);
        const uint4* m = reinterpret_cast<const uint4*>(a.bitmask + rs.row0 * (int64_t)a.W);
        uint4 u[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) u[i] = (4 * i < nw) ? __ldg(m + i) : make_uint4(0u, 0u, 0u, 0u);
        int ones = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) ones += __popc(u[i].x) + __popc(u[i].y) + __popc(u[i].z) + __popc(u[i].w);
        sparse = 2 * ones < nw * 32;
    }
    constexpr float es = (float)sizeof(ET);
    // a sparse row gathers a fraction of the bytes but is a chain of dependent steps (mask scan,
    // list, gathers, fold, reduce): in time it costs about 0.65 of a dense row
    const float row = sparse ? 0.65f : 1.f;
    // expected rows by kind: a draft model's drafts are mostly accepted (q close to p); a sampled
    // model-free draft is accepted with probability p(x), usually small, so such a request is
    // about one race row over logits + noise; a greedy draft only when it is the argmax
    float rows;
    if (greedy) rows = 1.f + 0.3f * (float)rs.k;
    else if (qmode) rows = 1.f + 0.6f * (float)rs.k;
    else rows = sparse ? 1.f : 0.85f * (es + 4.f) / es;
    float cost = rows * row;
    // a top-k / top-p request streams each row once more per digit of each threshold search
    const Filter f = request_filter(a, b);
    if (f.on) cost *= 1.f + (float)(((f.k > 0) + (f.p < 1.f)) * (sizeof(ET) == 2 ? 2 : 4));
    // a rejected draft-model row: a second pass over logits, noise and q
    if (!greedy && qmode) cost += sparse ? 0.7f : 0.85f * (es + 8.f) / es;
    return min(kSchedKeys - 1, (int)(cost * 16.f + 0.5f));
}

constexpr int kSchedSmemKeys = 8192;               // batches up to this size keep their keys on chip

struct SchedShared {
    int32_t cursor[kSchedKeys];                   // next output slot per key
    int32_t wcnt[kSchedWarps][kSchedKeys];        // requests per (warp, key) in the current tile
    uint8_t keys[kSchedSmemKeys];
};

// order[B]: the permutation; keys[B]: each request's cost key (read back here only when
// B > kSchedSmemKeys; smaller batches keep a copy on chip).
template <typename ET>
__global__ void __launch_bounds__(kSchedThreads) specdec_schedule_kernel(const Args a, int32_t* order, uint8_t* keys)
{
    __shared__ SchedShared sh;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int B = a.B;
    allow_dependent_launch();          // the verify grid may start; it waits for this grid to finish
    uint8_t* kp = B <= kSchedSmemKeys ? sh.keys : keys;

    for (int i = tid; i < kSchedKeys; i += kSchedThreads) sh.cursor[i] = 0;
    __syncthreads();
    // pass 1: keys and their histogram (one shared-memory atomic per distinct key in a warp)
    for (int b0 = 0; b0 < B; b0 += kSchedThreads) {
        const int b = b0 + tid;
        const int key = b < B ? request_cost_key<ET>(a, b) : -1;
        if (b < B) {
            keys[b] = (uint8_t)key;                        // kept in the workspace for inspection
            if (kp != keys) kp[b] = (uint8_t)key;
        }
        const unsigned peers = __match_any_sync(0xffffffffu, key);
        if (key >= 0 && lane == __ffs(peers) - 1) atomicAdd(&sh.cursor[key], __popc(peers));
    }
    __syncthreads();
    // exclusive prefix over keys in descending order: first slot of each key (warp 0, 8 keys a lane)
    if (warp == 0) {
        int v[kSchedKeys / 32], sum = 0;
#pragma unroll
        for (int e = 0; e < kSchedKeys / 32; ++e) { v[e] = sh.cursor[kSchedKeys - 1 - (lane * 8 + e)]; sum += v[e]; }
        int incl = sum;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += y;
        }
        int run = incl - sum;
#pragma unroll
        for (int e = 0; e < kSchedKeys / 32; ++e) { sh.cursor[kSchedKeys - 1 - (lane * 8 + e)] = run; run += v[e]; }
    }
    __syncthreads();
    // pass 2: stable placement, one tile of kSchedThreads requests at a time in index order
    const unsigned lt = (1u << lane) - 1u;
    for (int t0 = 0; t0 < B; t0 += kSchedThreads) {
        for (int i = tid; i < kSchedWarps * kSchedKeys; i += kSchedThreads) (&sh.wcnt[0][0])[i] = 0;
        __syncthreads();
        const int b = t0 + tid;
        const int key = b < B ? (int)kp[b] : -1;
        const unsigned peers = __match_any_sync(0xffffffffu, key);
        if (key >= 0 && (peers & lt) == 0u) sh.wcnt[warp][key] = __popc(peers);
        __syncthreads();
        if (key >= 0) {
            int pos = sh.cursor[key] + __popc(peers & lt);
            for (int w = 0; w < warp; ++w) pos += sh.wcnt[w][key];
            order[pos] = b;
        }
        __syncthreads();
        for (int k2 = tid; k2 < kSchedKeys; k2 += kSchedThreads) {
            int add = 0;
            for (int w = 0; w < kSchedWarps; ++w) add += sh.wcnt[w][k2];
            sh.cursor[k2] += add;
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------------------

struct LaunchShape {
    int stream;             // 1: streaming kernel (ring per CTA); 0: slice-resident cluster kernel
    int G, slice_units, smem, threads;
};

int device_sms()
{
    static int sms = -1;
    if (sms < 0) {
        int dev = 0, n = 0;
        if (cudaGetDevice(&dev) == cudaSuccess && cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && n > 0)
            sms = n;
        else {
            (void)cudaGetLastError();
            sms = 152;      // no device visible: assume a GB300
        }
    }
    return sms;
}

// CTAs per request for the streaming kernel. A request is a serial chain of row passes and
// one CTA streams at about its fair share of HBM (~1/300 of it with two CTAs per SM), so a batch
// far smaller than one wave of resident CTAs splits each row over as many CTAs as still fit in
// that wave (3 or 4); otherwise one CTA per request (the per-row exchange of a cluster of two
// costs about what the shorter chain gains). Measured on GB300: B=64 -> 3 or 4 (4 CTAs 24.6 us,
// 2 CTAs 25.6, 1 CTA 28.7); B=128 -> 1 (78 us vs 83 with 2); B >= 256 -> 1.
int stream_ctas_per_request(int32_t B, int sms)
{
    const int b = B > 0 ? B : 1;
    int G = (kResidentPerSM * sms) / b;
    if (G < 3) G = 1;
    if (G > 4) G = 4;
    return G;
}

// Launch choices forced for comparison and test runs (-1: the library decides). Initialised once
// per process from SPECDEC_KERNEL (=cluster: the slice-resident cluster kernel, kept as an
// independent decomposition of the same computation that parity runs cross-check the streaming
// kernel against), SPECDEC_CTAS_PER_REQUEST and SPECDEC_SCHEDULE; specdec_set_launch_options
// changes them afterwards. No call reads the environment.
struct LaunchOptions {
    std::atomic<int> kernel{-1};       // 0 streaming, 1 slice-resident cluster kernel
    std::atomic<int> ctas{-1};         // CTAs per request, 1..kMaxCluster
    std::atomic<int> schedule{-1};     // 0 off, 1 on (with a workspace)
    std::atomic<long long> wait_us{-1};  // limit of each wait in the streaming kernel (-1: 2 s)
    std::atomic<int> split{-1};        // requests split over a cluster of 2 (-1: automatic)
};

LaunchOptions& launch_options()
{
    static LaunchOptions* o = [] {
        LaunchOptions* d = new LaunchOptions;
        if (const char* e = std::getenv("SPECDEC_KERNEL")) d->kernel = std::strcmp(e, "cluster") == 0 ? 1 : 0;
        if (const char* e = std::getenv("SPECDEC_CTAS_PER_REQUEST")) {
            const long long v = std::atoll(e);
            if (v >= 1) d->ctas = (int)(v > kMaxCluster ? kMaxCluster : v);
        }
        if (const char* e = std::getenv("SPECDEC_SCHEDULE")) d->schedule = std::strcmp(e, "0") != 0 ? 1 : 0;
        return d;
    }();
    return *o;
}

specdec_status_t shape_for(int32_t V, specdec_dtype_t dt, int32_t B, LaunchShape* out)
{
    if (V <= 0 || B < 0) return SPECDEC_ERR_INVALID_ARG;
    if (dt != SPECDEC_F32 && dt != SPECDEC_BF16) return SPECDEC_ERR_UNSUPPORTED;
    const int es = dt == SPECDEC_F32 ? 4 : 2;
    const long long units = ((long long)V + kUnit - 1) / kUnit;
    const bool cluster = launch_options().kernel.load() == 1;
    long long G;
    if (cluster) {
        const long long row_bytes = (long long)V * es;
        G = (row_bytes + kTargetSliceBytes - 1) / kTargetSliceBytes;
    } else {
        G = stream_ctas_per_request(B, device_sms());
    }
    const int forced = launch_options().ctas.load();
    if (forced >= 1) G = forced;
    if (G < 1) G = 1;
    if (G > kMaxCluster) G = kMaxCluster;
    if (G > units) G = units;
    const long long su = (units + G - 1) / G;
    G = (units + su - 1) / su;                      // no CTA with an empty slice
    out->G = (int)G;
    out->slice_units = (int)su;
    if (!cluster) {
        out->stream = 1;
        out->smem = kRingBytes;
        out->threads = kStreamThreads;
        return SPECDEC_OK;
    }
    const long long slice_bytes = su * kUnit * es;
    if (slice_bytes > kMaxSliceBytes) return SPECDEC_ERR_UNSUPPORTED;
    out->stream = 0;
    out->smem = (int)(slice_bytes + su * (kUnit / 32) * 4);
    out->threads = kThreads;
    return SPECDEC_OK;
}

template <typename ET>
cudaError_t configure_kernel_once()
{
    static std::once_flag once;
    static cudaError_t err = cudaSuccess;
    std::call_once(once, [] {
        err = cudaFuncSetAttribute(specdec_verify_kernel<ET>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   kMaxSliceBytes + kMaxSliceBytes / 32 + 1024);
        if (err == cudaSuccess)
            err = cudaFuncSetAttribute(specdec_verify_kernel<ET>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (err == cudaSuccess)
            err = cudaFuncSetAttribute(specdec_verify_stream_kernel<ET, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kRingBytes);
        if (err == cudaSuccess)
            err = cudaFuncSetAttribute(specdec_verify_stream_kernel<ET, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kRingBytes);
        if (err == cudaSuccess)
            err = cudaFuncSetAttribute(specdec_verify_stream_kernel<ET, false>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (err == cudaSuccess)
            err = cudaFuncSetAttribute(specdec_verify_stream_kernel<ET, true>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    });
    return err;
}

// Largest cluster size <= G that the device can co-schedule for this kernel and shared memory.
int schedulable_cluster(void (*kernel)(Args), int G, int smem, int threads, cudaStream_t stream)
{
    for (; G > 1; --G) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)G, 1, 1);
        cfg.blockDim = dim3((unsigned)threads, 1, 1);
        cfg.dynamicSmemBytes = (size_t)smem;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)G;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) == cudaSuccess && n > 0) return G;
        (void)cudaGetLastError();
    }
    return 1;
}

template <typename ET>
specdec_status_t launch(Args args, LaunchShape sh, int32_t clusters, cudaStream_t stream, bool after_schedule)
{
    if (configure_kernel_once<ET>() != cudaSuccess) return SPECDEC_ERR_CUDA;
    void (*kernel)(Args) = !sh.stream ? specdec_verify_kernel<ET>
                           : (args.top_k || args.top_p) ? specdec_verify_stream_kernel<ET, true>
                                                        : specdec_verify_stream_kernel<ET, false>;
    if (sh.G > 1) {
        // the cluster size actually used, cached per (kernel, G, smem) request
        static std::mutex mu;
        static void (*cached_kernel)(Args) = nullptr;
        static int cached_req = -1, cached_smem = -1, cached_G = -1;
        std::lock_guard<std::mutex> lock(mu);
        if (cached_kernel != kernel || cached_req != sh.G || cached_smem != sh.smem) {
            cached_G = schedulable_cluster(kernel, sh.G, sh.smem, sh.threads, stream);
            cached_kernel = kernel;
            cached_req = sh.G;
            cached_smem = sh.smem;
        }
        if (cached_G != sh.G) {
            // re-slice the row over fewer CTAs; the cluster kernel gives up if a slice no longer fits
            const int es = (int)sizeof(ET);
            const long long units = ((long long)args.V + kUnit - 1) / kUnit;
            const long long su = (units + cached_G - 1) / cached_G;
            if (!sh.stream && su * kUnit * es > kMaxSliceBytes) return SPECDEC_ERR_UNSUPPORTED;
            sh.G = (int)((units + su - 1) / su);
            sh.slice_units = (int)su;
            if (!sh.stream) sh.smem = (int)(su * kUnit * es + su * (kUnit / 32) * 4);
            args.G = sh.G;
            args.slice_units = sh.slice_units;
            if (args.split_n > 0) {
                // no cluster of 2 fits: one CTA per request, in the same order
                clusters = args.B;
                args.split_n = 0;
            }
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)clusters * (unsigned)sh.G, 1, 1);
    cfg.blockDim = dim3((unsigned)sh.threads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)sh.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)sh.G;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = after_schedule ? 2 : 1;
    cudaError_t err = cudaLaunchKernelEx(&cfg, kernel, args);
    if (err != cudaSuccess) {
        (void)cudaGetLastError();
        return SPECDEC_ERR_CUDA;
    }
    return SPECDEC_OK;
}

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

inline size_t round16(size_t x) { return (x + 15) & ~(size_t)15; }

// How many of the heaviest requests a scheduled one-CTA-per-request launch splits over a cluster of
// 2 CTAs: automatically, when the batch exceeds one wave of resident CTAs, a sixth of that wave
// (their pairs of CTAs take a third of it; the rest starts the other requests). Measured on the
// large mixed batch (1024 requests, 304 resident CTAs): 0 -> 202.6 us, 32 -> 188.4, 48 -> 187.4,
// 64 -> 188.4, 96 -> 188.4, 128 -> 190.5. The launch options can force a number.
int32_t split_requests(int32_t B)
{
    if (launch_options().schedule.load() == 0) return 0;          // the split follows the schedule
    const int forced = launch_options().split.load();
    if (forced >= 0) return forced < B ? forced : B;
    const long long slots = (long long)kResidentPerSM * device_sms();
    if ((long long)B <= slots) return 0;
    return (int32_t)(slots / 6 < B ? slots / 6 : B);
}

// Whether a call with a workspace runs the schedule kernel first: only when the grid does not fit
// in one wave of resident CTAs (with everything resident at once the order changes nothing),
// unless the launch options force it on or off.
bool schedule_wanted(int32_t B, int G)
{
    const int forced = launch_options().schedule.load();
    if (forced >= 0) return forced == 1;
    return (long long)B * G > (long long)kResidentPerSM * device_sms();
}

// The schedule's scratch inside a caller workspace: order int32[B], then keys uint8[B].
struct ScheduleLayout {
    size_t order_off, keys_off, bytes;
};

ScheduleLayout schedule_layout(int32_t B)
{
    ScheduleLayout L;
    L.order_off = 0;
    L.keys_off = round16(sizeof(int32_t) * (size_t)B);
    L.bytes = round16(L.keys_off + (size_t)B);
    return L;
}

template <typename ET>
specdec_status_t launch_schedule(const Args& args, int32_t* order, uint8_t* keys, cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, 1, 1);
    cfg.blockDim = dim3(kSchedThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = nullptr;
    cfg.numAttrs = 0;
    if (cudaLaunchKernelEx(&cfg, specdec_schedule_kernel<ET>, args, order, keys) != cudaSuccess) {
        (void)cudaGetLastError();
        return SPECDEC_ERR_CUDA;
    }
    return SPECDEC_OK;
}

constexpr int kMaxDevices = 64;

}  // namespace

// Schedule scratch owned by the library, for specdec_verify_noalloc: the request order and cost
// keys of up to SPECDEC_NOALLOC_MAX_REQUESTS requests (80 KiB per device), laid out as in a
// caller workspace. Shared by every specdec_verify_noalloc call on a device.
constexpr size_t kNoallocScratchBytes = ((size_t)SPECDEC_NOALLOC_MAX_REQUESTS * 4 + 15) / 16 * 16 +
                                        ((size_t)SPECDEC_NOALLOC_MAX_REQUESTS + 15) / 16 * 16;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

namespace {

// The unique id of the calling thread's current context (0: none, or the driver entry points are
// unavailable). Ids are never reused within a process, unlike context handles, so a context
// created after cudaDeviceReset (or by the driver API) on the same ordinal has a new one.
unsigned long long current_context_id()
{
    using GetCurrent = int (*)(void**);
    using GetId = int (*)(void*, unsigned long long*);
    static GetCurrent get_current = nullptr;
    static GetId get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<GetCurrent>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<GetId>(p);
        (void)cudaGetLastError();
    });
    void* ctx = nullptr;
    unsigned long long id = 0;
    if (get_current && get_id && get_current(&ctx) == 0 && ctx != nullptr && get_id(ctx, &id) == 0) return id;
    return 0;
}

// Device address of g_noalloc_scratch on device `dev` (current), looked up with
// cudaGetSymbolAddress on the first call in each context and cached with that context's id.
void* noalloc_scratch(int dev)
{
    static std::mutex mu;
    static void* addr[kMaxDevices] = {};
    static unsigned long long ctx_of[kMaxDevices] = {};
    std::lock_guard<std::mutex> lock(mu);
    const unsigned long long ctx = current_context_id();
    if (addr[dev] == nullptr || ctx == 0 || ctx != ctx_of[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
            (void)cudaGetLastError();
            return nullptr;
        }
        addr[dev] = p;
        ctx_of[dev] = current_context_id();          // the lookup made the primary context current
    }
    return addr[dev];
}

}  // namespace

extern "C" specdec_status_t specdec_launch_config(int32_t B, int32_t V, specdec_dtype_t logits_dtype,
                                                  int32_t* ctas_per_request, int32_t* threads_per_cta,
                                                  int32_t* smem_bytes, int32_t* slice_ids,
                                                  int32_t* kernels_with_workspace, int32_t* split_requests_out)
{
    LaunchShape s;
    const specdec_status_t rc = shape_for(V, logits_dtype, B, &s);
    if (rc != SPECDEC_OK) return rc;
    const long long units = ((long long)V + kUnit - 1) / kUnit;
    const int32_t split = (B > 0 && s.stream && s.G == 1 && units >= 2) ? split_requests(B) : 0;
    if (ctas_per_request) *ctas_per_request = s.G;
    if (threads_per_cta) *threads_per_cta = s.threads;
    if (smem_bytes) *smem_bytes = s.smem;
    if (slice_ids) *slice_ids = s.slice_units * kUnit;
    if (kernels_with_workspace) *kernels_with_workspace = (B > 0 && (split > 0 || schedule_wanted(B, s.G))) ? 2 : 1;
    if (split_requests_out) *split_requests_out = split;
    return SPECDEC_OK;
}

extern "C" specdec_status_t specdec_verify(
    const void* target_logits, specdec_dtype_t logits_dtype, const int32_t* draft_ids,
    const float* draft_probs, const uint8_t* has_q, const int32_t* cu_num_draft, int32_t B, int32_t V,
    int32_t max_k, const int32_t* bitmask, const float* temperature, const int32_t* top_k, const float* top_p,
    const float* uniforms, const float* exp_noise, int32_t* out_tokens, int32_t* out_num_accepted,
    unsigned long long* counters, uint32_t* status, float* diag_accept_prob, float* diag_row_stats,
    unsigned long long* telemetry, void* workspace, size_t workspace_bytes, void* stream)
{
    if (logits_dtype != SPECDEC_F32 && logits_dtype != SPECDEC_BF16) return SPECDEC_ERR_UNSUPPORTED;
    if (B < 0 || V < 1 || max_k < 0 || max_k > SPECDEC_KMAX) return SPECDEC_ERR_INVALID_ARG;
    if (!target_logits || !cu_num_draft || !temperature || !uniforms || !exp_noise ||
        !out_tokens || !out_num_accepted || !counters)
        return SPECDEC_ERR_INVALID_ARG;
    const size_t es = logits_dtype == SPECDEC_F32 ? 4 : 2;
    if (!aligned(target_logits, es) || (draft_ids && !aligned(draft_ids, 4)) || (draft_probs && !aligned(draft_probs, 4)) ||
        !aligned(cu_num_draft, 4) || (bitmask && !aligned(bitmask, 4)) || !aligned(temperature, 4) ||
        !aligned(uniforms, 4) || !aligned(exp_noise, 4) || !aligned(out_tokens, 4) ||
        !aligned(out_num_accepted, 4) || !aligned(counters, 8) || (status && !aligned(status, 4)) ||
        (diag_accept_prob && !aligned(diag_accept_prob, 4)) || (diag_row_stats && !aligned(diag_row_stats, 4)) ||
        (telemetry && !aligned(telemetry, 8)) || (top_k && !aligned(top_k, 4)) || (top_p && !aligned(top_p, 4)))
        return SPECDEC_ERR_INVALID_ARG;
    LaunchShape shape;
    const specdec_status_t rc = shape_for(V, logits_dtype, B, &shape);
    if (rc != SPECDEC_OK) return rc;
    if (top_k || top_p) {
        // the threshold search reduces within one CTA: one CTA per request, streaming kernel only;
        // its 32-bit bin sums of 12-bit mass parts are exact up to 2^20 elements per row
        if (!shape.stream || V > (1 << 20)) return SPECDEC_ERR_UNSUPPORTED;
        const long long units = ((long long)V + kUnit - 1) / kUnit;
        shape.G = 1;
        shape.slice_units = (int)units;
    }
    if (B == 0) return SPECDEC_OK;
    if ((long long)B * shape.G > INT_MAX) return SPECDEC_ERR_UNSUPPORTED;

    Args a;
    a.logits = target_logits;
    a.draft_ids = draft_ids;
    a.q = draft_probs;
    a.has_q = has_q;
    a.cu = cu_num_draft;
    a.bitmask = bitmask;
    a.temperature = temperature;
    a.top_k = top_k;
    a.top_p = top_p;
    a.uniforms = uniforms;
    a.noise = exp_noise;
    a.out_tokens = out_tokens;
    a.out_num_accepted = out_num_accepted;
    a.counters = counters;
    a.status = status;
    a.diag_alpha = diag_accept_prob;
    a.diag_row = diag_row_stats;
    a.telemetry = telemetry;
    a.B = B;
    a.V = V;
    a.max_k = max_k;
    a.W = (V + 31) / 32;
    a.slice_units = shape.slice_units;
    a.G = shape.G;
    // bulk async copies need 16-byte aligned rows: row pitch and base of logits and bitmask
    // (the streaming kernel also bulk-copies noise and q rows: their bases must be aligned too)
    a.bulk = aligned(target_logits, 16) && ((size_t)V * es) % 16 == 0 &&
             (!bitmask || (aligned(bitmask, 16) && a.W % 4 == 0)) && aligned(exp_noise, 16) &&
             (!draft_probs || aligned(draft_probs, 16));
    a.vec_noise = aligned(exp_noise, 16) && V % 4 == 0 && (!draft_probs || aligned(draft_probs, 16));
    a.order = nullptr;
    a.split_n = 0;
    const long long wait_us = launch_options().wait_us.load();
    a.wait_ns = wait_us < 0 ? kWaitLimitNs : (unsigned long long)wait_us * 1000ull;
    const cudaStream_t st = (cudaStream_t)stream;
    if (workspace != nullptr) {
        const ScheduleLayout L = schedule_layout(B);
        if (!aligned(workspace, 16) || workspace_bytes < L.bytes) return SPECDEC_ERR_INVALID_ARG;
    }
    // A batch of more requests than resident CTAs, one CTA per request, scheduled: the chains of
    // the heaviest requests set the launch's length (they run at one CTA's share of HBM while the
    // rest fill in behind), so the first split_n requests of the order are split over a cluster
    // of 2 CTAs and the rest run two per cluster, one per CTA (split_requests()).
    int32_t clusters = B;
    const int32_t split = (workspace != nullptr && shape.stream && shape.G == 1 && !top_k && !top_p)
                              ? split_requests(B) : 0;
    if (split > 0) {
        const long long units = ((long long)V + kUnit - 1) / kUnit;
        const long long su = (units + 1) / 2;
        if ((units + su - 1) / su == 2) {                 // both CTAs own a non-empty half of every row
            shape.G = 2;
            shape.slice_units = (int)su;
            a.G = 2;
            a.slice_units = (int)su;
            a.split_n = split;
            clusters = split + (B - split + 1) / 2;
        }
    }
    // heaviest requests first: the schedule kernel writes the order the verify kernel reads
    if (workspace != nullptr && (a.split_n > 0 || schedule_wanted(B, shape.G))) {
        const ScheduleLayout L = schedule_layout(B);
        unsigned char* ws = static_cast<unsigned char*>(workspace);
        int32_t* order = reinterpret_cast<int32_t*>(ws + L.order_off);
        uint8_t* keys = ws + L.keys_off;
        const specdec_status_t rs = logits_dtype == SPECDEC_F32 ? launch_schedule<float>(a, order, keys, st)
                                                                : launch_schedule<uint16_t>(a, order, keys, st);
        if (rs != SPECDEC_OK) return rs;
        a.order = order;
    }
    const bool dep = a.order != nullptr;
    return logits_dtype == SPECDEC_F32 ? launch<float>(a, shape, clusters, st, dep)
                                       : launch<uint16_t>(a, shape, clusters, st, dep);
}

extern "C" specdec_status_t specdec_verify_noalloc(
    const void* target_logits, specdec_dtype_t logits_dtype, const int32_t* draft_ids,
    const float* draft_probs, const uint8_t* has_q, const int32_t* cu_num_draft, int32_t B, int32_t V,
    int32_t max_k, const int32_t* bitmask, const float* temperature, const int32_t* top_k, const float* top_p,
    const float* uniforms, const float* exp_noise, int32_t* out_tokens, int32_t* out_num_accepted,
    unsigned long long* counters, uint32_t* status, float* diag_accept_prob, float* diag_row_stats,
    unsigned long long* telemetry, void* stream)
{
    static_assert(kNoallocScratchBytes >= sizeof(int32_t) * SPECDEC_NOALLOC_MAX_REQUESTS + SPECDEC_NOALLOC_MAX_REQUESTS,
                  "scratch holds the order and the keys");
    if (B > SPECDEC_NOALLOC_MAX_REQUESTS) return SPECDEC_ERR_UNSUPPORTED;     // before any CUDA call
    void* scratch = nullptr;
    if (B > 0) {
        int dev = -1;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
            (void)cudaGetLastError();
            return SPECDEC_ERR_CUDA;
        }
        scratch = noalloc_scratch(dev);
        if (scratch == nullptr) return SPECDEC_ERR_CUDA;
    }
    return specdec_verify(target_logits, logits_dtype, draft_ids, draft_probs, has_q, cu_num_draft, B, V, max_k,
                          bitmask, temperature, top_k, top_p, uniforms, exp_noise, out_tokens, out_num_accepted,
                          counters, status, diag_accept_prob, diag_row_stats, telemetry, scratch,
                          scratch ? kNoallocScratchBytes : 0, stream);
}

extern "C" specdec_status_t specdec_set_launch_options(int32_t kernel, int32_t ctas_per_request, int32_t schedule,
                                                       int32_t wait_limit_us, int32_t split_requests)
{
    if (kernel < -1 || kernel > 1 || schedule < -1 || schedule > 1 || ctas_per_request == 0 ||
        ctas_per_request < -1 || ctas_per_request > kMaxCluster || wait_limit_us < -1 ||
        wait_limit_us > 2000000 || split_requests < -1)
        return SPECDEC_ERR_INVALID_ARG;
    LaunchOptions& o = launch_options();
    o.kernel = kernel;
    o.ctas = ctas_per_request;
    o.schedule = schedule;
    o.wait_us = wait_limit_us;
    o.split = split_requests;
    return SPECDEC_OK;
}

extern "C" size_t specdec_workspace_size(int32_t B, int32_t V)
{
    if (B <= 0 || V <= 0) return 0;
    return schedule_layout(B).bytes;
}

extern "C" specdec_status_t specdec_wait(void* stream, int32_t timeout_ms)
{
    const cudaStream_t s = (cudaStream_t)stream;
    if (timeout_ms < 0) return cudaStreamSynchronize(s) == cudaSuccess ? SPECDEC_OK : SPECDEC_ERR_CUDA;
    // poll with a host-side deadline (steady clock via CUDA events is not needed here)
    struct timespec t0;
    clock_gettime(CLOCK_MONOTONIC, &t0);
    while (true) {
        const cudaError_t e = cudaStreamQuery(s);
        if (e == cudaSuccess) return SPECDEC_OK;
        if (e != cudaErrorNotReady) return SPECDEC_ERR_CUDA;
        struct timespec t1;
        clock_gettime(CLOCK_MONOTONIC, &t1);
        const long long ms = (t1.tv_sec - t0.tv_sec) * 1000LL + (t1.tv_nsec - t0.tv_nsec) / 1000000LL;
        if (ms >= timeout_ms) return SPECDEC_ERR_TIMEOUT;
        struct timespec nap = {0, 50000};
        nanosleep(&nap, nullptr);
    }
}

extern "C" const char* specdec_status_string(specdec_status_t s)
{
    switch (s) {
    case SPECDEC_OK: return "SPECDEC_OK";
    case SPECDEC_ERR_INVALID_ARG: return "SPECDEC_ERR_INVALID_ARG";
    case SPECDEC_ERR_UNSUPPORTED: return "SPECDEC_ERR_UNSUPPORTED";
    case SPECDEC_ERR_CUDA: return "SPECDEC_ERR_CUDA";
    case SPECDEC_ERR_TIMEOUT: return "SPECDEC_ERR_TIMEOUT";
    }
    return "SPECDEC_UNKNOWN_STATUS";
}
