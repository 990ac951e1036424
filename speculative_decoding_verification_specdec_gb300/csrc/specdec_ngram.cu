/*
 * specdec_ngram.cu -- batched n-gram proposer (the model-free drafter that feeds the verify) for
 * GB300 (sm_103a), and its C-ABI entry point declared in include/specdec.h.
 *
 * What it computes ("5.2 Draft models and model-free methods", infra-guide, sections 4.1 and 6):
 * for each request's token history h of length L, the longest window length n in
 * [min_n, min(max_n, L - 1)] whose last-n tail also occurs earlier in h (the tail itself
 * excluded), at its earliest start; the proposal is the (up to) k tokens after that occurrence.
 *
 * GB300 mapping: one CTA per request. Every position e in [0, L - 2] is the end of a candidate
 * window; M(e) is the length of the common suffix of h[.. e] and h[.. L - 1], capped at
 * min(max_n, L - 1). A window of length n ending at e equals the tail iff M(e) >= n, so the rule
 * picks n* = max over e of M(e) (when >= min_n) and, among the ends with M(e) = n*, the smallest
 * (the earliest start e - n* + 1). The history goes through shared memory in tiles of 8192 window
 * ends plus the 64 tokens before each tile, copied with cp.async so that every load of a tile is
 * in flight at once (comparing straight from global memory left each thread waiting on one load
 * after another); threads then take ends strided across the tile and the CTA reduces the packed
 * key (M, -e) to its maximum. Nothing here is a contraction; the history is read once, so the
 * kernel is bound by HBM bandwidth and, for short histories, by launch latency.
 */
#include <cuda_runtime.h>
#include <stdint.h>

#include "specdec.h"

namespace {

constexpr int kNgramThreads = 256;
constexpr int kTile = 4096;                    // window ends per shared-memory tile (16 KB: 8 CTAs per SM)
constexpr int kHalo = SPECDEC_NGRAM_MAX_N;     // tokens before a tile that its windows may reach
constexpr int kSmemBytes = (kHalo + kTile) * 4;

__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" :: "r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all()
{
    asm volatile("cp.async.wait_all;" ::: "memory");
}

__global__ void __launch_bounds__(kNgramThreads)
specdec_ngram_kernel(const int32_t* __restrict__ tokens, const int64_t* __restrict__ cu_hist, int min_n,
                     int max_n, int k, int32_t* __restrict__ out_drafts, int32_t* __restrict__ out_num,
                     int32_t* __restrict__ out_match)
{
    extern __shared__ __align__(16) int32_t buf[];   // [kHalo + kTile]: h[p0 - kHalo, p0 + kTile)
    __shared__ int32_t tail[SPECDEC_NGRAM_MAX_N];
    __shared__ unsigned long long wbest[kNgramThreads / 32];
    const int b = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t h0 = cu_hist[b];
    int64_t L = cu_hist[b + 1] - h0;
    if (h0 < 0 || L < 0 || L > 0x7fffffffLL) L = 0;          // bad offsets: an empty history (a miss)
    const int32_t* h = tokens + (L > 0 ? h0 : 0);
    const int cap = (int)(L - 1 < (int64_t)max_n ? L - 1 : (int64_t)max_n);   // longest window tried

    if (tid < cap) tail[tid] = h[L - 1 - tid];                // tail[m] = h[L - 1 - m]
    unsigned long long best = 0ull;                           // (M << 32) | ~e; 0: no window
    if (cap >= min_n) {
        const uint32_t sbuf = static_cast<uint32_t>(__cvta_generic_to_shared(buf));
        // window ends e in [p0, p0 + kTile) of [0, L - 2], one tile at a time: the tile and the
        // kHalo tokens before it are copied to shared memory (all copies in flight at once)
        for (int64_t p0 = 0; p0 <= L - 2; p0 += kTile) {
            const int64_t lo = p0 - kHalo;
            const int64_t hi = (p0 + kTile < L - 1 ? p0 + kTile : L - 1);      // exclusive
            __syncthreads();                                  // the previous tile is no longer read
            for (int64_t i = (lo < 0 ? -lo : 0) + tid; i < hi - lo; i += kNgramThreads)
                cp_async4(sbuf + (uint32_t)i * 4u, h + lo + i);
            cp_async_wait_all();
            __syncthreads();
            // four consecutive ends per thread: one 16-byte load tests their last tokens against the
            // tail's last token, and only the (rare) ends that pass walk further back
            const int32_t last = tail[0];
            for (int64_t e4 = p0 + 4 * tid; e4 < hi; e4 += 4 * kNgramThreads) {
                const int4 v = *reinterpret_cast<const int4*>(buf + (e4 - lo));     // e4 - lo = 64 + 4 * j
                const int32_t vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int64_t e = e4 + q;
                    if (e >= hi || vv[q] != last) continue;
                    const int lim = (int)(e + 1 < (int64_t)cap ? e + 1 : (int64_t)cap);
                    const int32_t* he = buf + (e - lo);       // he[-m] = h[e - m]
                    int m = 1;
                    while (m < lim && he[-m] == tail[m]) ++m;
                    if (m >= min_n) {
                        const unsigned long long key = ((unsigned long long)m << 32) | (0xffffffffull - (unsigned long long)e);
                        best = best > key ? best : key;
                    }
                }
            }
        }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        const unsigned long long o = __shfl_xor_sync(0xffffffffu, best, off);
        best = best > o ? best : o;
    }
    __syncthreads();
    if (lane == 0) wbest[warp] = best;
    __syncthreads();
    if (warp == 0) {
        best = lane < kNgramThreads / 32 ? wbest[lane] : 0ull;
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) {
            const unsigned long long o = __shfl_xor_sync(0xffffffffu, best, off);
            best = best > o ? best : o;
        }
        if (lane == 0) wbest[0] = best;
    }
    __syncthreads();
    best = wbest[0];
    const int n = (int)(best >> 32);
    const int64_t e = n > 0 ? (int64_t)(0xffffffffull - (best & 0xffffffffull)) : -1;
    const int num = n > 0 ? (int)(L - 1 - e < (int64_t)k ? L - 1 - e : (int64_t)k) : 0;
    for (int j = tid; j < k; j += kNgramThreads) out_drafts[(int64_t)b * k + j] = j < num ? h[e + 1 + j] : -1;
    if (tid == 0) {
        out_num[b] = num;
        out_match[b] = n;
    }
}

}  // namespace

extern "C" specdec_status_t specdec_ngram_propose(const int32_t* tokens, const int64_t* cu_hist, int32_t B,
                                                  int32_t min_n, int32_t max_n, int32_t k, int32_t* out_drafts,
                                                  int32_t* out_num, int32_t* out_match, void* stream)
{
    if (B < 0 || min_n < 1 || max_n < 0 || k < 0 || k > SPECDEC_KMAX) return SPECDEC_ERR_INVALID_ARG;
    if (max_n > SPECDEC_NGRAM_MAX_N) return SPECDEC_ERR_UNSUPPORTED;
    if (B == 0) return SPECDEC_OK;
    if (!tokens || !cu_hist || !out_num || !out_match || (k > 0 && !out_drafts)) return SPECDEC_ERR_INVALID_ARG;
    auto misaligned = [](const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) != 0; };
    if (misaligned(tokens, 4) || misaligned(cu_hist, 8) || misaligned(out_num, 4) || misaligned(out_match, 4) ||
        (out_drafts && misaligned(out_drafts, 4)))
        return SPECDEC_ERR_INVALID_ARG;
    specdec_ngram_kernel<<<(unsigned)B, kNgramThreads, kSmemBytes, (cudaStream_t)stream>>>(
        tokens, cu_hist, min_n, max_n, k, out_drafts, out_num, out_match);
    if (cudaGetLastError() != cudaSuccess) return SPECDEC_ERR_CUDA;
    return SPECDEC_OK;
}
