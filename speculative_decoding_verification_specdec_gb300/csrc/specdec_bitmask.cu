/*
 * specdec_bitmask.cu -- the per-step grammar bitmask in batch order, built on the GPU from the
 * compacted masks the scheduler sends, for GB300 (sm_103a); C-ABI entry point in include/specdec.h.
 *
 * What it computes ("vLLM tour part 2", section "Grammar gates: structured output"): the scheduler
 * sends the masks of the constrained requests only, k_b + 1 rows each, in scheduler order; the
 * batch has its own order and per-request speculative offsets. Row t(b, j) = cu[b] + b + j of the
 * output takes the j-th compact row of request b when b is constrained, and all ones otherwise.
 *
 * GB300 mapping: one CTA per batch request b. Its threads find b's first listing i in the
 * scheduler order (a min-reduction over the list) and the compact offset of that listing
 * (a sum of k + 1 over the listings before it), then copy the request's rows -- or write all-ones
 * rows -- with 16-byte vector loads and streaming stores when the row pitch allows, word by word
 * otherwise. Pure data movement: bound by HBM (read the constrained rows, write every row).
 */
#include <cuda_runtime.h>
#include <stdint.h>

#include <climits>

#include "specdec.h"

namespace {

constexpr int kScatterThreads = 256;

__device__ __forceinline__ int block_reduce_min(int v, int* red)
{
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, off));
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    v = INT_MAX;
    for (int w = 0; w < kScatterThreads / 32; ++w) v = min(v, red[w]);
    return v;
}

__device__ __forceinline__ long long block_reduce_sum(long long v, long long* red)
{
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    v = 0;
    for (int w = 0; w < kScatterThreads / 32; ++w) v += red[w];
    return v;
}

__global__ void __launch_bounds__(kScatterThreads)
specdec_bitmask_scatter_kernel(const int32_t* __restrict__ compact, int64_t compact_rows,
                               const int32_t* __restrict__ constrained, int32_t n,
                               const int32_t* __restrict__ cu, int32_t B, int32_t W, int vec,
                               int32_t* __restrict__ bitmask)
{
    __shared__ int red_i[kScatterThreads / 32];
    __shared__ long long red_l[kScatterThreads / 32];
    const int b = blockIdx.x;
    const int tid = threadIdx.x;
    const int32_t ntot = cu[B];
    auto owned = [&](int r) -> int {                               // rows of request r, -1 if malformed
        const int32_t a0 = cu[r], a1 = cu[r + 1];
        return (cu[0] != 0 || a0 < 0 || a1 < a0 || a1 > ntot) ? -1 : a1 - a0 + 1;
    };
    const int nrows = owned(b);
    if (nrows < 0) return;                                         // malformed offsets: rows unknown
    const int k = nrows - 1;
    const int64_t t0 = (int64_t)cu[b] + b;

    // first listing of b in the scheduler order
    int first = INT_MAX;
    for (int i = tid; i < n; i += kScatterThreads)
        if (constrained[i] == b) { first = i; break; }
    first = block_reduce_min(first, red_i);

    int64_t off = -1;
    if (first != INT_MAX) {
        // rows owned by the listings before it: k + 1 each for an id inside [0, B)
        long long rows = 0;
        for (int i = tid; i < first; i += kScatterThreads) {
            const int bi = constrained[i];
            if (bi >= 0 && bi < B) rows += (long long)max(owned(bi), 0);
        }
        off = block_reduce_sum(rows, red_l);
    }

    // the request's rows as one flat range of (row, 16-byte group) items, kUnroll loads in flight
    // per thread before their stores (a load-then-store loop waits out one DRAM latency per item).
    // Item counts are 64-bit: k comes from the caller's offsets and is not bounded. The first
    // copy_items items are copied, the rest of a listed request's items (rows past the end of the
    // compact array) are zeroed; an unlisted request's rows are all ones.
    const int64_t rows_left = off < 0 ? 0 : max((int64_t)0, min(compact_rows - off, (int64_t)k + 1));
    if (vec) {
        const int64_t n4 = W >> 2;
        const int64_t items = ((int64_t)k + 1) * n4;
        const int64_t copy_items = rows_left * n4;
        int4* d4 = reinterpret_cast<int4*>(bitmask + t0 * (int64_t)W);
        const int4* s4 = off >= 0 ? reinterpret_cast<const int4*>(compact + off * (int64_t)W) : nullptr;
        constexpr int kUnroll = 8;
        for (int64_t base = tid; base < items; base += (int64_t)kScatterThreads * kUnroll) {
            int4 v[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int64_t it = base + (int64_t)u * kScatterThreads;
                if (it < items && off >= 0 && it < copy_items) v[u] = __ldcs(s4 + it);
                else v[u] = off < 0 ? make_int4(-1, -1, -1, -1) : make_int4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int64_t it = base + (int64_t)u * kScatterThreads;
                if (it < items) __stcs(d4 + it, v[u]);
            }
        }
    } else {
        const int64_t items = ((int64_t)k + 1) * W;
        const int64_t copy_items = rows_left * W;
        int32_t* dst = bitmask + t0 * (int64_t)W;
        const int32_t* src = off >= 0 ? compact + off * (int64_t)W : nullptr;
        for (int64_t it = tid; it < items; it += kScatterThreads)
            dst[it] = off < 0 ? -1 : (it < copy_items ? src[it] : 0);
    }
}

}  // namespace

extern "C" specdec_status_t specdec_bitmask_scatter(const int32_t* compact, int64_t compact_rows,
                                                    const int32_t* constrained, int32_t n,
                                                    const int32_t* cu_num_draft, int32_t B, int32_t V,
                                                    int32_t* bitmask, void* stream)
{
    if (B < 0 || V < 1 || n < 0 || compact_rows < 0) return SPECDEC_ERR_INVALID_ARG;
    if (V > (1 << 26)) return SPECDEC_ERR_UNSUPPORTED;
    if (B == 0) return SPECDEC_OK;
    if (!cu_num_draft || !bitmask || (n > 0 && !constrained) || (compact_rows > 0 && !compact))
        return SPECDEC_ERR_INVALID_ARG;
    auto misaligned = [](const void* p, size_t a) { return p && (reinterpret_cast<uintptr_t>(p) % a) != 0; };
    if (misaligned(compact, 4) || misaligned(constrained, 4) || misaligned(cu_num_draft, 4) || misaligned(bitmask, 4))
        return SPECDEC_ERR_INVALID_ARG;
    const int32_t W = (V + 31) / 32;
    const bool vec = (W % 4 == 0) && !misaligned(bitmask, 16) && (!compact || !misaligned(compact, 16));
    specdec_bitmask_scatter_kernel<<<(unsigned)B, kScatterThreads, 0, (cudaStream_t)stream>>>(
        compact, compact_rows, constrained, n, cu_num_draft, B, W, vec ? 1 : 0, bitmask);
    if (cudaGetLastError() != cudaSuccess) return SPECDEC_ERR_CUDA;
    return SPECDEC_OK;
}
