// K/V offload with the k-index kept on the GPU: fetch the selected pages on demand.
//
// "Together AI 解析如何高效服务 MiniMax M3…", section 未来工作: since only the top-k
// blocks are attended, the KV cache can sit in host memory while the (much
// smaller) k-index stays resident; the scan and the selection run on the GPU and
// only the selected KV pages are fetched.  On a Grace-Blackwell node the GPU
// reads pinned host memory directly over the chip-to-chip link, so the fetch is
// one gather kernel (zero copy) rather than a copy per page:
//   - one CTA per (decode row r = b*G + g, slot s) with a selected page: the
//     group-g slices (128 tokens x D) of K and V of host page pt[r][s] are read
//     with 16-byte loads and written to slot s of request b's pool page,
//     pool page b*topk + s, group slice g;
//   - the pool page table maps row r's slot s to that pool page (-1 stays -1),
//     so the ordinary decode attention runs on the pool unchanged.
// A pool page holds, per group, the slice of a different host page (each group
// selects its own blocks), which is all the attention of row (b, g) reads.
#include "msa_device.cuh"
#include "msa_internal.h"

namespace msa {
namespace {

constexpr int kThreads = 256;

template <int D>
__global__ void __launch_bounds__(kThreads) k_offload_gather(const uint4 *__restrict__ host_k,
                                                             const uint4 *__restrict__ host_v,
                                                             const int32_t *__restrict__ page_table, int B, int G,
                                                             int topk, int n_host_pages, uint4 *__restrict__ pool_k,
                                                             uint4 *__restrict__ pool_v,
                                                             int32_t *__restrict__ pool_page_table, int32_t *err) {
    constexpr int V16 = D * 2 / 16;                // 16-byte pieces of one token's group slice
    const int item = blockIdx.x;                   // (row, slot)
    const int r = item / topk, s = item - (item / topk) * topk;
    const int b = r / G, g = r - (r / G) * G;
    const int p = page_table[item];
    const int pool_page = b * topk + s;
    if (threadIdx.x == 0) pool_page_table[item] = p >= 0 ? pool_page : -1;
    if (p < 0) return;
    if (p >= n_host_pages) {
        if (threadIdx.x == 0) raise_flag(err, MSA_FLAG_BOUNDS);
        return;
    }
    // token t of group g of page x starts at ((x * 128 + t) * G + g) * V16 pieces
    const size_t src0 = (size_t(p) * 128 * G + g) * V16, dst0 = (size_t(pool_page) * 128 * G + g) * V16;
    constexpr int N = 128 * V16;                   // pieces of the slice
    constexpr int PER = N / kThreads;              // 8 (D = 128) or 4 (D = 64)
    static_assert(N % kThreads == 0, "whole pieces per thread");
    uint4 kv[PER], vv[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) {                // all loads first: host-link latency overlaps
        const int x = threadIdx.x + i * kThreads;
        const size_t off = size_t(x / V16) * G * V16 + (x % V16);
        kv[i] = host_k[src0 + off];
        vv[i] = host_v[src0 + off];
    }
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int x = threadIdx.x + i * kThreads;
        const size_t off = size_t(x / V16) * G * V16 + (x % V16);
        pool_k[dst0 + off] = kv[i];
        pool_v[dst0 + off] = vv[i];
    }
}

// A step's inputs staged from page-locked host memory by SM loads over the host link.
// A copy-engine transfer of a decode step's inputs (about 155 KB for 8 requests)
// carries a fixed cost of about 10 us on this link; a grid of 16-byte loads, each
// thread's loads issued before its stores, moves them in roughly one round trip.
constexpr int kStagePer = 4;   // 16-byte pieces per thread

__global__ void __launch_bounds__(kThreads) k_stage_from_host(const uint4 *__restrict__ src, uint4 *__restrict__ dst,
                                                              size_t n) {
    pdl_trigger();   // a decode step's scan may start launching; it waits for this kernel to complete
    const size_t base = size_t(blockIdx.x) * kThreads * kStagePer + threadIdx.x;
    uint4 v[kStagePer];
#pragma unroll
    for (int i = 0; i < kStagePer; ++i) {
        const size_t x = base + size_t(i) * kThreads;
        if (x < n) v[i] = src[x];
    }
#pragma unroll
    for (int i = 0; i < kStagePer; ++i) {
        const size_t x = base + size_t(i) * kThreads;
        if (x < n) dst[x] = v[i];
    }
}

}  // namespace

cudaError_t launch_stage_from_host(const void *src, void *dst, size_t bytes, cudaStream_t st) {
    const size_t n = bytes / 16;
    if (n == 0) return cudaSuccess;
    const size_t per_cta = size_t(kThreads) * kStagePer;
    const size_t grid = (n + per_cta - 1) / per_cta;
    if (grid > 0x7fffffffULL) return cudaErrorInvalidConfiguration;
    k_stage_from_host<<<unsigned(grid), kThreads, 0, st>>>(static_cast<const uint4 *>(src), static_cast<uint4 *>(dst),
                                                           n);
    return cudaGetLastError();
}

cudaError_t launch_offload_gather(const void *host_k, const void *host_v, const int32_t *page_table, int B,
                                  int n_host_pages, const Shape &s, void *pool_k, void *pool_v,
                                  int32_t *pool_page_table, int32_t *err, cudaStream_t st) {
    const long long items = 1LL * B * s.G * s.topk;
    if (items <= 0) return cudaSuccess;
    if (items > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
#define MSA_OG_CASE(DD)                                                                                        \
    if (s.D == DD) {                                                                                           \
        k_offload_gather<DD><<<unsigned(items), kThreads, 0, st>>>(                                            \
            static_cast<const uint4 *>(host_k), static_cast<const uint4 *>(host_v), page_table, B, s.G, s.topk,  \
            n_host_pages, static_cast<uint4 *>(pool_k), static_cast<uint4 *>(pool_v), pool_page_table, err);   \
        return cudaGetLastError();                                                                             \
    }
    MSA_OG_CASE(128) MSA_OG_CASE(64)
#undef MSA_OG_CASE
    return cudaErrorNotSupported;
}

}  // namespace msa
