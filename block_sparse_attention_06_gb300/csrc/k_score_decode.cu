// Decode index scoring: one CTA streams one 128-token k-index page for all KV
// groups of one query row and reduces it to one max score per group.
//
// "Together AI 解析如何高效服务 MiniMax M3…", section 解码索引评分内核优化: every
// decode query compares its query-side index vector with all candidate key-side
// index vectors and reduces each 128-token KV block to one score; the scan sits
// on the critical path of every generated token and grows with the context.
// The page's own kernel used AB-swapped HMMA tiles; here the scan is treated as
// what it is on GB300 -- a pure HBM stream (about 2 flop per byte) -- so the
// kernel issues fully coalesced 16-byte non-caching loads with eight loads in
// flight per thread and reduces with warp shuffles, leaving the tensor cores idle.
#include "msa_device.cuh"
#include "msa_internal.h"

namespace msa {
namespace {

template <int G, int DI>
__global__ void __launch_bounds__(256) k_score_decode(
    const uint16_t *__restrict__ q_idx, const uint8_t *__restrict__ kidx,
    const int32_t *__restrict__ block_table, const int32_t *__restrict__ q_req,
    const int32_t *__restrict__ q_pos, const int32_t *__restrict__ seq_lens, int n_req, int n_pages,
    int max_blocks, float *__restrict__ scores, int32_t *err) {
    constexpr int SUBS = DI / 8;             // 16-byte chunks per (token, group)
    constexpr int CPT = G * SUBS;            // chunks per token
    constexpr int TPP = 256 / CPT;           // tokens per pass of the CTA
    constexpr int PASSES = 128 / TPP;
    constexpr int UNROLL = PASSES < 8 ? PASSES : 8;
    constexpr size_t PAGE_BYTES = size_t(128) * G * DI * 2;
    static_assert(256 % CPT == 0 && PASSES % UNROLL == 0, "unsupported (G, Di)");

    const int r = blockIdx.x / max_blocks;
    const int j = blockIdx.x - r * max_blocks;
    const int tid = threadIdx.x;
    float *out = scores + size_t(r) * G * max_blocks + j;

    // In a decode step the scan may be a programmatic dependent of the kernel that staged its
    // inputs: nothing is read before that kernel completes.  Launched plainly, this returns at once.
    pdl_wait();
    pdl_trigger();   // the selection kernel may start launching once every scan CTA runs

    // rows are either (q_req, q_pos) pairs or the requests themselves at seq_lens - 1
    const int p = q_pos ? q_pos[r] : seq_lens[r] - 1;
    const int req = q_req ? q_req[r] : r;
    if (p < 0 || req < 0 || req >= n_req || (p >> 7) >= max_blocks) {
        if (tid < G) out[size_t(tid) * max_blocks] = -INFINITY;
        if (tid == 0 && j == 0) raise_flag(err, MSA_FLAG_BOUNDS);
        return;
    }
    if (j > (p >> 7)) {                       // not a candidate of this row
        if (tid < G) out[size_t(tid) * max_blocks] = -INFINITY;
        return;
    }
    const int page = block_table[size_t(req) * max_blocks + j];
    if (page < 0 || page >= n_pages) {
        if (tid < G) out[size_t(tid) * max_blocks] = -INFINITY;
        if (tid == 0) raise_flag(err, MSA_FLAG_BOUNDS);
        return;
    }

    const int sub = tid % SUBS;
    const int g = (tid / SUBS) % G;
    const uint4 qw = *reinterpret_cast<const uint4 *>(q_idx + (size_t(r) * G + g) * DI + sub * 8);
    const float q0 = bf16_lo(qw.x), q1 = bf16_hi(qw.x), q2 = bf16_lo(qw.y), q3 = bf16_hi(qw.y);
    const float q4 = bf16_lo(qw.z), q5 = bf16_hi(qw.z), q6 = bf16_lo(qw.w), q7 = bf16_hi(qw.w);

    const uint8_t *base = kidx + size_t(page) * PAGE_BYTES + size_t(tid) * 16;
    const int lim = p - j * 128;              // tokens t <= lim are visible
    const int t0 = tid / CPT;
    float best = -INFINITY;

#pragma unroll
    for (int m0 = 0; m0 < PASSES; m0 += UNROLL) {
        uint4 v[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) v[u] = ldg_stream_v4(base + size_t(m0 + u) * 4096);
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            float d = q0 * bf16_lo(v[u].x);
            d = fmaf(q1, bf16_hi(v[u].x), d);
            d = fmaf(q2, bf16_lo(v[u].y), d);
            d = fmaf(q3, bf16_hi(v[u].y), d);
            d = fmaf(q4, bf16_lo(v[u].z), d);
            d = fmaf(q5, bf16_hi(v[u].z), d);
            d = fmaf(q6, bf16_lo(v[u].w), d);
            d = fmaf(q7, bf16_hi(v[u].w), d);
#pragma unroll
            for (int o = 1; o < SUBS; o <<= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
            const int t = t0 + (m0 + u) * TPP;
            if (t <= lim) best = fmaxf(best, d);
        }
    }

    __shared__ float red[256 / SUBS];
    if (sub == 0) red[tid / SUBS] = best;
    __syncthreads();
    if (tid < G) {
        float b = -INFINITY;
        for (int e = tid; e < 256 / SUBS; e += G) b = fmaxf(b, red[e]);
        out[size_t(tid) * max_blocks] = b;
    }
}

template <int G, int DI>
cudaError_t launch_g(const void *q_idx, const void *kidx, const int32_t *bt, const int32_t *q_req,
                     const int32_t *q_pos, const int32_t *seq_lens, int n_rows, int n_req, int n_pages,
                     int max_blocks, float *scores, int32_t *err, cudaStream_t st, bool pdl) {
    const long long grid = 1LL * n_rows * max_blocks;
    if (grid <= 0) return cudaSuccess;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    return launch_kernel(k_score_decode<G, DI>, dim3(unsigned(grid)), dim3(256), 0, st, pdl,
                         static_cast<const uint16_t *>(q_idx), static_cast<const uint8_t *>(kidx), bt, q_req, q_pos,
                         seq_lens, n_req, n_pages, max_blocks, scores, err);
}

}  // namespace

static cudaError_t launch_any(const void *q_idx, const void *kidx, const int32_t *block_table, const int32_t *q_req,
                              const int32_t *q_pos, const int32_t *seq_lens, int n_rows, int n_req, int n_pages,
                              const Shape &s, float *scores, int32_t *err, cudaStream_t st, bool pdl) {
#define MSA_SD_CASE(GG, DD)                                                                               \
    if (s.G == GG && s.Di == DD)                                                                          \
        return launch_g<GG, DD>(q_idx, kidx, block_table, q_req, q_pos, seq_lens, n_rows, n_req, n_pages, \
                                s.max_blocks, scores, err, st, pdl);
    MSA_SD_CASE(1, 32) MSA_SD_CASE(1, 64) MSA_SD_CASE(2, 32) MSA_SD_CASE(2, 64)
    MSA_SD_CASE(4, 32) MSA_SD_CASE(4, 64) MSA_SD_CASE(8, 32) MSA_SD_CASE(8, 64)
    MSA_SD_CASE(16, 32) MSA_SD_CASE(16, 64)
#undef MSA_SD_CASE
    return cudaErrorNotSupported;
}

cudaError_t launch_score_decode(const void *q_idx, const void *kidx, const int32_t *block_table,
                                const int32_t *q_req, const int32_t *q_pos, int n_rows, int n_req,
                                int n_pages, const Shape &s, float *scores, int32_t *err,
                                cudaStream_t st) {
    return launch_any(q_idx, kidx, block_table, q_req, q_pos, nullptr, n_rows, n_req, n_pages, s, scores, err, st,
                      false);
}

cudaError_t launch_score_decode_seq(const void *q_idx, const void *kidx, const int32_t *block_table,
                                    const int32_t *seq_lens, int B, int n_pages, const Shape &s,
                                    float *scores, int32_t *err, cudaStream_t st, bool pdl) {
    return launch_any(q_idx, kidx, block_table, nullptr, nullptr, seq_lens, B, B, n_pages, s, scores, err, st, pdl);
}

}  // namespace msa
