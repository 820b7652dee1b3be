// Multi-token decode index scoring: the rows of one request share each page read.
//
// "Together AI 解析如何高效服务 MiniMax M3…", section 解码索引评分内核优化: the decode
// index-scoring kernel treats 128 key tokens of a page as the M side of a bf16
// tensor-core product and pads the few query rows of a request to a small N
// ("AB-swapped"), then reduces each 128-token block to one score per KV group.
// With one query row per request the scan is a pure HBM stream and the plain
// decode kernel (k_score_decode.cu) serves it.  With several rows per request
// (speculative or multi-token decode) that kernel would read every page once per
// row; this one reads it once per request:
//   - one CTA per (request, page); warp w scores KV group w (and w + 8);
//   - the warp stages its group's 128 x Di slice of the page in 32-token chunks
//     (16-byte cp.async, double-buffered, chunk columns XOR-swizzled so that
//     ldmatrix reads them without bank conflicts);
//   - m16n8k16 bf16 MMAs with tokens as M (ldmatrix fragments of the k-index) and
//     the request's rows as N (up to 16 rows in two n-tiles, q_idx fragments held
//     in registers for the whole page);
//   - the causal mask (token position <= the row's position) and the max over
//     the 128 tokens are taken on the fp32 accumulators; each block score is
//     written as in the single-row kernel, -inf past the row's own block.
// Rows must be grouped by request (q_req non-decreasing), with at most 16 rows
// per request.
#include "msa_device.cuh"
#include "msa_internal.h"

namespace msa {
namespace {

constexpr int kWarps = 8;
constexpr int kChunkTok = 32;        // tokens per staged chunk
constexpr int kMaxRows = 16;         // rows per request (two n-tiles of 8)

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Position of the 16-byte chunk q of token row i in a staged chunk: rows of DI bf16, chunk index
// XOR-swizzled so that the 8 rows an ldmatrix phase reads fall in 8 distinct bank groups.
template <int DI>
__device__ __forceinline__ uint32_t stage_off(int i, int q) {
    if constexpr (DI == 64) return uint32_t(i * 128 + ((q ^ (i & 7)) << 4));
    else return uint32_t(i * 64 + ((q ^ ((i >> 1) & 3)) << 4));
}

template <int DI>
__global__ void __launch_bounds__(kWarps * 32) k_score_decode_mt(
    const uint16_t *__restrict__ q_idx, const uint8_t *__restrict__ kidx, const int32_t *__restrict__ block_table,
    const int32_t *__restrict__ q_req, const int32_t *__restrict__ q_pos, int n_rows, int n_req, int n_pages, int G,
    int max_blocks, float *__restrict__ scores, int32_t *err) {
    constexpr int CH = DI / 8;                     // 16-byte chunks per token row
    constexpr int KS = DI / 16;                    // k-steps of 16
    constexpr int STAGE = kChunkTok * DI * 2;      // bytes of one staged chunk
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int s_lo, s_hi;
    const int b = blockIdx.x, j = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    if (tid == 0) {
        // rows of request b: q_req is non-decreasing, so they are [lower bound, upper bound)
        int lo = 0, hi = n_rows;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (q_req[mid] < b) lo = mid + 1; else hi = mid;
        }
        int lo2 = lo, hi2 = n_rows;
        while (lo2 < hi2) {
            const int mid = (lo2 + hi2) >> 1;
            if (q_req[mid] <= b) lo2 = mid + 1; else hi2 = mid;
        }
        s_lo = lo;
        s_hi = lo2;
        if (b == 0 && j == 0) {
            // one CTA checks the grouping the search relies on
            for (int r = 0; r < n_rows; ++r) {
                const int rq = q_req[r];
                if (rq < 0 || rq >= n_req) raise_flag(err, MSA_FLAG_BOUNDS);
                else if (r > 0 && rq < q_req[r - 1]) raise_flag(err, MSA_FLAG_UNSUPPORTED);
            }
        }
    }
    __syncthreads();
    const int row0 = s_lo, T = s_hi - s_lo;
    if (T <= 0) return;
    if (T > kMaxRows) {
        if (tid == 0 && j == 0) raise_flag(err, MSA_FLAG_UNSUPPORTED);
        return;
    }
    // own block of each row; a block past every row's own block scores -inf without a read
    int own_max = -1;
    for (int t = 0; t < T; ++t) own_max = max(own_max, q_pos[row0 + t] >> 7);
    if (j > own_max) {
        for (int i = tid; i < T * G; i += kWarps * 32)
            scores[(size_t(row0 + i / G) * G + (i % G)) * max_blocks + j] = -INFINITY;
        return;
    }
    const int page = block_table[size_t(b) * max_blocks + j];
    if (page < 0 || page >= n_pages) {
        if (tid == 0) raise_flag(err, MSA_FLAG_BOUNDS);
        return;
    }

    // this lane's accumulator columns: rows n = nt * 8 + (lane & 3) * 2 + e
    int pos[2][2];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int n = nt * 8 + (lane & 3) * 2 + e;
            pos[nt][e] = n < T ? q_pos[row0 + n] : -1;
        }
    const int NT = (T + 7) >> 3;
    uint8_t *stage = smem + warp * 2 * STAGE;
    const uint32_t stage_s = smem_u32(stage);

    for (int g = warp; g < G; g += kWarps) {
        // q_idx fragments (B operand, "col": k = d, n = row): b0 = k 0..7 pair, b1 = k 8..15 pair
        uint32_t bq[2][KS][2];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                const int n = nt * 8 + (lane >> 2);
                const int d = ks * 16 + (lane & 3) * 2;
                uint32_t v0 = 0, v1 = 0;
                if (n < T) {
                    const uint16_t *qp = q_idx + (size_t(row0 + n) * G + g) * DI;
                    v0 = *reinterpret_cast<const uint32_t *>(qp + d);
                    v1 = *reinterpret_cast<const uint32_t *>(qp + d + 8);
                }
                bq[nt][ks][0] = v0;
                bq[nt][ks][1] = v1;
            }
        // the group's 128 token rows of the page: token i at ((page * 128 + i) * G + g) * DI
        const uint8_t *src = kidx + (size_t(page) * 128 * G + g) * DI * 2;
        auto issue = [&](int c) {
            const uint32_t dst = stage_s + uint32_t((c & 1) * STAGE);
#pragma unroll
            for (int k = 0; k < kChunkTok * CH / 32; ++k) {
                const int p = lane + 32 * k;
                const int i = p / CH, q = p % CH;
                cp_async_16(dst + stage_off<DI>(i, q), src + (size_t(c * kChunkTok + i) * G) * DI * 2 + q * 16);
            }
            cp_async_commit();
        };
        float mx[2][2];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) mx[nt][0] = mx[nt][1] = -INFINITY;
        issue(0);
        issue(1);
#pragma unroll 1
        for (int c = 0; c < 128 / kChunkTok; ++c) {
            cp_async_wait<1>();   // chunk c has landed (chunk c + 1 may be in flight)
            __syncwarp();
            const uint32_t buf = stage_s + uint32_t((c & 1) * STAGE);
#pragma unroll
            for (int mt = 0; mt < kChunkTok / 16; ++mt) {
                float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    // A = 16 tokens x 16 index dims: matrices (rows 0-7 | 8-15) x (cols 0-7 | 8-15)
                    const int r = mt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                    const int q = ks * 2 + (lane >> 4);
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4(buf + stage_off<DI>(r, q), a0, a1, a2, a3);
                    mma16816(acc[0], a0, a1, a2, a3, bq[0][ks][0], bq[0][ks][1]);
                    if (NT > 1) mma16816(acc[1], a0, a1, a2, a3, bq[1][ks][0], bq[1][ks][1]);
                }
                // accumulator: acc[nt][h * 2 + e] = token (lane >> 2) + 8 h, row nt * 8 + (lane & 3) * 2 + e
                const int tok0 = j * 128 + c * kChunkTok + mt * 16 + (lane >> 2);
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int h = 0; h < 2; ++h)
#pragma unroll
                        for (int e = 0; e < 2; ++e)
                            if (tok0 + 8 * h <= pos[nt][e]) mx[nt][e] = fmaxf(mx[nt][e], acc[nt][h * 2 + e]);
            }
            __syncwarp();
            if (c + 2 < 128 / kChunkTok) issue(c + 2);
            else cp_async_commit();   // keep one group per chunk so that wait<1> stays exact
        }
        cp_async_wait<0>();
        // max over the 8 lanes that share the columns
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                float v = mx[nt][e];
                v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
                v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
                v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
                mx[nt][e] = v;
            }
        if (lane < 4) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int n = nt * 8 + lane * 2 + e;
                    if (n < T)
                        scores[(size_t(row0 + n) * G + g) * max_blocks + j] =
                            j <= (pos[nt][e] >> 7) ? mx[nt][e] : -INFINITY;
                }
        }
        __syncwarp();   // the stage buffers are reused by the next group
    }
}

template <int DI>
cudaError_t launch_di(const void *q_idx, const void *kidx, const int32_t *bt, const int32_t *q_req,
                      const int32_t *q_pos, int n_rows, int n_req, int n_pages, const Shape &s, float *scores,
                      int32_t *err, cudaStream_t st) {
    if (s.max_blocks > 65535) return cudaErrorInvalidConfiguration;
    const size_t smem = size_t(kWarps) * 2 * kChunkTok * DI * 2;
    cudaError_t e =
        cudaFuncSetAttribute(k_score_decode_mt<DI>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    dim3 grid(unsigned(n_req), unsigned(s.max_blocks));
    k_score_decode_mt<DI><<<grid, kWarps * 32, smem, st>>>(
        static_cast<const uint16_t *>(q_idx), static_cast<const uint8_t *>(kidx), bt, q_req, q_pos, n_rows, n_req,
        n_pages, s.G, s.max_blocks, scores, err);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_score_decode_mt(const void *q_idx, const void *kidx, const int32_t *block_table,
                                   const int32_t *q_req, const int32_t *q_pos, int n_rows, int n_req, int n_pages,
                                   const Shape &s, float *scores, int32_t *err, cudaStream_t st) {
    if (n_rows <= 0) return cudaSuccess;
    if (s.Di == 64)
        return launch_di<64>(q_idx, kidx, block_table, q_req, q_pos, n_rows, n_req, n_pages, s, scores, err, st);
    if (s.Di == 32)
        return launch_di<32>(q_idx, kidx, block_table, q_req, q_pos, n_rows, n_req, n_pages, s, scores, err, st);
    return cudaErrorNotSupported;
}

}  // namespace msa
