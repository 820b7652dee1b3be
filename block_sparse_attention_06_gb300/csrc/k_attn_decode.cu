// Decode sparse attention over per-(request, group) page tables.
//
// "Together AI 解析如何高效服务 MiniMax M3…", section 将 MSA 与分页注意力集成: the
// selected blocks become a page table per flattened (request, KV group) row and a
// GQA paged-attention kernel reads the pages through a strided view of the
// physical [pages][128][G][D] cache.  This file is that kernel, written as one
// persistent CTA per GB300 SM that walks (row, page) work items:
//   - K and V of one page of one group (128 rows of D bf16, row stride G*D) are
//     fetched by two 4-D TMA boxes each (128B-swizzled, 64 columns per box);
//   - the Hq/G heads of the group are the N = 8 side of an AB-swapped
//     m16n8k16 bf16 MMA (tokens = M), the way the page's own index-scoring kernel
//     uses 128-token tiles as M; decode attention moves ~8 flop per byte, so
//     these small legacy tiles keep it HBM-bound;
//   - each row segment (the row's pages inside one CTA's range) writes one
//     normalised partial (O, lse) to the workspace and counts its pages done on
//     the row's counter; the segment that completes a row merges the row's
//     partials by Log-Sum-Exp (the reduction of section KV 块主序稀疏注意力) and
//     writes the output, so no second kernel runs.
#include "msa_device.cuh"
#include "msa_internal.h"

#include <algorithm>

namespace msa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                          uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
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

// Byte offset of the 16-byte chunk `c` (0 .. D/8-1) of row `t` in a tile stored as
// D/64 boxes of [128 rows][64 bf16] with the TMA 128-byte swizzle.
__device__ __forceinline__ uint32_t swz_off(int t, int c) {
    return uint32_t((c >> 3) * 16384 + t * 128 + (((c & 7) ^ (t & 7)) << 4));
}

// Work split (stream-K over pages): the n = B*G*topk (row, page) work items, item =
// r*topk + slot, are cut into gridDim.x contiguous ranges, one per CTA and one CTA
// per SM.  Inside its range a CTA keeps one online-softmax state per row segment
// (the pages of one row that fall in the range), so it writes one partial per
// segment rather than one per page: at most 1 + ceil(topk / shortest range) per
// row, e.g. four for 16 pages per row over ranges of 6 or 7 pages.  Warp 4 (lane
// 0) streams the range's K and V pages through an NS-deep ring of shared-memory
// stages with TMA while warps 0-3 attend: loads of later pages stay in flight
// during the compute of the current one.
template <int D, int HPG>
struct DecodeSmem {
    static constexpr int NS = D == 128 ? 3 : 6;   // stages of K and V (64 KB or 32 KB each)
    alignas(1024) uint8_t k[NS][D * 128 * 2];
    alignas(1024) uint8_t v[NS][D * 128 * 2];
    uint16_t p[8][136];          // unnormalised probabilities, [head][token], padded rows
    float red[4][8];
    float red2[4][8];
    float m[8];       // the segment's max per head, log2 units (for its lse)
    float mlse[32 * 8];   // merge: lse of every (slot, head) of the row
    uint64_t k_full[NS], v_full[NS], empty[NS];
    int abort;
    int last;
};

constexpr int kConsumerThreads = 128;   // warps 0-3: attention and merge
constexpr int kThreads = kConsumerThreads + 32;   // + warp 4: the TMA producer

// Named barrier over the four consumer warps (the producer warp never joins it).
__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// First work item of CTA c when n items are cut into C ranges.
__device__ __forceinline__ int range_begin(int c, int n, int C) { return int((long long)c * n / C); }

// The CTA whose range holds item x: the c with range_begin(c) <= x < range_begin(c + 1).
__device__ __forceinline__ int range_owner(int x, int n, int C) { return int(((long long)(x + 1) * C - 1) / n); }

// Tokens of work item `item` to attend: 0 for an empty slot (page -1, or past the
// row's length) and for an out-of-range page.  Producer and consumers derive it
// from the same global words, so every consumer thread takes the same branch.
__device__ __forceinline__ int item_tokens(const int32_t *__restrict__ pt, const int32_t *__restrict__ row_len,
                                           int item, int topk, int n_pages, int *page_out) {
    const int r = item / topk, slot = item - r * topk;
    const int page = pt[item];
    const int n_tok = min(128, row_len[r] - slot * 128);
    *page_out = page;
    return (page < 0 || page >= n_pages || n_tok <= 0) ? 0 : n_tok;
}

// Q of row r's group as the B operand (col-major K x N: column n = head n).
template <int D, int HPG>
__device__ __forceinline__ void load_q(uint32_t (&qb)[D / 16][2], const uint16_t *__restrict__ q, int r, int G) {
    const int lane = threadIdx.x & 31;
    const int n_head = lane >> 2;
    const int b = r / G, g = r - b * G;
    const uint16_t *qh = q + (size_t(b) * (G * HPG) + size_t(g) * HPG + n_head) * D;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        if (n_head < HPG) {
            qb[kk][0] = __ldg(reinterpret_cast<const uint32_t *>(qh + kk * 16 + 2 * (lane & 3)));
            qb[kk][1] = __ldg(reinterpret_cast<const uint32_t *>(qh + kk * 16 + 8 + 2 * (lane & 3)));
        } else {
            qb[kk][0] = qb[kk][1] = 0u;
        }
    }
}

// One page of the current segment in stage `stg`: S^T = K Q^T on the tensor cores
// (tokens = M, the group's heads = N), the online-softmax update (page max over the
// four warps, rescale alpha, exp2, bf16 P), then O^T = alpha * O^T + V^T P^T into the
// warp's accumulators; the stage goes back to the producer.  Each thread keeps the
// segment's running max of its two heads (2*(lane&3), +1; equal in every thread)
// and running partial sums over its own tokens in registers, so a page costs two
// barriers: the max exchange and P.  Run by the four consumer warps together.
template <int D, int HPG>
__device__ __forceinline__ void attend_page(DecodeSmem<D, HPG> &sm, int stg, uint32_t ph,
                                            const uint32_t (&qb)[D / 16][2], int n_tok, float sm_scale,
                                            float (&oacc)[D / 64][4], float (&mrun)[2], float (&lrun)[2],
                                            float (&lerun)[2], int32_t *err) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // warp-uniform outcome: the MMAs below are warp-collective
    const bool k_ok = __all_sync(0xffffffffu, mbar_wait(&sm.k_full[stg], ph, err, &sm.abort));
    // S^T = K Q^T: this warp's 32 tokens as two m16 tiles.
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    const uint32_t kbase = smem_u32(sm.k[stg]);
    if (k_ok) {
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
            const int t = warp * 32 + mt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                uint32_t a0, a1, a2, a3;
                ldsm_x4(kbase + swz_off(t, kk * 2 + (lane >> 4)), a0, a1, a2, a3);
                mma16816(acc[mt], a0, a1, a2, a3, qb[kk][0], qb[kk][1]);
            }
        }
    }
    // logits in log2 units; mask tokens past the row's length.
    const float sc = sm_scale * kLog2e;
    float mx0 = -INFINITY, mx1 = -INFINITY;   // heads 2*(lane&3) and +1
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int t = warp * 32 + mt * 16 + (lane >> 2) + h * 8;
            const bool ok = t < n_tok;
            acc[mt][2 * h + 0] = ok ? acc[mt][2 * h + 0] * sc : -INFINITY;
            acc[mt][2 * h + 1] = ok ? acc[mt][2 * h + 1] * sc : -INFINITY;
            mx0 = fmaxf(mx0, acc[mt][2 * h + 0]);
            mx1 = fmaxf(mx1, acc[mt][2 * h + 1]);
        }
    }
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
    }
    if (lane < 4) {
        sm.red[warp][2 * lane] = mx0;
        sm.red[warp][2 * lane + 1] = mx1;
    }
    consumer_sync();   // the four warps' page maxima are in sm.red
    // The page holds at least one visible token, so the new max is finite and
    // alpha = 0 while the segment's running max is still -inf.
    const int n0 = 2 * (lane & 3);
    const float m0 = fmaxf(mrun[0], fmaxf(fmaxf(sm.red[0][n0], sm.red[1][n0]), fmaxf(sm.red[2][n0], sm.red[3][n0])));
    const float m1 = fmaxf(mrun[1], fmaxf(fmaxf(sm.red[0][n0 + 1], sm.red[1][n0 + 1]),
                                          fmaxf(sm.red[2][n0 + 1], sm.red[3][n0 + 1])));
    const float al0 = exp2f(mrun[0] - m0), al1 = exp2f(mrun[1] - m1);
    mrun[0] = m0;
    mrun[1] = m1;
    // Two normalisers: the sum of the bf16-rounded probabilities that the PV MMA
    // consumes (normalises O, so its weights sum to one) and the exact fp32 sum
    // (gives the lse).
    float s0 = 0.f, s1 = 0.f, e0 = 0.f, e1 = 0.f;
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int t = warp * 32 + mt * 16 + (lane >> 2) + h * 8;
            const float p0 = exp2f(acc[mt][2 * h + 0] - m0);
            const float p1 = exp2f(acc[mt][2 * h + 1] - m1);
            const uint32_t pk = pack_bf16x2(p0, p1);
            s0 += bf16_lo(pk);
            s1 += bf16_hi(pk);
            e0 += p0;
            e1 += p1;
            sm.p[n0][t] = uint16_t(pk & 0xffffu);
            sm.p[n0 + 1][t] = uint16_t(pk >> 16);
        }
    }
    lrun[0] = fmaf(al0, lrun[0], s0);
    lrun[1] = fmaf(al1, lrun[1], s1);
    lerun[0] = fmaf(al0, lerun[0], e0);
    lerun[1] = fmaf(al1, lerun[1], e1);
    const bool v_ok = __all_sync(0xffffffffu, mbar_wait(&sm.v_full[stg], ph, err, &sm.abort));
    consumer_sync();   // P of all 128 tokens is in sm.p; every warp has read sm.red

    // O^T = alpha * O^T + V^T P^T: this warp's D/4 output columns as m16 tiles over 128 tokens.
    constexpr int MT = D / 64;   // m16 tiles per warp (D/4 columns each warp)
#pragma unroll
    for (int i = 0; i < MT; ++i) {
        oacc[i][0] *= al0;
        oacc[i][1] *= al1;
        oacc[i][2] *= al0;
        oacc[i][3] *= al1;
    }
    const uint32_t vbase = smem_u32(sm.v[stg]);
    if (v_ok && k_ok) {
#pragma unroll
        for (int kt = 0; kt < 8; ++kt) {
            const int tk0 = kt * 16;
            const uint32_t b0 = *reinterpret_cast<const uint32_t *>(&sm.p[lane >> 2][tk0 + 2 * (lane & 3)]);
            const uint32_t b1 = *reinterpret_cast<const uint32_t *>(&sm.p[lane >> 2][tk0 + 8 + 2 * (lane & 3)]);
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                const int d0 = warp * (D / 4) + mt * 16;
                const int t = tk0 + (lane & 7) + ((lane >> 4) & 1) * 8;
                const int c = (d0 >> 3) + ((lane >> 3) & 1);
                uint32_t x0, x1, x2, x3;
                ldsm_x4_t(vbase + swz_off(t, c), x0, x1, x2, x3);
                mma16816(oacc[mt], x0, x1, x2, x3, b0, b1);
            }
        }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.empty[stg]);   // this warp is done with the stage
}

// Merge the partials of row r = b*G + g into out[b][g*HPG + n][:] and lse.  The row's
// partials sit at the slots where one of its segments starts (slot 0 and every slot
// that begins a CTA's range); the other slots hold nothing.  Called by the four
// consumer warps of the CTA whose segment completed the row; the partials of other
// CTAs are read through L2 (ld.global.cg), never a stale L1 line.
template <int D, int HPG>
__device__ __forceinline__ void merge_row(DecodeSmem<D, HPG> &sm, const float *__restrict__ o_ws,
                                          const float *__restrict__ lse_ws, int r, int G, int topk, int n_items,
                                          uint16_t *__restrict__ out, float *__restrict__ lse) {
    const int tid = threadIdx.x;
    const float *ls = lse_ws + size_t(r) * topk * HPG;
    for (int i = tid; i < topk * HPG; i += kConsumerThreads) {
        const int s = i / HPG, x = r * topk + s;
        const bool start = s == 0 || range_begin(range_owner(x, n_items, gridDim.x), n_items, gridDim.x) == x;
        sm.mlse[i] = start ? __ldcg(ls + i) : -INFINITY;
    }
    consumer_sync();
    constexpr int TPH = D / 8;              // threads per head, 8 columns each
    const int n = tid / TPH;
    const int d = (tid % TPH) * 8;
    if (n >= HPG) return;
    const int b = r / G, g = r - b * G;
    float m = -INFINITY;
    for (int s = 0; s < topk; ++s) m = fmaxf(m, sm.mlse[s * HPG + n]);
    const size_t h = size_t(b) * G * HPG + size_t(g) * HPG + n;
    uint16_t *o = out + h * D + d;
    if (m == -INFINITY) {
        *reinterpret_cast<uint4 *>(o) = make_uint4(0u, 0u, 0u, 0u);
        if (d == 0) lse[h] = -INFINITY;
        return;
    }
    float sum = 0.f;
    for (int s = 0; s < topk; ++s) {
        const float l = sm.mlse[s * HPG + n];
        if (l != -INFINITY) sum += __expf(l - m);
    }
    const float tot = m + __logf(sum);
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    const float *src = o_ws + (size_t(r) * topk * HPG + n) * D + d;
    for (int s = 0; s < topk; ++s) {
        const float l = sm.mlse[s * HPG + n];
        if (l == -INFINITY) continue;
        const float w = __expf(l - tot);
        const float4 v0 = __ldcg(reinterpret_cast<const float4 *>(src + size_t(s) * HPG * D));
        const float4 v1 = __ldcg(reinterpret_cast<const float4 *>(src + size_t(s) * HPG * D + 4));
        acc[0] = fmaf(w, v0.x, acc[0]);
        acc[1] = fmaf(w, v0.y, acc[1]);
        acc[2] = fmaf(w, v0.z, acc[2]);
        acc[3] = fmaf(w, v0.w, acc[3]);
        acc[4] = fmaf(w, v1.x, acc[4]);
        acc[5] = fmaf(w, v1.y, acc[5]);
        acc[6] = fmaf(w, v1.z, acc[6]);
        acc[7] = fmaf(w, v1.w, acc[7]);
    }
    *reinterpret_cast<uint4 *>(o) = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                                               pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
    if (d == 0) lse[h] = tot;
}

template <int D, int HPG>
__global__ void __launch_bounds__(kThreads, 1) k_attn_decode(
    const uint16_t *__restrict__ q, const __grid_constant__ CUtensorMap kmap,
    const __grid_constant__ CUtensorMap vmap, const int32_t *__restrict__ pt,
    const int32_t *__restrict__ row_len, int G, int topk, int n_items, int n_pages, float sm_scale,
    float *__restrict__ o_ws, float *__restrict__ lse_ws, int32_t *__restrict__ counters,
    uint16_t *__restrict__ out, float *__restrict__ lse, int32_t *err) {
    static_assert(HPG == 4 || HPG == 8, "heads per group");
    using Smem = DecodeSmem<D, HPG>;
    constexpr int NS = Smem::NS;
    constexpr int NB = D / 64;   // TMA boxes per tile
    constexpr int MT = D / 64;
    extern __shared__ uint8_t smem_raw[];
    Smem &sm = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int x0 = range_begin(blockIdx.x, n_items, gridDim.x);
    const int x1 = range_begin(blockIdx.x + 1, n_items, gridDim.x);
    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&sm.k_full[s], 1);
            mbar_init(&sm.v_full[s], 1);
            mbar_init(&sm.empty[s], kConsumerThreads / 32);
        }
        sm.abort = 0;
        fence_mbar_init();
    }
    if (tid == 32 * 4) {
        tma_prefetch_desc(&kmap);
        tma_prefetch_desc(&vmap);
    }
    __syncthreads();
    pdl_wait();   // the page table, the row lengths and the zeroed counters come from the previous kernel
    pdl_trigger();

    if (warp == 4) {
        // ------------------------------------------------------------ TMA producer (lane 0)
        if (lane != 0) return;
        int issued = 0;
        int page_n;
        int tok_n = x0 < x1 ? item_tokens(pt, row_len, x0, topk, n_pages, &page_n) : 0;
        for (int x = x0; x < x1; ++x) {
            const int it = x - x0, stg = it % NS;
            const int page = page_n, n_tok = tok_n;
            if (x + 1 < x1) tok_n = item_tokens(pt, row_len, x + 1, topk, n_pages, &page_n);   // one ahead
            if (it >= NS && !mbar_wait(&sm.empty[stg], ((it / NS) - 1) & 1, err, &sm.abort)) break;
            if (*reinterpret_cast<volatile int *>(&sm.abort)) break;
            if (n_tok > 0) {
                const int g = (x / topk) % G;
                mbar_arrive_expect_tx(&sm.k_full[stg], D * 128 * 2);
#pragma unroll
                for (int i = 0; i < NB; ++i) tma_load_4d(sm.k[stg] + i * 16384, &kmap, &sm.k_full[stg], i * 64, g, 0, page);
                mbar_arrive_expect_tx(&sm.v_full[stg], D * 128 * 2);
#pragma unroll
                for (int i = 0; i < NB; ++i) tma_load_4d(sm.v[stg] + i * 16384, &vmap, &sm.v_full[stg], i * 64, g, 0, page);
            } else {
                if (page >= n_pages) raise_flag(err, MSA_FLAG_BOUNDS);
                mbar_arrive(&sm.k_full[stg]);   // nothing to load: the consumers still see the phase complete
                mbar_arrive(&sm.v_full[stg]);
            }
            issued = it + 1;
        }
        if (sm.abort) {   // drain: the copies still in flight land before the CTA exits
            for (int it = max(0, issued - NS); it < issued; ++it) {
                mbar_wait(&sm.k_full[it % NS], (it / NS) & 1, err, nullptr);
                mbar_wait(&sm.v_full[it % NS], (it / NS) & 1, err, nullptr);
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumers (warps 0-3)
    uint32_t qb[D / 16][2];
    int page_n;
    int tok_n = x0 < x1 ? item_tokens(pt, row_len, x0, topk, n_pages, &page_n) : 0;
    for (int x = x0; x < x1;) {
        // one segment: the pages x .. seg_end-1 of row r
        const int r = x / topk;
        const int seg_start = x, seg_end = min(x1, (r + 1) * topk);
        load_q<D, HPG>(qb, q, r, G);
        float oacc[MT][4];
#pragma unroll
        for (int i = 0; i < MT; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;
        float mrun[2] = {-INFINITY, -INFINITY}, lrun[2] = {0.f, 0.f}, lerun[2] = {0.f, 0.f};
        for (; x < seg_end; ++x) {
            const int it = x - x0, stg = it % NS;
            const uint32_t ph = (it / NS) & 1;
            const int n_tok = tok_n;
            if (x + 1 < x1) tok_n = item_tokens(pt, row_len, x + 1, topk, n_pages, &page_n);   // one ahead
            if (n_tok > 0) {
                attend_page<D, HPG>(sm, stg, ph, qb, n_tok, sm_scale, oacc, mrun, lrun, lerun, err);
            } else {
                mbar_wait(&sm.k_full[stg], ph, err, &sm.abort);
                mbar_wait(&sm.v_full[stg], ph, err, &sm.abort);
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.empty[stg]);
            }
        }
        // The segment's normalised partial goes to the slot where the segment starts.
        float *o_out = o_ws + size_t(seg_start) * HPG * D;
        float *lse_out = lse_ws + size_t(seg_start) * HPG;
        // The segment's sums: over the lanes of equal lane&3, then over the four warps.
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            lrun[0] += __shfl_xor_sync(0xffffffffu, lrun[0], o);
            lrun[1] += __shfl_xor_sync(0xffffffffu, lrun[1], o);
            lerun[0] += __shfl_xor_sync(0xffffffffu, lerun[0], o);
            lerun[1] += __shfl_xor_sync(0xffffffffu, lerun[1], o);
        }
        // sm.red's last readers passed the page's P barrier (or, with no page attended
        // here, the previous segment's count barriers) before these writes
        if (lane < 4) {
            sm.red[warp][2 * lane] = lrun[0];
            sm.red[warp][2 * lane + 1] = lrun[1];
            sm.red2[warp][2 * lane] = lerun[0];
            sm.red2[warp][2 * lane + 1] = lerun[1];
            if (warp == 0) {
                sm.m[2 * lane] = mrun[0];
                sm.m[2 * lane + 1] = mrun[1];
            }
        }
        consumer_sync();
        const int n0 = 2 * (lane & 3);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int n = n0 + h;
            const float l = (sm.red[0][n] + sm.red[1][n]) + (sm.red[2][n] + sm.red[3][n]);
            const float inv = l > 0.f ? 1.0f / l : 0.f;
            if (n < HPG) {
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    const int d = warp * (D / 4) + mt * 16 + (lane >> 2);
                    o_out[size_t(n) * D + d] = oacc[mt][h] * inv;
                    o_out[size_t(n) * D + d + 8] = oacc[mt][2 + h] * inv;
                }
            }
        }
        if (tid < HPG) {
            const float le = (sm.red2[0][tid] + sm.red2[1][tid]) + (sm.red2[2][tid] + sm.red2[3][tid]);
            lse_out[tid] = le > 0.f ? (sm.m[tid] + log2f(le)) * kLn2 : -INFINITY;
        }

        // Count the segment's pages done; the segment that completes the row merges it.
        consumer_sync();   // every partial store of this CTA precedes thread 0's release below
        if (tid == 0) {
            __threadfence();
            const int n_seg = seg_end - seg_start;
            sm.last = atomicAdd(counters + r, n_seg) + n_seg == topk;
            if (sm.last) {
                __threadfence();
                counters[r] = 0;   // leave the counter clean
            }
        }
        consumer_sync();
        if (sm.last) merge_row<D, HPG>(sm, o_ws, lse_ws, r, G, topk, n_items, out, lse);
    }
}


struct DecodeWs {
    size_t o_off, lse_off, cnt_off, bytes;
};

inline DecodeWs decode_ws(int B, const Shape &s) {
    DecodeWs w;
    const size_t units = size_t(B) * s.G * s.topk;
    w.o_off = 0;
    w.lse_off = (units * s.hpg * s.D * 4 + 255) & ~size_t(255);
    w.cnt_off = w.lse_off + ((units * s.hpg * 4 + 255) & ~size_t(255));
    w.bytes = w.cnt_off + ((size_t(B) * s.G * 4 + 255) & ~size_t(255));
    return w;
}

template <int D, int HPG>
cudaError_t launch_t(const void *q, const CUtensorMap &km, const CUtensorMap &vm, const int32_t *pt,
                     const int32_t *row_len, int B, int n_pages, const Shape &s, void *out, float *lse,
                     void *ws, int32_t *err, cudaStream_t st, bool counters_zeroed, bool pdl) {
    const DecodeWs w = decode_ws(B, s);
    uint8_t *base = static_cast<uint8_t *>(ws);
    float *o_ws = reinterpret_cast<float *>(base + w.o_off);
    float *l_ws = reinterpret_cast<float *>(base + w.lse_off);
    int32_t *cnt = reinterpret_cast<int32_t *>(base + w.cnt_off);
    cudaError_t e;
    if (!counters_zeroed) {
        e = cudaMemsetAsync(cnt, 0, size_t(B) * s.G * 4, st);
        if (e != cudaSuccess) return e;
    }
    const size_t smem = sizeof(DecodeSmem<D, HPG>) + 1024;
    e = cudaFuncSetAttribute(k_attn_decode<D, HPG>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    const int n_items = B * s.G * s.topk;
    const int grid = std::min(n_items, sm_count());   // persistent: one CTA per SM (the stages fill its smem)
    return launch_kernel(k_attn_decode<D, HPG>, dim3(unsigned(grid)), dim3(kThreads), smem, st,
                         pdl && counters_zeroed, static_cast<const uint16_t *>(q), km, vm, pt, row_len, s.G, s.topk,
                         n_items, n_pages, s.sm_scale, o_ws, l_ws, cnt, static_cast<uint16_t *>(out), lse, err);
}

}  // namespace

size_t decode_workspace_bytes(int B, const Shape &s) { return decode_ws(B, s).bytes; }

int32_t *decode_ws_counters(void *ws, int B, const Shape &s) {
    return reinterpret_cast<int32_t *>(static_cast<uint8_t *>(ws) + decode_ws(B, s).cnt_off);
}

cudaError_t launch_attn_decode(const void *q, const void *k_cache, const void *v_cache, const int32_t *pt,
                               const int32_t *row_len, int B, int n_pages, const Shape &s, void *out,
                               float *lse, void *ws, int32_t *err, cudaStream_t st, bool counters_zeroed,
                               bool pdl) {
    if (B <= 0) return cudaSuccess;
    alignas(64) CUtensorMap km, vm;
    const uint64_t dims[4] = {uint64_t(s.D), uint64_t(s.G), 128ull, uint64_t(n_pages)};
    const uint64_t strides[3] = {uint64_t(s.D) * 2, uint64_t(s.G) * s.D * 2, 128ull * s.G * s.D * 2};
    const uint32_t box[4] = {64u, 1u, 128u, 1u};
    const char *why = nullptr;
    if (!encode_tensor_map(&km, 4, k_cache, dims, strides, box, 128, &why)) return cudaErrorInvalidValue;
    if (!encode_tensor_map(&vm, 4, v_cache, dims, strides, box, 128, &why)) return cudaErrorInvalidValue;
#define MSA_AD_CASE(DD, HH)                                                                                    \
    if (s.D == DD && s.hpg == HH)                                                                              \
        return launch_t<DD, HH>(q, km, vm, pt, row_len, B, n_pages, s, out, lse, ws, err, st, counters_zeroed, pdl);
    MSA_AD_CASE(128, 8) MSA_AD_CASE(128, 4) MSA_AD_CASE(64, 8) MSA_AD_CASE(64, 4)
#undef MSA_AD_CASE
    return cudaErrorNotSupported;
}

}  // namespace msa
