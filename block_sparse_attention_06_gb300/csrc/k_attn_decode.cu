// Decode sparse attention over per-(request, group) page tables.
//
// "Together AI 解析如何高效服务 MiniMax M3…", section 将 MSA 与分页注意力集成: the
// selected blocks become a page table per flattened (request, KV group) row and a
// GQA paged-attention kernel reads the pages through a strided view of the
// physical [pages][128][G][D] cache.  This file is that kernel, written for one
// GB300 SM per (row, page) work item:
//   - K and V of one page of one group (128 rows of D bf16, row stride G*D) are
//     fetched by two 4-D TMA boxes each (128B-swizzled, 64 columns per box);
//   - the Hq/G heads of the group are the N = 8 side of an AB-swapped
//     m16n8k16 bf16 MMA (tokens = M), the way the page's own index-scoring kernel
//     uses 128-token tiles as M; decode attention moves ~8 flop per byte, so
//     these small legacy tiles keep it HBM-bound;
//   - each work item writes a normalised partial (O, lse) to the workspace and
//     counts itself done on the row's counter; the work item that finishes a row
//     last merges the row's partials by Log-Sum-Exp (the reduction of section
//     KV 块主序稀疏注意力) and writes the output, so no second kernel runs.
#include "msa_device.cuh"
#include "msa_internal.h"

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

template <int D, int HPG>
struct DecodeSmem {
    alignas(1024) uint8_t k[D * 128 * 2];
    alignas(1024) uint8_t v[D * 128 * 2];
    uint16_t p[8][136];          // unnormalised probabilities, [head][token], padded rows
    float red[4][8];
    float red2[4][8];
    float m[8];
    float l[8];    // sum of the bf16-rounded probabilities
    float le[8];   // exact fp32 sum
    float mlse[32 * 8];   // merge: lse of every (slot, head) of the row
    uint64_t kbar, vbar;
    int abort;
    int last;
};

// One (row, page) work item: S^T = K Q^T on the tensor cores (tokens = M, the
// group's heads = N), softmax over the page's n_tok tokens, O^T = V^T P^T, and the
// normalised partial (O, lse) of the page into o_out / lse_out.
template <int D, int HPG>
__device__ __forceinline__ void attend_page(DecodeSmem<D, HPG> &sm, const uint16_t *__restrict__ q,
                                            const CUtensorMap &kmap, const CUtensorMap &vmap, int r, int G,
                                            int page, int n_tok, float sm_scale, float *__restrict__ o_out,
                                            float *__restrict__ lse_out, int32_t *err) {
    constexpr int NB = D / 64;   // TMA boxes per tile
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b = r / G, g = r - b * G;
    if (tid == 0) {
        mbar_init(&sm.kbar, 1);
        mbar_init(&sm.vbar, 1);
        sm.abort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0) {
        mbar_arrive_expect_tx(&sm.kbar, D * 128 * 2);
#pragma unroll
        for (int i = 0; i < NB; ++i) tma_load_4d(sm.k + i * 16384, &kmap, &sm.kbar, i * 64, g, 0, page);
        mbar_arrive_expect_tx(&sm.vbar, D * 128 * 2);
#pragma unroll
        for (int i = 0; i < NB; ++i) tma_load_4d(sm.v + i * 16384, &vmap, &sm.vbar, i * 64, g, 0, page);
    }

    // Q of this group as the B operand (col-major K x N: column n = head n).
    const int n_head = lane >> 2;
    const uint16_t *qh = q + (size_t(b) * (G * HPG) + size_t(g) * HPG + n_head) * D;
    uint32_t qb[D / 16][2];
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        if (n_head < HPG) {
            qb[kk][0] = *reinterpret_cast<const uint32_t *>(qh + kk * 16 + 2 * (lane & 3));
            qb[kk][1] = *reinterpret_cast<const uint32_t *>(qh + kk * 16 + 8 + 2 * (lane & 3));
        } else {
            qb[kk][0] = qb[kk][1] = 0u;
        }
    }

    // warp-uniform outcome: the MMAs below are warp-collective
    const bool k_ok = __all_sync(0xffffffffu, mbar_wait(&sm.kbar, 0, err, &sm.abort));
    // S^T = K Q^T: this warp's 32 tokens as two m16 tiles.
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    const uint32_t kbase = smem_u32(sm.k);
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
    __syncthreads();
    if (tid < 8) sm.m[tid] = fmaxf(fmaxf(sm.red[0][tid], sm.red[1][tid]), fmaxf(sm.red[2][tid], sm.red[3][tid]));
    __syncthreads();
    const float m0 = sm.m[2 * (lane & 3)], m1 = sm.m[2 * (lane & 3) + 1];
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
            sm.p[2 * (lane & 3)][t] = uint16_t(pk & 0xffffu);
            sm.p[2 * (lane & 3) + 1][t] = uint16_t(pk >> 16);
        }
    }
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
        s0 += __shfl_xor_sync(0xffffffffu, s0, o);
        s1 += __shfl_xor_sync(0xffffffffu, s1, o);
        e0 += __shfl_xor_sync(0xffffffffu, e0, o);
        e1 += __shfl_xor_sync(0xffffffffu, e1, o);
    }
    __syncthreads();   // everyone read sm.red / wrote sm.p
    if (lane < 4) {
        sm.red[warp][2 * lane] = s0;
        sm.red[warp][2 * lane + 1] = s1;
        sm.red2[warp][2 * lane] = e0;
        sm.red2[warp][2 * lane + 1] = e1;
    }
    __syncthreads();
    if (tid < 8) {
        sm.l[tid] = (sm.red[0][tid] + sm.red[1][tid]) + (sm.red[2][tid] + sm.red[3][tid]);
        sm.le[tid] = (sm.red2[0][tid] + sm.red2[1][tid]) + (sm.red2[2][tid] + sm.red2[3][tid]);
    }
    const bool v_ok = __all_sync(0xffffffffu, mbar_wait(&sm.vbar, 0, err, &sm.abort));
    __syncthreads();

    // O^T = V^T P^T: this warp's D/4 output columns as m16 tiles over 128 tokens.
    constexpr int MT = D / 64;   // m16 tiles per warp (D/4 columns each warp)
    float oacc[MT][4];
#pragma unroll
    for (int i = 0; i < MT; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;
    const uint32_t vbase = smem_u32(sm.v);
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
                uint32_t a0, a1, a2, a3;
                ldsm_x4_t(vbase + swz_off(t, c), a0, a1, a2, a3);
                mma16816(oacc[mt], a0, a1, a2, a3, b0, b1);
            }
        }
    }
    // write the normalised partial: c0/c1 -> (d0 + lane/4, heads 2*(lane&3), +1); c2/c3 -> d + 8
    const int n0 = 2 * (lane & 3);
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
        const int d = warp * (D / 4) + mt * 16 + (lane >> 2);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int n = n0 + h;
            if (n < HPG) {
                const float inv = 1.0f / sm.l[n];
                o_out[size_t(n) * D + d] = oacc[mt][h] * inv;
                o_out[size_t(n) * D + d + 8] = oacc[mt][2 + h] * inv;
            }
        }
    }
    if (tid < HPG) lse_out[tid] = (k_ok && v_ok) ? (sm.m[tid] + log2f(sm.le[tid])) * kLn2 : -INFINITY;
}

// Merge the topk partials of row r = b*G + g into out[b][g*HPG + n][:] and lse.
// Called by all 128 threads of the CTA that finished the row last; the partials
// of the other CTAs are read through L2 (ld.global.cg), never a stale L1 line.
template <int D, int HPG>
__device__ __forceinline__ void merge_row(DecodeSmem<D, HPG> &sm, const float *__restrict__ o_ws,
                                          const float *__restrict__ lse_ws, int r, int G, int topk,
                                          uint16_t *__restrict__ out, float *__restrict__ lse) {
    const int tid = threadIdx.x;
    const float *ls = lse_ws + size_t(r) * topk * HPG;
    for (int i = tid; i < topk * HPG; i += 128) sm.mlse[i] = __ldcg(ls + i);
    __syncthreads();
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
#pragma unroll 4
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
__global__ void __launch_bounds__(128) k_attn_decode(
    const uint16_t *__restrict__ q, const __grid_constant__ CUtensorMap kmap,
    const __grid_constant__ CUtensorMap vmap, const int32_t *__restrict__ pt,
    const int32_t *__restrict__ row_len, int G, int topk, int n_pages, float sm_scale,
    float *__restrict__ o_ws, float *__restrict__ lse_ws, int32_t *__restrict__ counters,
    uint16_t *__restrict__ out, float *__restrict__ lse, int32_t *err) {
    static_assert(HPG == 4 || HPG == 8, "heads per group");
    extern __shared__ uint8_t smem_raw[];
    DecodeSmem<D, HPG> &sm =
        *reinterpret_cast<DecodeSmem<D, HPG> *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const int slot = blockIdx.x, r = blockIdx.y;
    const int tid = threadIdx.x;
    float *lse_out = lse_ws + (size_t(r) * topk + slot) * HPG;
    float *o_out = o_ws + (size_t(r) * topk + slot) * HPG * D;

    tma_prefetch_desc(&kmap);
    tma_prefetch_desc(&vmap);
    pdl_wait();   // the page table comes from the previous kernel
    pdl_trigger();

    const int page = pt[size_t(r) * topk + slot];
    const int n_tok = min(128, row_len[r] - slot * 128);
    if (page < 0 || n_tok <= 0 || page >= n_pages) {
        if (page >= n_pages && tid == 0) raise_flag(err, MSA_FLAG_BOUNDS);
        if (tid < HPG) lse_out[tid] = -INFINITY;
    } else {
        attend_page<D, HPG>(sm, q, kmap, vmap, r, G, page, n_tok, sm_scale, o_out, lse_out, err);
    }

    // Count this work item done; the last of the row's topk work items merges.
    __threadfence();
    __syncthreads();
    if (tid == 0) sm.last = atomicAdd(counters + r, 1) == topk - 1;
    __syncthreads();
    if (!sm.last) return;
    __threadfence();
    if (tid == 0) counters[r] = 0;   // leave the counter clean
    merge_row<D, HPG>(sm, o_ws, lse_ws, r, G, topk, out, lse);
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
    return launch_kernel(k_attn_decode<D, HPG>, dim3(unsigned(s.topk), unsigned(B * s.G)), dim3(128), smem, st,
                         pdl && counters_zeroed, static_cast<const uint16_t *>(q), km, vm, pt, row_len, s.G, s.topk,
                         n_pages, s.sm_scale, o_ws, l_ws, cnt, static_cast<uint16_t *>(out), lse, err);
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
