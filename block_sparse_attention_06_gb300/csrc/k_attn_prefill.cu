// KV-block-major sparse attention for prefill on the 5th-generation tensor cores.
//
// "Together AI 解析如何高效服务 MiniMax M3…", section KV 块主序稀疏注意力: several
// queries attend the same KV block, so looping over KV blocks outside and over
// the queries that selected them inside moves each block from HBM once; the page
// "NVIDIA 加速インフラ上で MiniMax M3 を…" (MSA paragraph after Table 1) states the
// same operator property.  Each block yields a partial O per (query, head) that
// is later combined by a Log-Sum-Exp reduction.
//
// One CTA owns one CSR key (KV group g, request, logical block j):
//   warp 0     TMA: K_j and V_j once (4-D boxes of [128 tokens][64 dims],
//              128B swizzle), then per tile of 128/HPG entries the HPG query
//              heads of group g of each entry's query row (one 3-D box per entry
//              and 64-column half) into a double-buffered Q tile;
//   warp 1     TMEM owner and MMA issuer: S = Q K^T (M = 128 query-head rows,
//              N = 128 tokens, K = D) into one of two TMEM S buffers, then
//              O = P V (N = D, V used MN-major) into a TMEM O buffer; S of the
//              next tile is issued before P of this one is ready;
//   warps 2-5  thread = query-head row: tcgen05.ld of S, causal mask against the
//              entry's position, exp2 softmax, P as bf16 into shared memory for
//              the second MMA, then tcgen05.ld of O, normalisation, bf16 store of
//              the partial and its lse.
// All waits are bounded; a timeout raises MSA_FLAG_TIMEOUT and drains.
#include "msa_device.cuh"
#include "msa_internal.h"

namespace msa {
namespace {

constexpr int kThreads = 192;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <int D>
struct AttnSmem {
    alignas(1024) uint8_t k[D * 128 * 2];
    alignas(1024) uint8_t v[D * 128 * 2];
    alignas(1024) uint8_t q[2][128 * D * 2];
    alignas(1024) uint8_t p[128 * 128 * 2];
    uint64_t kv_full;
    uint64_t q_full[2], q_empty[2];
    uint64_t s_full[2], s_free[2];
    uint64_t p_full, o_full, o_free;
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};

template <int D, int HPG>
__global__ void __launch_bounds__(kThreads, 1) k_attn_prefill(
    const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
    const __grid_constant__ CUtensorMap vmap, const int32_t *__restrict__ block_table,
    const int32_t *__restrict__ q_req, const int32_t *__restrict__ q_pos, const int32_t *__restrict__ blk_off,
    const int32_t *__restrict__ blk_ent, int n_rows, int n_req, int n_pages, int G, int topk, int max_blocks,
    float sm_scale, uint16_t *__restrict__ o_part, float *__restrict__ lse_part, int32_t *err) {
    constexpr int EPT = 128 / HPG;                 // entries per tile
    constexpr int NSUB = D / 64;                   // 64-column sub-tiles
    constexpr uint32_t kIdescS = make_idesc_bf16(128, 128, 0, 0);
    constexpr uint32_t kIdescO = make_idesc_bf16(128, D, 0, 1);
    constexpr uint32_t kTmemO = 256;
    extern __shared__ uint8_t smem_raw[];
    AttnSmem<D> &sm =
        *reinterpret_cast<AttnSmem<D> *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const int key = blockIdx.x;
    const int off = blk_off[key];
    const int end = blk_off[key + 1];
    if (end <= off) return;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const long long cap = 1LL * n_rows * G * topk;
    const int per_g = n_req * max_blocks;
    const int g = key / per_g;
    const int req = (key - g * per_g) / max_blocks;
    const int j = key - g * per_g - req * max_blocks;
    int page = block_table[size_t(req) * max_blocks + j];
    if (off < 0 || end > cap || page < 0 || page >= n_pages) {
        if (tid == 0) raise_flag(err, MSA_FLAG_BOUNDS);
        return;
    }
    const int n_ent = end - off;
    const int n_tiles = (n_ent + EPT - 1) / EPT;

    if (tid == 0) {
        mbar_init(&sm.kv_full, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sm.q_full[b], 1);
            mbar_init(&sm.q_empty[b], 1);
            mbar_init(&sm.s_full[b], 1);
            mbar_init(&sm.s_free[b], 4);
        }
        mbar_init(&sm.p_full, 4);
        mbar_init(&sm.o_full, 1);
        mbar_init(&sm.o_free, 4);
        mbar_init(&sm.drain, 1);
        sm.abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&sm.tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;

    if (warp == 0) {
        if (lane == 0) {
            tma_prefetch_desc(&qmap);
            mbar_arrive_expect_tx(&sm.kv_full, 2 * D * 128 * 2);
#pragma unroll
            for (int i = 0; i < NSUB; ++i) tma_load_4d(sm.k + i * 16384, &kmap, &sm.kv_full, i * 64, g, 0, page);
#pragma unroll
            for (int i = 0; i < NSUB; ++i) tma_load_4d(sm.v + i * 16384, &vmap, &sm.kv_full, i * 64, g, 0, page);
            int issued = 0;
            for (int t = 0; t < n_tiles; ++t) {
                const int b = t & 1;
                if (t >= 2 && !mbar_wait(&sm.q_empty[b], ((t >> 1) - 1) & 1, err, &sm.abort)) break;
                mbar_arrive_expect_tx(&sm.q_full[b], 128 * D * 2);
                for (int e = 0; e < EPT; ++e) {
                    const int idx = off + t * EPT + e;
                    int qq = n_rows;                    // fully out of bounds -> zero rows
                    if (idx < end) {
                        const int v = blk_ent[idx] / topk;
                        if (v >= 0 && v < n_rows) qq = v;
                    }
#pragma unroll
                    for (int i = 0; i < NSUB; ++i)
                        tma_load_3d(sm.q[b] + i * 16384 + e * HPG * 128, &qmap, &sm.q_full[b], i * 64, g * HPG, qq);
                }
                issued = t + 1;
            }
            if (sm.abort) {
                mbar_wait(&sm.kv_full, 0, err, nullptr);
                for (int t = max(0, issued - 2); t < issued; ++t) mbar_wait(&sm.q_full[t & 1], (t >> 1) & 1, err, nullptr);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t k_addr = smem_u32(sm.k), v_addr = smem_u32(sm.v), p_addr = smem_u32(sm.p);
            auto issue_s = [&](int t) -> bool {
                const int b = t & 1;
                if (!mbar_wait(&sm.q_full[b], (t >> 1) & 1, err, &sm.abort)) return false;
                if (t >= 2 && !mbar_wait(&sm.s_free[b], ((t >> 1) - 1) & 1, err, &sm.abort)) return false;
                tc_fence_after();
                const uint32_t q_addr = smem_u32(sm.q[b]);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t o = uint32_t((kk >> 2) * 16384 + (kk & 3) * 32);
                    mma_bf16(tmem + uint32_t(b * 128), make_smem_desc(q_addr + o, 16, 1024, 2),
                             make_smem_desc(k_addr + o, 16, 1024, 2), kIdescS, kk > 0 ? 1u : 0u);
                }
                mma_commit(&sm.s_full[b]);
                mma_commit(&sm.q_empty[b]);
                return true;
            };
            bool ok = mbar_wait(&sm.kv_full, 0, err, &sm.abort) && issue_s(0);
            for (int t = 0; ok && t < n_tiles; ++t) {
                if (t + 1 < n_tiles && !issue_s(t + 1)) break;
                if (!mbar_wait(&sm.p_full, t & 1, err, &sm.abort)) break;
                if (t >= 1 && !mbar_wait(&sm.o_free, (t - 1) & 1, err, &sm.abort)) break;
                tc_fence_after();
#pragma unroll
                for (int kt = 0; kt < 8; ++kt) {
                    const uint64_t ad = make_smem_desc(p_addr + uint32_t((kt >> 2) * 16384 + (kt & 3) * 32), 16, 1024, 2);
                    const uint64_t bd = make_smem_desc(v_addr + uint32_t(kt * 2048), 16384, 1024, 2);
                    mma_bf16(tmem + kTmemO, ad, bd, kIdescO, kt > 0 ? 1u : 0u);
                }
                mma_commit(&sm.o_full);
            }
            mma_commit(&sm.drain);
            mbar_wait(&sm.drain, 0, err, nullptr);
        }
    } else {
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const int e = row / HPG, h = row - (row / HPG) * HPG;
        const uint32_t lane_addr = tmem + (uint32_t(quad * 32) << 16);
        const float scale = sm_scale * kLog2e;
        const uint32_t p_row = smem_u32(sm.p) + uint32_t(row * 128);
        for (int t = 0; t < n_tiles; ++t) {
            const int b = t & 1;
            const int idx = off + t * EPT + e;
            bool valid = idx < end;
            int qq = 0, slot = 0, lim = 127;
            if (valid) {
                const int ent = blk_ent[idx];
                qq = ent / topk;
                slot = ent - qq * topk;
                if (ent < 0 || qq >= n_rows || q_req[qq] != req) {
                    raise_flag(err, MSA_FLAG_BOUNDS);
                    valid = false;
                } else {
                    lim = q_pos[qq] - j * 128;
                    if (lim < 0) {                      // block past the row's position: not a candidate
                        raise_flag(err, MSA_FLAG_BOUNDS);
                        valid = false;
                        lim = 127;
                    }
                }
            }
            if (!__all_sync(0xffffffffu, mbar_wait(&sm.s_full[b], (t >> 1) & 1, err, &sm.abort))) break;
            tc_fence_after();
            float s[128];
#pragma unroll
            for (int c0 = 0; c0 < 128; c0 += 32) {
                uint32_t v[32];
                tmem_ld32(lane_addr + uint32_t(b * 128 + c0), v);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) s[c0 + i] = __uint_as_float(v[i]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.s_free[b]);
            float m = -INFINITY;
#pragma unroll
            for (int c = 0; c < 128; ++c) {
                s[c] = (c <= lim) ? s[c] * scale : -INFINITY;
                m = fmaxf(m, s[c]);
            }
            // l: sum of the bf16-rounded probabilities the PV MMA consumes (normalises O);
            // le: exact fp32 sum (gives the lse)
            float l = 0.f, le = 0.f;
#pragma unroll
            for (int c0 = 0; c0 < 128; c0 += 8) {
                uint32_t w[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float pa = exp2f(s[c0 + 2 * i] - m), pb = exp2f(s[c0 + 2 * i + 1] - m);
                    w[i] = pack_bf16x2(pa, pb);
                    l += bf16_lo(w[i]) + bf16_hi(w[i]);
                    le += pa + pb;
                }
                const int cc = (c0 & 63) >> 3;
                const uint32_t addr = p_row + uint32_t((c0 >> 6) * 16384) + uint32_t((cc ^ (row & 7)) << 4);
                asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w[0]), "r"(w[1]), "r"(w[2]),
                             "r"(w[3])
                             : "memory");
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.p_full);

            if (!__all_sync(0xffffffffu, mbar_wait(&sm.o_full, t & 1, err, &sm.abort))) break;
            tc_fence_after();
            const float inv = 1.0f / l;
            uint16_t *dst = o_part + ((size_t(qq) * topk + slot) * (size_t(G) * HPG) + size_t(g) * HPG + h) * D;
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t v[32];
                tmem_ld32(lane_addr + kTmemO + uint32_t(c0), v);
                tmem_ld_wait();
                if (valid) {
#pragma unroll
                    for (int i = 0; i < 32; i += 8) {
                        uint4 w;
                        w.x = pack_bf16x2(__uint_as_float(v[i + 0]) * inv, __uint_as_float(v[i + 1]) * inv);
                        w.y = pack_bf16x2(__uint_as_float(v[i + 2]) * inv, __uint_as_float(v[i + 3]) * inv);
                        w.z = pack_bf16x2(__uint_as_float(v[i + 4]) * inv, __uint_as_float(v[i + 5]) * inv);
                        w.w = pack_bf16x2(__uint_as_float(v[i + 6]) * inv, __uint_as_float(v[i + 7]) * inv);
                        *reinterpret_cast<uint4 *>(dst + c0 + i) = w;
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.o_free);
            if (valid)
                lse_part[(size_t(qq) * topk + slot) * (size_t(G) * HPG) + size_t(g) * HPG + h] = (m + log2f(le)) * kLn2;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

template <int D, int HPG>
cudaError_t launch_t(const void *q, const void *k_cache, const void *v_cache, const int32_t *bt, const int32_t *q_req,
                     const int32_t *q_pos, const int32_t *blk_off, const int32_t *blk_ent, int n_rows, int n_req,
                     int n_pages, const Shape &s, void *o_part, float *lse_part, int32_t *err, cudaStream_t st) {
    alignas(64) CUtensorMap qm, km, vm;
    const char *why = nullptr;
    {
        const uint64_t dims[3] = {uint64_t(D), uint64_t(s.Hq), uint64_t(n_rows)};
        const uint64_t strides[2] = {uint64_t(D) * 2, uint64_t(s.Hq) * D * 2};
        const uint32_t box[3] = {64u, uint32_t(HPG), 1u};
        if (!encode_tensor_map(&qm, 3, q, dims, strides, box, 128, &why)) return cudaErrorInvalidValue;
    }
    {
        const uint64_t dims[4] = {uint64_t(D), uint64_t(s.G), 128ull, uint64_t(n_pages)};
        const uint64_t strides[3] = {uint64_t(D) * 2, uint64_t(s.G) * D * 2, 128ull * s.G * D * 2};
        const uint32_t box[4] = {64u, 1u, 128u, 1u};
        if (!encode_tensor_map(&km, 4, k_cache, dims, strides, box, 128, &why)) return cudaErrorInvalidValue;
        if (!encode_tensor_map(&vm, 4, v_cache, dims, strides, box, 128, &why)) return cudaErrorInvalidValue;
    }
    const long long n_keys = 1LL * s.G * n_req * s.max_blocks;
    if (n_keys > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const size_t smem = sizeof(AttnSmem<D>) + 1024;
    cudaError_t e =
        cudaFuncSetAttribute(k_attn_prefill<D, HPG>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    k_attn_prefill<D, HPG><<<unsigned(n_keys), kThreads, smem, st>>>(
        qm, km, vm, bt, q_req, q_pos, blk_off, blk_ent, n_rows, n_req, n_pages, s.G, s.topk, s.max_blocks,
        s.sm_scale, static_cast<uint16_t *>(o_part), lse_part, err);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_prefill(const void *q, const void *k_cache, const void *v_cache, const int32_t *block_table,
                                const int32_t *q_req, const int32_t *q_pos, const int32_t *blk_off,
                                const int32_t *blk_ent, int n_rows, int n_req, int n_pages, const Shape &s,
                                void *o_part, float *lse_part, int32_t *err, cudaStream_t st) {
#define MSA_AP_CASE(DD, HH)                                                                                  \
    if (s.D == DD && s.hpg == HH)                                                                            \
        return launch_t<DD, HH>(q, k_cache, v_cache, block_table, q_req, q_pos, blk_off, blk_ent, n_rows, n_req, \
                                n_pages, s, o_part, lse_part, err, st);
    MSA_AP_CASE(128, 8) MSA_AP_CASE(128, 4) MSA_AP_CASE(64, 8) MSA_AP_CASE(64, 4)
#undef MSA_AP_CASE
    return cudaErrorNotSupported;
}

}  // namespace msa
