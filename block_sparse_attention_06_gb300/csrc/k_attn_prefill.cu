// KV-block-major sparse attention for prefill on the 5th-generation tensor cores.
//
// "Together AI 解析如何高效服务 MiniMax M3…", section KV 块主序稀疏注意力: several
// queries attend the same KV block, so looping over KV blocks outside and over
// the queries that selected them inside moves each block from HBM once; the page
// "NVIDIA 加速インフラ上で MiniMax M3 を…" (MSA paragraph after Table 1) states the
// same operator property.  Each block yields a partial O per (query, head) that
// is later combined by a Log-Sum-Exp reduction.
//
// Work.  A CSR key (KV group g, request, logical block j) lists the (query,
// slot) entries that selected block j.  A tile is 128/HPG consecutive entries of
// one key times the HPG query heads of group g = 128 rows of the tensor-core M
// dimension.  A plan kernel cuts every key into chunks of at most kChunkTiles
// tiles; the attention kernel runs one persistent CTA per SM that takes chunks
// from an atomic counter in key order, so a block selected by thousands of
// queries is spread over many SMs while its K/V stays in L2.
//
// One CTA (11 warps):
//   warp 0     decoder: takes chunks, loads K_j and V_j by TMA (128B swizzle,
//              64-column boxes) into one of two K/V buffers, and decodes a whole
//              chunk's entries (query row, slot, causal limit) at once, four per
//              lane with the loads batched, into a ring of tile descriptors;
//   warp 10    Q loader: per described tile, gathers the HPG heads of each
//              entry's query row by TMA into one of two Q buffers as soon as the
//              buffer is free, then hands the descriptor to the consumers;
//   warp 1     TMEM owner and MMA issuer: S = Q K^T (M = 128, N = 128 tokens,
//              K = D) into the S buffer of the tile's softmax group, then, once P
//              is back in TMEM, O = P V with P as the TMEM A operand and V as an
//              MN-major shared-memory B operand;
//   warps 2-5, 6-9  two softmax groups that take alternate tiles: tcgen05.ld of
//              S (thread = row), causal mask, exp2 softmax, P as packed bf16
//              written over S (tcgen05.st), then tcgen05.ld of O, normalisation,
//              bf16 partial and lse stores.  Partials are written in CSR-entry
//              order: a tile's output rows are one contiguous block.  While one group runs its softmax
//              the tensor core works on the other group's tile.
// TMEM: S0 | S1 | O0 | O1 (128 + 128 + D + D of 512 columns).
// Every wait is bounded; a timeout raises MSA_FLAG_TIMEOUT and every role drains.
#include "msa_device.cuh"
#include "msa_internal.h"

namespace msa {
namespace {

constexpr int kThreads = 352;
constexpr int kChunkTiles = 8;   // tiles per work chunk
constexpr int kRing = 16;        // tile descriptors in flight (two chunks)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

constexpr int kFlagKv1 = 1;      // K/V buffer 1 (else 0)
constexpr int kFlagFirst = 2;    // first tile of its chunk
constexpr int kFlagLast = 4;     // last tile of its chunk
constexpr int kFlagEnd = 8;      // no more work

struct TileDesc {
    int32_t flags;
    int32_t g;
    int32_t ent0;      // CSR index of the tile's first entry (its output goes to partial rows ent0 ..)
    int32_t qq[32];    // query row of each entry, -1 for padding / rejected entries
    int32_t slot[32];  // selection slot of the entry
    int32_t lim[32];   // tokens t <= lim of the block are visible to the entry
};

template <int D>
struct AttnSmem {
    alignas(1024) uint8_t k[2][D * 128 * 2];
    alignas(1024) uint8_t v[2][D * 128 * 2];
    alignas(1024) uint8_t q[2][128 * D * 2];
    TileDesc desc[kRing];
    uint64_t kv_full[2], kv_empty[2];
    uint64_t q_full[2], q_empty[2];
    uint64_t s_full[2], p_full[2], o_full[2], o_free[2];
    uint64_t desc_ready[kRing], desc_full[kRing], desc_empty[kRing];
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};

// 2^x by the MUFU.EX2 hardware approximation (PTX ex2.approx.ftz.f32; relative
// error about 2^-22, far below the bf16 rounding of P); 2^-inf = +0.
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Work-list header in the workspace: [0] next chunk (atomic), [1] chunk count.
constexpr size_t kPlanHeaderBytes = 16;

__host__ __device__ inline long long max_chunks_of(long long n_keys, long long n_entries, int ept) {
    const long long per_chunk = static_cast<long long>(ept) * kChunkTiles;
    return n_keys + (n_entries + per_chunk - 1) / per_chunk;
}

// ------------------------------------------------------------------ plan
//
// One CTA: chunk counts per key (ceil(ceil(n/EPT)/kChunkTiles)), an exclusive
// scan, and the chunk list {key, first tile} in key order.
__global__ void __launch_bounds__(1024) k_attn_plan(const int32_t *__restrict__ blk_off, int n_keys, int ept,
                                                    long long max_chunks, int32_t *__restrict__ hdr,
                                                    int2 *__restrict__ chunks, int32_t *err) {
    __shared__ int32_t wsum[32];
    __shared__ long long carry_s;
    pdl_trigger();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) carry_s = 0;
    __syncthreads();
    for (int base = 0; base < n_keys; base += 1024) {
        const int k = base + tid;
        int nc = 0;
        if (k < n_keys) {
            const int n = blk_off[k + 1] - blk_off[k];
            if (n < 0) {
                raise_flag(err, MSA_FLAG_BOUNDS);
            } else {
                const int nt = (n + ept - 1) / ept;
                nc = (nt + kChunkTiles - 1) / kChunkTiles;
            }
        }
        int x = nc;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) wsum[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int w = wsum[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += y;
            }
            wsum[lane] = w;
        }
        __syncthreads();
        const long long start = carry_s + (warp ? wsum[warp - 1] : 0) + x - nc;
        for (int i = 0; i < nc; ++i) {
            if (start + i < max_chunks) chunks[start + i] = make_int2(k, i * kChunkTiles);
            else raise_flag(err, MSA_FLAG_BOUNDS);
        }
        __syncthreads();
        if (tid == 1023) carry_s = start + nc;
        __syncthreads();
    }
    if (tid == 0) {
        hdr[0] = 0;
        hdr[1] = int32_t(carry_s < max_chunks ? carry_s : max_chunks);
    }
}

// ------------------------------------------------------------------ attention

template <int D, int HPG>
__global__ void __launch_bounds__(kThreads, 1) k_attn_prefill(
    const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
    const __grid_constant__ CUtensorMap vmap, const int32_t *__restrict__ block_table,
    const int32_t *__restrict__ q_req, const int32_t *__restrict__ q_pos, const int32_t *__restrict__ blk_off,
    const int32_t *__restrict__ blk_ent, int32_t *__restrict__ plan_hdr, const int2 *__restrict__ chunks,
    int n_rows, int n_req, int n_pages, int G, int topk, int max_blocks, float sm_scale,
    uint16_t *__restrict__ o_part, float *__restrict__ lse_part, int32_t *err) {
    constexpr int EPT = 128 / HPG;                 // entries per tile
    constexpr int NSUB = D / 64;                   // 64-column sub-tiles
    constexpr uint32_t kIdescS = make_idesc_bf16(128, 128, 0, 0);
    constexpr uint32_t kIdescO = make_idesc_bf16(128, D, 0, 1);
    extern __shared__ uint8_t smem_raw[];
    AttnSmem<D> &sm =
        *reinterpret_cast<AttnSmem<D> *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const long long cap = 1LL * n_rows * G * topk;

    if (tid == 0) {
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sm.kv_full[b], 1);
            mbar_init(&sm.kv_empty[b], 1);
            mbar_init(&sm.q_full[b], 1);
            mbar_init(&sm.q_empty[b], 1);
            mbar_init(&sm.s_full[b], 1);
            mbar_init(&sm.p_full[b], 4);
            mbar_init(&sm.o_full[b], 1);
            mbar_init(&sm.o_free[b], 4);
        }
        for (int r = 0; r < kRing; ++r) {
            mbar_init(&sm.desc_ready[r], 32);
            mbar_init(&sm.desc_full[r], 32);
            mbar_init(&sm.desc_empty[r], 5);
        }
        mbar_init(&sm.drain, 1);
        sm.abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&sm.tmem_base, 512);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&qmap);
        tma_prefetch_desc(&kmap);
        tma_prefetch_desc(&vmap);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;

    if (warp == 0) {
        // ------------------------------------------------------------ decoder
        constexpr int ENT_MAX = kChunkTiles * EPT;   // entries of a full chunk
        constexpr int PER_LANE = ENT_MAX / 32;
        pdl_wait();   // the work list and the CSR come from the preceding kernels
        const int n_chunks = plan_hdr[1];
        const int per_g = n_req * max_blocks;
        auto claim = [&]() {
            int v = 0;
            if (lane == 0) v = atomicAdd(plan_hdr, 1);
            return __shfl_sync(0xffffffffu, v, 0);
        };
        int u = 0;          // tiles described
        int cs = 0;         // chunks whose K/V were loaded
        bool ok = true;
        int c = claim();
        int2 ch = c < n_chunks ? chunks[c] : make_int2(0, 0);
        while (ok && c < n_chunks) {
            const int cn = claim();                                   // next chunk, header in flight
            const int2 chn = cn < n_chunks ? chunks[cn] : make_int2(0, 0);
            const int key = ch.x, t0 = ch.y;
            const int g = key / per_g;
            const int req = (key - g * per_g) / max_blocks;
            const int j = key - g * per_g - req * max_blocks;
            const int off0 = blk_off[key], end0 = blk_off[key + 1];
            const int page = block_table[size_t(req) * max_blocks + j];
            c = cn;
            ch = chn;
            if (off0 < 0 || end0 > cap || off0 > end0 || page < 0 || page >= n_pages || g >= G) {
                if (lane == 0) raise_flag(err, MSA_FLAG_BOUNDS);
                continue;
            }
            const int off = off0 + t0 * EPT;
            const int end = min(end0, off + ENT_MAX);
            if (off >= end) continue;
            const int nt = (end - off + EPT - 1) / EPT;
            const int kvb = cs & 1;
            if (cs >= 2) {
                bool w = true;
                if (lane == 0) w = mbar_wait(&sm.kv_empty[kvb], ((cs >> 1) - 1) & 1, err, &sm.abort);
                if (!__shfl_sync(0xffffffffu, w, 0)) {
                    ok = false;
                    break;
                }
            }
            if (lane == 0) {
                mbar_arrive_expect_tx(&sm.kv_full[kvb], 2 * D * 128 * 2);
#pragma unroll
                for (int i = 0; i < NSUB; ++i)
                    tma_load_4d(sm.k[kvb] + i * 16384, &kmap, &sm.kv_full[kvb], i * 64, g, 0, page);
#pragma unroll
                for (int i = 0; i < NSUB; ++i)
                    tma_load_4d(sm.v[kvb] + i * 16384, &vmap, &sm.kv_full[kvb], i * 64, g, 0, page);
            }
            ++cs;
            // decode the chunk's entries: all loads of a lane's PER_LANE entries are issued together
            int ent[PER_LANE];
#pragma unroll
            for (int r = 0; r < PER_LANE; ++r) {
                const int idx = off + lane + 32 * r;
                ent[r] = idx < end ? blk_ent[idx] : -1;
            }
            int rq[PER_LANE], ps[PER_LANE];
#pragma unroll
            for (int r = 0; r < PER_LANE; ++r) {
                const int v = ent[r] / topk;
                const bool in = ent[r] >= 0 && v < n_rows;
                rq[r] = in ? q_req[v] : -1;
                ps[r] = in ? q_pos[v] : -1;
            }
            // the ring slots of this chunk's tiles must be free
            for (int t = 0; t < nt; ++t) {
                const int ut = u + t;
                if (ut >= kRing) {
                    bool w = true;
                    if (lane == 0) w = mbar_wait(&sm.desc_empty[ut % kRing], ((ut / kRing) - 1) & 1, err, &sm.abort);
                    if (!__shfl_sync(0xffffffffu, w, 0)) {
                        ok = false;
                        break;
                    }
                }
            }
            if (!ok) break;
#pragma unroll
            for (int r = 0; r < PER_LANE; ++r) {
                const int i = lane + 32 * r;
                if (i < nt * EPT) {
                    const int idx = off + i;
                    int qq = -1, sl = 0, lim = -1;
                    if (idx < end) {
                        const int v = ent[r] / topk;
                        if (ent[r] < 0 || v >= n_rows || rq[r] != req) {
                            raise_flag(err, MSA_FLAG_BOUNDS);
                        } else {
                            lim = ps[r] - j * 128;
                            if (lim < 0) {   // block past the row's position: not a candidate
                                raise_flag(err, MSA_FLAG_BOUNDS);
                            } else {
                                qq = v;
                                sl = ent[r] - v * topk;
                            }
                        }
                    }
                    TileDesc &d = sm.desc[(u + i / EPT) % kRing];
                    d.qq[i % EPT] = qq;
                    d.slot[i % EPT] = sl;
                    d.lim[i % EPT] = lim;
                }
            }
            if (lane < nt) {
                TileDesc &d = sm.desc[(u + lane) % kRing];
                d.flags = (kvb ? kFlagKv1 : 0) | (lane == 0 ? kFlagFirst : 0) | (lane == nt - 1 ? kFlagLast : 0);
                d.g = g;
                d.ent0 = off + lane * EPT;
            }
            for (int t = 0; t < nt; ++t) mbar_arrive(&sm.desc_ready[(u + t) % kRing]);
            u += nt;
        }
        // two end markers, one for each softmax group (the MMA warp stops at the first)
        for (int e = 0; ok && e < 2; ++e) {
            const int slot = u % kRing;
            if (u >= kRing) {
                bool w = true;
                if (lane == 0) w = mbar_wait(&sm.desc_empty[slot], ((u / kRing) - 1) & 1, err, &sm.abort);
                if (!__shfl_sync(0xffffffffu, w, 0)) break;
            }
            if (lane == 0) sm.desc[slot].flags = kFlagEnd;
            mbar_arrive(&sm.desc_ready[slot]);
            ++u;
        }
        if (sm.abort && lane == 0) {
            // drain: the K/V copies still in flight land before the CTA exits
            for (int t = max(0, cs - 2); t < cs; ++t) mbar_wait(&sm.kv_full[t & 1], (t >> 1) & 1, err, nullptr);
        }
    } else if (warp == 10) {
        // ------------------------------------------------------------ Q loader
        int n_q = 0;        // tiles whose Q copies were issued
        int ends = 0;
        for (int u = 0; ends < 2; ++u) {
            const int slot = u % kRing;
            // every lane waits (acquires) before it reads the descriptor
            bool w = __all_sync(0xffffffffu, mbar_wait(&sm.desc_ready[slot], (u / kRing) & 1, err, &sm.abort));
            if (!w) break;
            const volatile TileDesc &d = sm.desc[slot];
            if (d.flags & kFlagEnd) {
                ++ends;
                mbar_arrive(&sm.desc_full[slot]);
                continue;
            }
            const int qb = n_q & 1;
            if (n_q >= 2) {
                if (lane == 0) w = mbar_wait(&sm.q_empty[qb], ((n_q >> 1) - 1) & 1, err, &sm.abort);
                if (!__shfl_sync(0xffffffffu, w, 0)) break;
            }
            const int g = d.g;
            const int qq = lane < EPT ? d.qq[lane] : -1;
            if (lane == 0) mbar_arrive_expect_tx(&sm.q_full[qb], 128 * D * 2);
            __syncwarp();
            if (lane < EPT) {
                const int row = qq >= 0 ? qq : n_rows;   // fully out of bounds -> zero rows
#pragma unroll
                for (int i = 0; i < NSUB; ++i)
                    tma_load_3d(sm.q[qb] + i * 16384 + lane * HPG * 128, &qmap, &sm.q_full[qb], i * 64, g * HPG,
                                row);
            }
            ++n_q;
            mbar_arrive(&sm.desc_full[slot]);
        }
        if (sm.abort && lane == 0) {
            // drain: the Q copies still in flight land before the CTA exits
            for (int t = max(0, n_q - 2); t < n_q; ++t) mbar_wait(&sm.q_full[t & 1], (t >> 1) & 1, err, nullptr);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int u = 0, cs = -1;
            bool have_prev = false;
            int p_u = 0, p_flags = 0;
            auto do_pv = [&](int t, int flags) -> bool {
                const int b = t & 1;
                if (!mbar_wait(&sm.p_full[b], (t >> 1) & 1, err, &sm.abort)) return false;
                if (t >= 2 && !mbar_wait(&sm.o_free[b], ((t >> 1) - 1) & 1, err, &sm.abort)) return false;
                tc_fence_after();
                const int kvb = flags & kFlagKv1;
                const uint32_t v_addr = smem_u32(sm.v[kvb]);
#pragma unroll
                for (int kt = 0; kt < 8; ++kt) {
                    const uint64_t bd = make_smem_desc(v_addr + uint32_t(kt * 2048), 16384, 1024, 2);
                    mma_bf16_ts(tmem + uint32_t(256 + b * D), tmem + uint32_t(b * 128 + kt * 8), bd, kIdescO,
                                kt > 0 ? 1u : 0u);
                }
                mma_commit(&sm.o_full[b]);
                if (flags & kFlagLast) mma_commit(&sm.kv_empty[kvb]);
                return true;
            };
            for (;;) {
                const int slot = u % kRing;
                if (!mbar_wait(&sm.desc_full[slot], (u / kRing) & 1, err, &sm.abort)) break;
                const int flags = *reinterpret_cast<volatile int32_t *>(&sm.desc[slot].flags);
                if (flags & kFlagEnd) break;
                mbar_arrive(&sm.desc_empty[slot]);
                const int kvb = flags & kFlagKv1;
                if (flags & kFlagFirst) {
                    ++cs;
                    if (!mbar_wait(&sm.kv_full[kvb], (cs >> 1) & 1, err, &sm.abort)) break;
                }
                const int b = u & 1;
                if (!mbar_wait(&sm.q_full[b], (u >> 1) & 1, err, &sm.abort)) break;
                tc_fence_after();
                const uint32_t q_addr = smem_u32(sm.q[b]), k_addr = smem_u32(sm.k[kvb]);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t o = uint32_t((kk >> 2) * 16384 + (kk & 3) * 32);
                    mma_bf16(tmem + uint32_t(b * 128), make_smem_desc(q_addr + o, 16, 1024, 2),
                             make_smem_desc(k_addr + o, 16, 1024, 2), kIdescS, kk > 0 ? 1u : 0u);
                }
                mma_commit(&sm.s_full[b]);
                mma_commit(&sm.q_empty[b]);
                if (have_prev && !do_pv(p_u, p_flags)) {
                    have_prev = false;
                    break;
                }
                have_prev = true;
                p_u = u;
                p_flags = flags;
                ++u;
            }
            if (have_prev && !sm.abort) do_pv(p_u, p_flags);
            mma_commit(&sm.drain);
            mbar_wait(&sm.drain, 0, err, nullptr);
        }
    } else if (warp >= 2 && warp < 10) {
        // ------------------------------------------------------------ softmax groups
        const int wg = (warp - 2) >> 2;
        const int quad = warp & 3;                 // TMEM lanes this warp may access
        const int row = quad * 32 + lane;
        const int e = row / HPG, h = row - (row / HPG) * HPG;
        const uint32_t lane_off = uint32_t(quad * 32) << 16;
        const uint32_t t_s = tmem + lane_off + uint32_t(wg * 128);
        const uint32_t t_o = tmem + lane_off + uint32_t(256 + wg * D);
        const float scale = sm_scale * kLog2e;
        for (int u = wg;; u += 2) {
            const int slot = u % kRing;
            const int k = u >> 1;
            if (!__all_sync(0xffffffffu, mbar_wait(&sm.desc_full[slot], (u / kRing) & 1, err, &sm.abort))) break;
            const volatile TileDesc &d = sm.desc[slot];
            if (d.flags & kFlagEnd) break;
            const int qq = d.qq[e];
            const int idx = d.ent0 + e;                  // CSR entry of this row
            const int lim = qq >= 0 ? d.lim[e] : 127;   // padding rows: any finite softmax, never stored
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.desc_empty[slot]);

            if (!__all_sync(0xffffffffu, mbar_wait(&sm.s_full[wg], k & 1, err, &sm.abort))) break;
            tc_fence_after();
            float s[128];
            {
                uint32_t v[4][32];
#pragma unroll
                for (int c = 0; c < 4; ++c) tmem_ld32(t_s + uint32_t(c * 32), v[c]);
                tmem_ld_wait();
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int i = 0; i < 32; ++i) s[c * 32 + i] = __uint_as_float(v[c][i]);
            }
            // row max as eight independent chains
            float mx[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) mx[i] = -INFINITY;
            if (lim >= 127) {
#pragma unroll
                for (int c = 0; c < 128; ++c) mx[c & 7] = fmaxf(mx[c & 7], s[c]);
            } else {
#pragma unroll
                for (int c = 0; c < 128; ++c) {
                    s[c] = c <= lim ? s[c] : -INFINITY;
                    mx[c & 7] = fmaxf(mx[c & 7], s[c]);
                }
            }
            const float m = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                  fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
            const float ms = m * scale;
            // probabilities 2^(s*scale - ms) as packed bf16 into TMEM; their fp32 sum in eight
            // chains normalises O and gives the lse
            float acc[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll
            for (int c0 = 0; c0 < 128; c0 += 64) {
                uint32_t w[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const float pa = fast_exp2(fmaf(s[c0 + 2 * i], scale, -ms));
                    const float pb = fast_exp2(fmaf(s[c0 + 2 * i + 1], scale, -ms));
                    w[i] = pack_bf16x2(pa, pb);
                    acc[i & 7] += pa + pb;
                }
                tmem_st32(t_s + uint32_t(c0 >> 1), w);
            }
            const float le = ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.p_full[wg]);

            if (!__all_sync(0xffffffffu, mbar_wait(&sm.o_full[wg], k & 1, err, &sm.abort))) break;
            tc_fence_after();
            uint32_t ov[D / 32][32];
#pragma unroll
            for (int c = 0; c < D / 32; ++c) tmem_ld32(t_o + uint32_t(c * 32), ov[c]);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.o_free[wg]);
            if (qq >= 0) {
                const float inv = 1.0f / le;
                const size_t unit = size_t(idx) * HPG + h;
                uint16_t *dst = o_part + unit * D;
#pragma unroll
                for (int i = 0; i < D; i += 8) {
                    const uint32_t *o8 = &ov[i >> 5][i & 31];
                    uint4 w;
                    w.x = pack_bf16x2(__uint_as_float(o8[0]) * inv, __uint_as_float(o8[1]) * inv);
                    w.y = pack_bf16x2(__uint_as_float(o8[2]) * inv, __uint_as_float(o8[3]) * inv);
                    w.z = pack_bf16x2(__uint_as_float(o8[4]) * inv, __uint_as_float(o8[5]) * inv);
                    w.w = pack_bf16x2(__uint_as_float(o8[6]) * inv, __uint_as_float(o8[7]) * inv);
                    *reinterpret_cast<uint4 *>(dst + i) = w;
                }
                lse_part[unit] = (ms + log2f(le)) * kLn2;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

struct PlanLayout {
    long long max_chunks;
    size_t bytes;
};

inline PlanLayout plan_layout(int n_rows, int n_req, const Shape &s) {
    const long long n_keys = 1LL * s.G * n_req * s.max_blocks;
    const long long n_ent = 1LL * n_rows * s.G * s.topk;
    PlanLayout p;
    p.max_chunks = max_chunks_of(n_keys, n_ent, 128 / s.hpg);
    p.bytes = kPlanHeaderBytes + size_t(p.max_chunks) * sizeof(int2);
    return p;
}

template <int D, int HPG>
cudaError_t launch_t(const void *q, const void *k_cache, const void *v_cache, const int32_t *bt, const int32_t *q_req,
                     const int32_t *q_pos, const int32_t *blk_off, const int32_t *blk_ent, int n_rows, int n_req,
                     int n_pages, const Shape &s, void *o_part, float *lse_part, void *ws, int32_t *err,
                     cudaStream_t st) {
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
    if (n_keys > 0x7ffffffeLL) return cudaErrorInvalidConfiguration;
    const PlanLayout pl = plan_layout(n_rows, n_req, s);
    int32_t *hdr = static_cast<int32_t *>(ws);
    int2 *chunks = reinterpret_cast<int2 *>(static_cast<uint8_t *>(ws) + kPlanHeaderBytes);
    cudaError_t e = launch_kernel(k_attn_plan, dim3(1), dim3(1024), 0, st, false, blk_off, int(n_keys), 128 / HPG,
                                  pl.max_chunks, hdr, chunks, err);
    if (e != cudaSuccess) return e;
    const size_t smem = sizeof(AttnSmem<D>) + 1024;
    e = cudaFuncSetAttribute(k_attn_prefill<D, HPG>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    return launch_kernel(k_attn_prefill<D, HPG>, dim3(unsigned(sm_count())), dim3(kThreads), smem, st, true, qm, km,
                         vm, bt, q_req, q_pos, blk_off, blk_ent, hdr, static_cast<const int2 *>(chunks), n_rows, n_req,
                         n_pages, s.G, s.topk, s.max_blocks, s.sm_scale, static_cast<uint16_t *>(o_part), lse_part,
                         err);
}

}  // namespace

size_t prefill_workspace_bytes(int n_rows, int n_req, const Shape &s) { return plan_layout(n_rows, n_req, s).bytes; }

cudaError_t launch_attn_prefill(const void *q, const void *k_cache, const void *v_cache, const int32_t *block_table,
                                const int32_t *q_req, const int32_t *q_pos, const int32_t *blk_off,
                                const int32_t *blk_ent, int n_rows, int n_req, int n_pages, const Shape &s,
                                void *o_part, float *lse_part, void *ws, int32_t *err, cudaStream_t st) {
#define MSA_AP_CASE(DD, HH)                                                                                  \
    if (s.D == DD && s.hpg == HH)                                                                            \
        return launch_t<DD, HH>(q, k_cache, v_cache, block_table, q_req, q_pos, blk_off, blk_ent, n_rows, n_req, \
                                n_pages, s, o_part, lse_part, ws, err, st);
    MSA_AP_CASE(128, 8) MSA_AP_CASE(128, 4) MSA_AP_CASE(64, 8) MSA_AP_CASE(64, 4)
#undef MSA_AP_CASE
    return cudaErrorNotSupported;
}

}  // namespace msa
