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
// queries is spread over many SMs while its K/V stays in L2.  Partials are
// written in CSR-entry order, so the output of one tile is one contiguous block.
//
// One CTA (19 warps):
//   warp 0     decoder: takes chunks, warms L2 with their K_j and V_j, hands
//              each chunk to the K/V loader, and decodes a whole chunk's entries
//              (query row, slot, causal limit) at once, with the loads batched,
//              into a ring of tile descriptors;
//   warp 1     TMEM owner and MMA issuer: S = Q K^T (M = 128, N = 128 tokens,
//              K = D) into the S buffer of the tile's softmax group, then, once P
//              is back in TMEM, O = P V with P as the TMEM A operand and V as an
//              MN-major shared-memory B operand.  Warps share a sub-partition's
//              issue slots by warp index mod 4, and an MMA issuer that competes
//              with busy warps feeds the tensor core at a fraction of its rate:
//              sub-partition 1 holds only this warp and one warp of each softmax
//              group and of the epilogue (those must cover all four TMEM lane
//              quarters), and each group of MMAs is issued from one asm block.
//              The tensor core takes an MMA about when the one before it ends, so
//              the issuer's own waits are idle tensor time: per tile it waits on
//              the Q buffer (whose loader has read the tile's descriptor first, so
//              the flags can be read after it), on K or V at a chunk's start, and
//              for the previous tile's PV twice: once for P of tokens 0..63 and the
//              O buffer (the first four MMAs), once for the rest of P;
//   warp 2     K/V loader: K_j by TMA (128B swizzle, 64-column boxes) once the
//              previous chunk's last S has completed, V_j once its last PV has;
//   warps 4-7, 8-11  two softmax groups that take alternate tiles: S is read
//              from TMEM in 32-column chunks twice (row max, then exp2 and P as
//              packed bf16 written over S, signalled after the first 64 tokens
//              and again at the end); the row's 1/sum goes to a four-slot
//              ring in shared memory (so a group never waits for the epilogue to
//              read the previous one) and its lse to the partials; while one group
//              runs its softmax the tensor core works on the other group's tile;
//   warps 12-15  epilogue: every tile in order, O chunk by chunk from TMEM,
//              normalised, and stored from registers, so a softmax group goes on
//              to its next tile as soon as its P is in TMEM.  The partials are
//              laid out for these stores: within each entry's HPG x D block the
//              16-byte column chunk is the outer index and the head the inner one,
//              so the 32 rows of a warp (4 entries x 8 heads, or 8 x 4), one per
//              lane, write whole 128-byte lines per store instruction.  No staging
//              buffer, no TMA store, and no shared-memory traffic for the output;
//   warp 17    idle (it would share the MMA warp's sub-partition);
//   warps 16, 3, 18  Q loaders, one per Q buffer, one tile each in turn: the HPG
//              heads of each entry's query row (HPG * D * 2 contiguous bytes) in
//              the 128B-swizzled layout the MMA reads.  With HPG = 8 an entry's
//              heads fill whole 1024-byte swizzle atoms, so one TMA box of 64
//              columns x 8 heads per entry and sub-tile moves them (a query row of
//              -1, padding, reads the zero fill): 16 instructions of one lane per
//              tile instead of 512 cp.async, which leaves the loaders' issue slots
//              to the softmax and epilogue warps on their sub-partitions.  With
//              HPG = 4 a box would cover half an atom, so the warp copies the rows
//              by 16-byte cp.async.  A buffer has one loader, so its barriers'
//              phases are waited in order.
// TMEM: S0 | S1 | O0 | O1 (128 + 128 + D + D of 512 columns).
// Every wait is bounded; a timeout raises MSA_FLAG_TIMEOUT and every role drains.
#include "msa_device.cuh"
#include "msa_internal.h"

namespace msa {
namespace {

constexpr int kThreads = 608;
constexpr int kChunkTiles = 8;   // tiles per work chunk
constexpr int kRing = 16;        // tile descriptors in flight (two chunks)
constexpr int kQBuf = 3;         // Q buffers
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

constexpr int kFlagFirst = 2;    // first tile of its chunk
constexpr int kFlagLast = 4;     // last tile of its chunk
constexpr int kFlagEnd = 8;      // no more work

struct TileDesc {
    int32_t flags;
    int32_t g;
    int32_t ent0;      // CSR index of the tile's first entry (its output goes to partial rows ent0 ..)
    int32_t n_valid;   // entries of this tile that exist (the rest is padding)
    int32_t qq[32];    // query row of each entry, -1 for padding / rejected entries
    int32_t slot[32];  // selection slot of the entry
    int32_t lim[32];   // tokens t <= lim of the block are visible to the entry
};

template <int D>
struct AttnSmem {
    alignas(1024) uint8_t k[D * 128 * 2];
    alignas(1024) uint8_t v[D * 128 * 2];
    alignas(1024) uint8_t q[kQBuf][128 * D * 2];
    TileDesc desc[kRing];
    float inv_le[4][128];                           // 1 / row sum of P, per tile mod 4 (softmax -> epilogue)
    int32_t chunk_page[4], chunk_g[4];              // decoder -> K/V loader
    uint64_t k_full, k_empty, v_full, v_empty;
    uint64_t q_full[kQBuf], q_empty[kQBuf];
    uint64_t s_full[2], o_full[2];
    uint64_t p_lo[2];       // P of tokens 0..63 written (softmax group) and the O buffer read out (epilogue)
    uint64_t pv_ready[2];   // all of P written by the tile's softmax group
    uint64_t stat_full[4], stat_free[4];            // inv_le[i] written / read by the epilogue
    uint64_t desc_ready[kRing], desc_full[kRing], desc_empty[kRing];
    uint64_t chunk_ready[4], chunk_free[4];
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

// Two fp32 lanes per instruction (the f32x2 datapath of sm_100-class SMs); b2 / c2 hold one value
// in both halves.
__device__ __forceinline__ uint64_t dup2(float x) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %1};" : "=l"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ void ffma2(float &d0, float &d1, float a0, float a1, uint64_t b2, uint64_t c2) {
    asm("{\n\t.reg .b64 x, d;\n\tmov.b64 x, {%2, %3};\n\tfma.rn.f32x2 d, x, %4, %5;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "l"(b2), "l"(c2));
}
__device__ __forceinline__ void fmul2(float &d0, float &d1, float a0, float a1, uint64_t b2) {
    asm("{\n\t.reg .b64 x, d;\n\tmov.b64 x, {%2, %3};\n\tmul.rn.f32x2 d, x, %4;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "l"(b2));
}
// acc2 += (a0, a1), lane-wise
__device__ __forceinline__ void fadd2_acc(uint64_t &acc2, float a0, float a1) {
    asm("{\n\t.reg .b64 x;\n\tmov.b64 x, {%1, %2};\n\tadd.rn.f32x2 %0, %0, x;\n\t}" : "+l"(acc2) : "f"(a0), "f"(a1));
}
__device__ __forceinline__ float sum2(uint64_t acc2) {
    float a, b;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(acc2));
    return a + b;
}

// KSTEPS MMAs of S = Q K^T (M = N = 128, K = 16 each), A and B K-major 128B-swizzled: the k-step
// advances 32 bytes within a 64-column sub-tile and 16 KB between sub-tiles, i.e. +2 / +1024 in the
// descriptors' 16-byte address units.  Issued by the threads with `leader` set (one thread).  The
// first MMA overwrites D, the others accumulate.
template <int KSTEPS>
__device__ __forceinline__ void mma_s_block(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t leader) {
    static_assert(KSTEPS == 4 || KSTEPS == 8, "D of 64 or 128");
    if constexpr (KSTEPS == 8) {
        asm volatile(
            "{\n\t.reg .pred f, t, e;\n\t.reg .b64 a1, a2, a3, a4, a5, a6, a7, b1, b2, b3, b4, b5, b6, b7;\n\t"
            "setp.ne.b32 e, %4, 0;\n\tsetp.ne.b32 f, %4, %4;\n\tsetp.eq.b32 t, %4, %4;\n\t"
            "add.s64 a1, %1, 2;\n\tadd.s64 a2, %1, 4;\n\tadd.s64 a3, %1, 6;\n\tadd.s64 a4, %1, 1024;\n\t"
            "add.s64 a5, %1, 1026;\n\tadd.s64 a6, %1, 1028;\n\tadd.s64 a7, %1, 1030;\n\t"
            "add.s64 b1, %2, 2;\n\tadd.s64 b2, %2, 4;\n\tadd.s64 b3, %2, 6;\n\tadd.s64 b4, %2, 1024;\n\t"
            "add.s64 b5, %2, 1026;\n\tadd.s64 b6, %2, 1028;\n\tadd.s64 b7, %2, 1030;\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, f;\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, t;\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a2, b2, %3, t;\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a3, b3, %3, t;\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a4, b4, %3, t;\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a5, b5, %3, t;\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a6, b6, %3, t;\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a7, b7, %3, t;\n\t}" ::"r"(d),
            "l"(a), "l"(b), "r"(idesc), "r"(leader)
            : "memory");
    } else {
        asm volatile(
            "{\n\t.reg .pred f, t, e;\n\t.reg .b64 a1, a2, a3, b1, b2, b3;\n\t"
            "setp.ne.b32 e, %4, 0;\n\tsetp.ne.b32 f, %4, %4;\n\tsetp.eq.b32 t, %4, %4;\n\t"
            "add.s64 a1, %1, 2;\n\tadd.s64 a2, %1, 4;\n\tadd.s64 a3, %1, 6;\n\t"
            "add.s64 b1, %2, 2;\n\tadd.s64 b2, %2, 4;\n\tadd.s64 b3, %2, 6;\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, f;\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, t;\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a2, b2, %3, t;\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a3, b3, %3, t;\n\t}" ::"r"(d),
            "l"(a), "l"(b), "r"(idesc), "r"(leader)
            : "memory");
    }
}

// 16-byte global store with an L2 cache policy (l2_policy_evict_first and the like).
__device__ __forceinline__ void st_global_v4_hint(void *p, const uint32_t (&w)[4], uint64_t policy) {
    asm volatile("st.global.L2::cache_hint.v4.b32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "r"(w[0]), "r"(w[1]),
                 "r"(w[2]), "r"(w[3]), "l"(policy)
                 : "memory");
}

__device__ __forceinline__ int sm_flags(const TileDesc &d) {
    return *reinterpret_cast<const volatile int32_t *>(&d.flags);
}

// Four MMAs of O = P V (64 tokens): A = P in TMEM at columns a, a + 8, a + 16, a + 24; B = V at
// descriptors b, b + 128, b + 256, b + 384.  The first overwrites D when acc == 0.
__device__ __forceinline__ void mma_pv_half(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p, t;\n\t.reg .b64 b1, b2, b3;\n\t.reg .b32 a1, a2, a3;\n\t"
        "setp.ne.b32 p, %4, 0;\n\tsetp.eq.b32 t, %4, %4;\n\t"
        "add.s32 a1, %1, 8;\n\tadd.s32 a2, %1, 16;\n\tadd.s32 a3, %1, 24;\n\t"
        "add.s64 b1, %2, 128;\n\tadd.s64 b2, %2, 256;\n\tadd.s64 b3, %2, 384;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %3, t;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a2], b2, %3, t;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a3], b3, %3, t;\n\t}" ::"r"(d),
        "r"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
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
    const uint8_t *__restrict__ qg, int Hq, const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
    const __grid_constant__ CUtensorMap vmap, uint8_t *__restrict__ o_part,
    const int32_t *__restrict__ block_table, const int32_t *__restrict__ q_req, const int32_t *__restrict__ q_pos,
    const int32_t *__restrict__ blk_off, const int32_t *__restrict__ blk_ent, int32_t *__restrict__ plan_hdr,
    const int2 *__restrict__ chunks, int n_rows, int n_req, int n_pages, int G, int topk, int max_blocks,
    float sm_scale, float *__restrict__ lse_part, int32_t *err) {
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
        for (int b = 0; b < kQBuf; ++b) {
            mbar_init(&sm.q_full[b], 1);
            mbar_init(&sm.q_empty[b], 1);
        }
        mbar_init(&sm.k_full, 1);
        mbar_init(&sm.k_empty, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sm.s_full[b], 1);
            mbar_init(&sm.p_lo[b], 8);       // 4 softmax warps (P, tokens 0..63) + 4 epilogue warps (O)
            mbar_init(&sm.pv_ready[b], 4);   // 4 softmax warps (all of P)
            mbar_init(&sm.o_full[b], 1);
        }
        mbar_init(&sm.v_full, 1);
        mbar_init(&sm.v_empty, 1);
        for (int r = 0; r < 4; ++r) {
            mbar_init(&sm.stat_full[r], 4);
            mbar_init(&sm.stat_free[r], 4);
        }
        for (int r = 0; r < kRing; ++r) {
            mbar_init(&sm.desc_ready[r], 32);
            mbar_init(&sm.desc_full[r], 1);   // the tile's Q loader, once it has read the descriptor
            mbar_init(&sm.desc_empty[r], 9);   // MMA, a softmax group's 4 warps, the epilogue's 4
        }
        for (int r = 0; r < 4; ++r) {
            mbar_init(&sm.chunk_ready[r], 1);
            mbar_init(&sm.chunk_free[r], 1);
        }
        mbar_init(&sm.drain, 1);
        sm.abort = 0;
        for (int b = 0; b < 2; ++b)   // the first tile of each O buffer has no earlier tile to read out
            for (int i = 0; i < 4; ++i) mbar_arrive(&sm.p_lo[b]);
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
        auto wait_lane0 = [&](uint64_t *bar, uint32_t parity) -> bool {
            bool w = true;
            if (lane == 0) w = mbar_wait(bar, parity, err, &sm.abort);
            return __shfl_sync(0xffffffffu, w, 0);
        };
        int u = 0;          // tiles described
        int cs = 0;         // chunks issued
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
            // the K/V loader fetches this block after the chunks before it: warm L2 now
            if (lane == 0) {
#pragma unroll
                for (int i = 0; i < NSUB; ++i) {
                    tma_prefetch_l2_4d(&kmap, i * 64, g, 0, page);
                    tma_prefetch_l2_4d(&vmap, i * 64, g, 0, page);
                }
            }
            if (cs >= 4 && !wait_lane0(&sm.chunk_free[cs & 3], ((cs >> 2) - 1) & 1)) {
                ok = false;
                break;
            }
            if (lane == 0) {
                sm.chunk_page[cs & 3] = page;
                sm.chunk_g[cs & 3] = g;
                mbar_arrive(&sm.chunk_ready[cs & 3]);
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
            for (int t = 0; ok && t < nt; ++t) {
                const int ut = u + t;
                if (ut >= kRing && !wait_lane0(&sm.desc_empty[ut % kRing], ((ut / kRing) - 1) & 1)) ok = false;
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
                d.flags = (lane == 0 ? kFlagFirst : 0) | (lane == nt - 1 ? kFlagLast : 0);
                d.g = g;
                d.ent0 = off + lane * EPT;
                d.n_valid = min(EPT, end - (off + lane * EPT));
            }
            for (int t = 0; t < nt; ++t) mbar_arrive(&sm.desc_ready[(u + t) % kRing]);
            u += nt;
        }
        // end markers: three tiles (one per Q loader, and so one per softmax group; the MMA and epilogue
        // warps stop at the first), one chunk
        for (int e = 0; ok && e < kQBuf; ++e) {
            const int slot = u % kRing;
            if (u >= kRing && !wait_lane0(&sm.desc_empty[slot], ((u / kRing) - 1) & 1)) break;
            if (lane == 0) sm.desc[slot].flags = kFlagEnd;
            mbar_arrive(&sm.desc_ready[slot]);
            ++u;
        }
        if (ok && (cs < 4 || wait_lane0(&sm.chunk_free[cs & 3], ((cs >> 2) - 1) & 1))) {
            if (lane == 0) {
                sm.chunk_page[cs & 3] = -1;
                mbar_arrive(&sm.chunk_ready[cs & 3]);
            }
        }
    } else if (warp == 2) {
        // ------------------------------------------------------------ K/V loader (lane 0)
        if (lane == 0) {
            int n_k = 0, n_v = 0;   // copies issued
            for (int cs = 0;; ++cs) {
                if (!mbar_wait(&sm.chunk_ready[cs & 3], (cs >> 2) & 1, err, &sm.abort)) break;
                const int page = *reinterpret_cast<volatile int32_t *>(&sm.chunk_page[cs & 3]);
                const int g = *reinterpret_cast<volatile int32_t *>(&sm.chunk_g[cs & 3]);
                mbar_arrive(&sm.chunk_free[cs & 3]);
                if (page < 0) break;
                // K once the previous chunk's last S has completed, V once its last PV has
                if (cs >= 1 && !mbar_wait(&sm.k_empty, (cs - 1) & 1, err, &sm.abort)) break;
                mbar_arrive_expect_tx(&sm.k_full, D * 128 * 2);
#pragma unroll
                for (int i = 0; i < NSUB; ++i) tma_load_4d(sm.k + i * 16384, &kmap, &sm.k_full, i * 64, g, 0, page);
                n_k = cs + 1;
                if (cs >= 1 && !mbar_wait(&sm.v_empty, (cs - 1) & 1, err, &sm.abort)) break;
                mbar_arrive_expect_tx(&sm.v_full, D * 128 * 2);
#pragma unroll
                for (int i = 0; i < NSUB; ++i) tma_load_4d(sm.v + i * 16384, &vmap, &sm.v_full, i * 64, g, 0, page);
                n_v = cs + 1;
            }
            if (sm.abort) {   // drain: the copies still in flight land before the CTA exits
                if (n_k > 0) mbar_wait(&sm.k_full, (n_k - 1) & 1, err, nullptr);
                if (n_v > 0) mbar_wait(&sm.v_full, (n_v - 1) & 1, err, nullptr);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (lane 0)
        // The warp shares its sub-partition with busy softmax and epilogue warps, and every issue
        // slot it needs per MMA slows the tensor core down: each group of MMAs is one asm block.
        // Every MMA is accepted about when the one before it finishes, so a wait of this thread between
        // two MMA groups leaves the tensor core idle: a tile costs the issuer three waits (its Q,
        // which also publishes its descriptor; the previous tile's P and O buffer, one barrier; K or V
        // on a chunk's first tile) and one read of its flags.
        if (lane == 0) {
            const uint64_t kd = make_smem_desc(smem_u32(sm.k), 16, 1024, 2);
            const uint64_t vd = make_smem_desc(smem_u32(sm.v), 16384, 1024, 2);
            int cs_k = -1, cs_v = -1;
            // PV in two halves of 64 tokens: the first as soon as the softmax has written P for tokens
            // 0..63 (and the O buffer is free), the second once all of P is written, so half of PV runs
            // while the softmax finishes
            auto issue_pv = [&](int t, int flags) -> bool {
                const int b = t & 1;
                if (!mbar_wait(&sm.p_lo[b], (t >> 1) & 1, err, &sm.abort)) return false;
                if (flags & kFlagFirst) {
                    ++cs_v;
                    if (!mbar_wait(&sm.v_full, cs_v & 1, err, &sm.abort)) return false;
                }
                tc_fence_after();
                mma_pv_half(tmem + uint32_t(256 + b * D), tmem + uint32_t(b * 128), vd, kIdescO, 0u);
                if (!mbar_wait(&sm.pv_ready[b], (t >> 1) & 1, err, &sm.abort)) return false;
                tc_fence_after();
                mma_pv_half(tmem + uint32_t(256 + b * D), tmem + uint32_t(b * 128 + 32), vd + 512, kIdescO, 1u);
                mma_commit(&sm.o_full[b]);
                if (flags & kFlagLast) mma_commit(&sm.v_empty);
                return true;
            };
            int pu = -1, pflags = 0;   // the tile whose PV is pending (issued after the next tile's S)
            for (int u = 0;; ++u) {
                // the Q loader reads the tile's descriptor before it loads Q (an end marker completes
                // the phase with no bytes), so a full Q buffer means the flags can be read
                const int qb = u % kQBuf;
                if (!mbar_wait(&sm.q_full[qb], (u / kQBuf) & 1, err, &sm.abort)) break;
                const int slot = u % kRing;
                const int flags = sm_flags(sm.desc[slot]);
                if (flags & kFlagEnd) break;
                mbar_arrive(&sm.desc_empty[slot]);
                if (flags & kFlagFirst) {
                    ++cs_k;
                    if (!mbar_wait(&sm.k_full, cs_k & 1, err, &sm.abort)) break;
                }
                tc_fence_after();
                const int b = u & 1;
                mma_s_block<D / 16>(tmem + uint32_t(b * 128), make_smem_desc(smem_u32(sm.q[qb]), 16, 1024, 2), kd,
                                    kIdescS, 1u);
                mma_commit(&sm.s_full[b]);
                mma_commit(&sm.q_empty[qb]);
                if (flags & kFlagLast) mma_commit(&sm.k_empty);
                if (pu >= 0 && !issue_pv(pu, pflags)) {
                    pu = -1;
                    break;
                }
                pu = u;
                pflags = flags;
            }
            if (pu >= 0 && !sm.abort) issue_pv(pu, pflags);
            mma_commit(&sm.drain);
            mbar_wait(&sm.drain, 0, err, nullptr);
        }
    } else if (warp == 17) {
        // idle: this warp would take issue slots from the MMA warp's sub-partition
    } else if (warp == 3 || warp == 16 || warp == 18) {
        // ------------------------------------------------------------ Q loaders (warps 16, 3, 18)
        // (sub-partitions 0, 3 and 2: the MMA warp's sub-partition 1 keeps its issue slots)
        constexpr int CPH = D / 8;         // 16-byte chunks of one head row
        constexpr int CPE = HPG * CPH;     // of one entry (a multiple of 32)
        static_assert(CPE % 32 == 0, "an entry spans whole warps of 16-byte chunks");
        // this lane's chunks of an entry: head and chunk column of chunk j * 32 + lane
        const uint8_t *q_row0 = qg + size_t(lane % CPH) * 16;   // + head row offset below
        const int qb = warp == 16 ? 0 : warp == 3 ? 1 : 2;   // this warp's Q buffer: tiles u % kQBuf == qb
        int n_tma = 0;   // tiles of this buffer whose Q boxes were issued
        for (int u = qb;; u += kQBuf) {
            const int slot = u % kRing;
            if (!__all_sync(0xffffffffu, mbar_wait(&sm.desc_ready[slot], (u / kRing) & 1, err, &sm.abort))) break;
            const volatile TileDesc &d = sm.desc[slot];
            if (d.flags & kFlagEnd) {
                __syncwarp();
                // the MMA issuer learns of the end through this tile's Q barrier: its phase completes
                // (with no bytes) once the buffer's previous tile has been consumed
                if (lane == 0) {
                    mbar_arrive(&sm.desc_full[slot]);
                    if (u < kQBuf || mbar_wait(&sm.q_empty[qb], ((u / kQBuf) - 1) & 1, err, &sm.abort))
                        mbar_arrive(&sm.q_full[qb]);
                }
                break;
            }
            if (u >= kQBuf &&
                !__all_sync(0xffffffffu, mbar_wait(&sm.q_empty[qb], ((u / kQBuf) - 1) & 1, err, &sm.abort)))
                break;
            const int g = d.g;
            if constexpr (HPG == 8) {
                // one TMA box of 64 columns x 8 heads (one whole 1024-byte swizzle atom) per entry and
                // sub-tile; a query row of -1 (padding, rejected entry) lies outside the tensor: zeros
                const int qq = lane < EPT ? d.qq[lane] : -1;
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&sm.desc_full[slot]);   // the descriptor has been read
                    mbar_arrive_expect_tx(&sm.q_full[qb], 128 * D * 2);
                }
                __syncwarp();
                if (lane < EPT) {
#pragma unroll
                    for (int i = 0; i < NSUB; ++i)
                        tma_load_3d(sm.q[qb] + i * 16384 + lane * (HPG * 128), &qmap, &sm.q_full[qb], i * 64,
                                    g * HPG, qq);
                }
                ++n_tma;
                continue;
            }
            const uint32_t qdst = smem_u32(sm.q[qb]);
#pragma unroll 1
            for (int e = 0; e < EPT; ++e) {
                const int qq = d.qq[e];
                const uint8_t *src = q_row0 + (size_t(qq) * Hq + size_t(g) * HPG) * (D * 2);
#pragma unroll
                for (int j = 0; j < CPE / 32; ++j) {
                    const int c = j * 32 + lane;
                    const int h = c / CPH, cw = c % CPH;
                    const int r = e * HPG + h;   // row of the 128-row tile
                    const uint32_t dst = qdst + uint32_t((cw >> 3) * 16384 + r * 128 + (((cw & 7) ^ (r & 7)) << 4));
                    if (qq >= 0) {
                        cp_async_16(dst, src + size_t(h) * (D * 2));
                    } else {   // padding or rejected entry: zero rows
                        asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(dst), "r"(0) : "memory");
                    }
                }
            }
            cp_async_commit();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.desc_full[slot]);   // the descriptor has been read
            cp_async_wait<0>();
            fence_proxy_async_smem();   // the copied rows are read by the tensor core
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.q_full[qb]);
        }
        cp_async_wait<0>();   // nothing in flight when the CTA exits
        // on abort, this buffer's last Q boxes land before the CTA exits (its earlier phases completed)
        if (n_tma > 0 && sm.abort && lane == 0) mbar_wait(&sm.q_full[qb], (n_tma - 1) & 1, err, nullptr);
    } else if (warp < 12) {
        // ------------------------------------------------------------ softmax groups (warps 4-11)
        const int wg = (warp - 4) >> 2;
        const int quad = warp & 3;                 // TMEM lanes this warp may access
        const int row = quad * 32 + lane;
        const int e = row / HPG, h = row - (row / HPG) * HPG;
        const uint32_t lane_off = uint32_t(quad * 32) << 16;
        const uint32_t t_s = tmem + lane_off + uint32_t(wg * 128);
        const float scale = sm_scale * kLog2e;
        const uint64_t scale2 = dup2(scale);
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
            // pass 1: row max over the visible tokens, two 32-column TMEM loads per wait (half the
            // load round trips; the loops stay rolled so the code stays small enough for the
            // instruction cache of a 19-warp CTA -- unrolling pass 2 the same way was slower)
            float mx[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) mx[i] = -INFINITY;
#pragma unroll 1
            for (int c0 = 0; c0 < 128; c0 += 64) {
                uint32_t vv[2][32];
                tmem_ld32(t_s + uint32_t(c0), vv[0]);
                tmem_ld32(t_s + uint32_t(c0 + 32), vv[1]);
                tmem_ld_wait();
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int c = c0 + 32 * hh;
                    const uint32_t(&v)[32] = vv[hh];
                    if (c + 31 <= lim) {   // fully visible chunk (every block but a row's own one)
#pragma unroll
                        for (int i = 0; i < 32; i += 16)
#pragma unroll
                            for (int j = 0; j < 8; ++j)
                                mx[j] = fmax3(mx[j], __uint_as_float(v[i + j]), __uint_as_float(v[i + 8 + j]));
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            mx[i & 7] = fmaxf(mx[i & 7], (c + i <= lim) ? __uint_as_float(v[i]) : -INFINITY);
                    }
                }
            }
            const float m = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
            const float ms = m * scale;
            const uint64_t nms2 = dup2(-ms);
            // pass 2: probabilities 2^(s*scale - ms) as packed bf16 over the columns already read
            // (P of chunk c lands in columns c/2 .. c/2+15, below the chunks still to read); their
            // fp32 sum in eight chains (four lane pairs) normalises O and gives the lse
            uint64_t acc2[4] = {0, 0, 0, 0};
#pragma unroll 1
            for (int c = 0; c < 128; c += 32) {
                uint32_t v[32];
                tmem_ld32(t_s + uint32_t(c), v);
                tmem_ld_wait();
                uint32_t w[16];
                if (c + 31 <= lim) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        float xa, xb;
                        ffma2(xa, xb, __uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]), scale2, nms2);
                        const float pa = fast_exp2(xa), pb = fast_exp2(xb);
                        w[i] = pack_bf16x2(pa, pb);
                        fadd2_acc(acc2[i & 3], pa, pb);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float sa = (c + 2 * i <= lim) ? __uint_as_float(v[2 * i]) : -INFINITY;
                        const float sb = (c + 2 * i + 1 <= lim) ? __uint_as_float(v[2 * i + 1]) : -INFINITY;
                        float xa, xb;
                        ffma2(xa, xb, sa, sb, scale2, nms2);
                        const float pa = fast_exp2(xa), pb = fast_exp2(xb);
                        w[i] = pack_bf16x2(pa, pb);
                        fadd2_acc(acc2[i & 3], pa, pb);
                    }
                }
                tmem_st16(t_s + uint32_t(c >> 1), w);
                if (c == 32) {   // P of tokens 0..63 is in TMEM: the first half of PV may start
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sm.p_lo[wg]);
                }
            }
            const float le = (sum2(acc2[0]) + sum2(acc2[1])) + (sum2(acc2[2]) + sum2(acc2[3]));
            // slot u % 4 is free once the epilogue has read tile u - 4's row sums
            if (u >= 4 && !__all_sync(0xffffffffu, mbar_wait(&sm.stat_free[u & 3], ((u >> 2) - 1) & 1, err, &sm.abort)))
                break;
            sm.inv_le[u & 3][row] = 1.0f / le;
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&sm.stat_full[u & 3]);
                mbar_arrive(&sm.pv_ready[wg]);
            }
            float lg;
            asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(lg) : "f"(le));
            if (qq >= 0) lse_part[size_t(idx) * HPG + h] = (ms + lg) * kLn2;
        }
    } else {
        // ------------------------------------------------------------ epilogue (warps 12-15)
        const int quad = warp & 3;                 // TMEM lanes this warp may access
        const int row = quad * 32 + lane;
        const uint32_t lane_off = uint32_t(quad * 32) << 16;
        // the partials are read back only by the merge kernel: evict them from L2 before Q, K and V
        const uint64_t store_policy = l2_policy_evict_first();
        for (int u = 0;; ++u) {
            const int slot = u % kRing;
            if (!__all_sync(0xffffffffu, mbar_wait(&sm.desc_full[slot], (u / kRing) & 1, err, &sm.abort))) break;
            const volatile TileDesc &d = sm.desc[slot];
            const int flags = d.flags;
            const int ent0 = d.ent0, n_valid = d.n_valid;
            __syncwarp();
            if (flags & kFlagEnd) break;
            if (lane == 0) mbar_arrive(&sm.desc_empty[slot]);
            const int b = u & 1, k = u >> 1;
            const uint32_t t_o = tmem + lane_off + uint32_t(256 + b * D);
            if (!__all_sync(0xffffffffu, mbar_wait(&sm.o_full[b], k & 1, err, &sm.abort))) break;
            if (!__all_sync(0xffffffffu, mbar_wait(&sm.stat_full[u & 3], (u >> 2) & 1, err, &sm.abort))) break;
            const uint64_t inv2 = dup2(sm.inv_le[u & 3][row]);
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.stat_free[u & 3]);
            // row `row` of the tile is head h of CSR entry ent0 + row / HPG; its 16-byte chunk cc sits
            // at byte (cc * HPG + h) * 16 of the entry's HPG x D block
            const bool live = row < n_valid * HPG;
            uint8_t *const gp = o_part + (size_t(ent0) + row / HPG) * (HPG * D * 2) + size_t(row % HPG) * 16;
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < D; c += 32) {
                uint32_t o[32];
                tmem_ld32(t_o + uint32_t(c), o);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; i += 8) {
                    uint32_t w4[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        float a, bb;
                        fmul2(a, bb, __uint_as_float(o[i + 2 * j]), __uint_as_float(o[i + 2 * j + 1]), inv2);
                        w4[j] = pack_bf16x2(a, bb);
                    }
                    if (live) st_global_v4_hint(gp + size_t((c + i) >> 3) * (HPG * 16), w4, store_policy);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.p_lo[b]);   // O buffer b is free for tile u + 2
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
    return launch_kernel(k_attn_prefill<D, HPG>, dim3(unsigned(sm_count())), dim3(kThreads), smem, st, true,
                         static_cast<const uint8_t *>(q), s.Hq, qm, km,
                         vm, static_cast<uint8_t *>(o_part), bt, q_req, q_pos, blk_off, blk_ent, hdr, static_cast<const int2 *>(chunks), n_rows,
                         n_req, n_pages, s.G, s.topk, s.max_blocks, s.sm_scale, lse_part, err);
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
