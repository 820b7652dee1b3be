// Prefill index scoring on the 5th-generation tensor cores.
//
// For a chunk of prefill queries the score step is a dense contraction per KV
// group, [128 rows x Di] . [Di x 128 tokens] per KV block, followed by a block
// max with a causal mask ("Together AI 解析如何高效服务 MiniMax M3…", sections
// 架构/特性 and 解码索引评分内核优化: one score per 128-token block and KV group).
//
// One CTA owns (KV group g, 128 consecutive query rows, a chunk of up to 128
// blocks).  The rows may belong to several requests (a ragged multi-request
// chunk): the CTA then scores the tile once per request it holds, against that
// request's pages, and keeps each row's scores from its own request's pass.
// Warp roles:
//   warp 0     TMA producer: the q_idx tile once, then one k-index page per block
//              into a 4-stage ring (128B / 64B swizzle);
//   warp 1     TMEM owner and MMA issuer: tcgen05.mma kind::f16, M = 128 rows,
//              N = 128 tokens, K = Di, into one of two TMEM accumulators;
//   warps 2-5  epilogue: tcgen05.ld of the accumulator (thread = row), masked max
//              over the 128 token columns, 32 blocks staged in shared memory and
//              written out by each warp for its own 32 rows as coalesced 128-byte
//              row segments (no barrier across warps, so a timeout cannot leave a
//              warp waiting for another).
// With top-k fused in (section 未来工作 lists the small top-k kernel as a fusion
// candidate) the epilogue writes no scores: each thread keeps its row's best
// kListLen candidates of the chunk (top-k sort keys, blocks before the row's own
// block) in registers and writes that list; a merge kernel then picks each
// row's selection from the lists of all chunks.
// All waits are bounded; a timeout raises MSA_FLAG_TIMEOUT and drains.
#include "msa_device.cuh"
#include "msa_internal.h"

namespace msa {
namespace {

constexpr int kStages = 4;
constexpr int kChunk = 128;            // blocks per CTA
constexpr int kThreads = 192;
constexpr int kListLen = kSelectListLen;   // candidates kept per (row, chunk) with top-k fused: topk <= 16

template <int DI>
struct ScoreSmem {
    static constexpr int kTileBytes = 128 * DI * 2;
    alignas(1024) uint8_t a[kTileBytes];
    alignas(1024) uint8_t b[kStages][kTileBytes];
    float sc[128][33];
    uint64_t a_full;
    uint64_t full[kStages], empty[kStages];
    uint64_t acc_full[2], acc_empty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
    int n_pass;                 // distinct requests among the tile's rows
    int pass_req[128];          // request of each pass, in order of first appearance
    int pass_j1[128];           // one past the last candidate block of the pass's rows (chunk-clipped later)
    int row_req[128];           // request of each tile row, -1 past n_rows or for an invalid row
    int row_pass[128];          // pass index of each valid row
};


template <int DI, bool FUSED>
__global__ void __launch_bounds__(kThreads, 1) k_score_prefill(
    const __grid_constant__ CUtensorMap amap, const __grid_constant__ CUtensorMap bmap,
    const int32_t *__restrict__ block_table, const int32_t *__restrict__ q_req,
    const int32_t *__restrict__ q_pos, int n_rows, int n_req, int n_pages, int G, int max_blocks,
    int n_chunks, float *__restrict__ scores, uint64_t *__restrict__ lists, int32_t *err) {
    using Smem = ScoreSmem<DI>;
    constexpr uint32_t kSw = DI == 64 ? 2u : 4u;           // descriptor swizzle: 128B / 64B
    constexpr uint32_t kSbo = 8u * DI * 2u;                // 8 rows of DI bf16
    constexpr uint32_t kIdesc = make_idesc_bf16(128, 128, 0, 0);
    extern __shared__ uint8_t smem_raw[];
    Smem &sm = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const int tile = blockIdx.x / n_chunks;
    const int chunk = blockIdx.x - tile * n_chunks;
    const int g = blockIdx.y;
    const int row0 = tile * 128;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int j0 = chunk * kChunk;

    int row_jmax = -1;          // (thread < 128) own block of the thread's row
    int rq = -1;                // (thread < 128) request of the thread's row, -1 if none / invalid
    const int rq0 = q_req[min(row0, n_rows - 1)];
    if (tid == 0) sm.abort = 0;
    if (tid < 128) {
        const int grow = row0 + tid;
        if (grow < n_rows) {
            const int p = q_pos[grow];
            rq = q_req[grow];
            if (rq < 0 || rq >= n_req || p < 0 || (p >> 7) >= max_blocks) {
                if (chunk == 0 && g == 0) raise_flag(err, MSA_FLAG_BOUNDS);
                rq = -1;
            } else {
                row_jmax = p >> 7;
            }
        }
        sm.row_req[tid] = rq;
        sm.pass_j1[tid] = -1;
    }
    // the common case: every valid row of the tile belongs to the first row's request
    const bool one_req =
        __syncthreads_and(tid >= 128 || rq < 0 || rq == rq0) && rq0 >= 0 && rq0 < n_req;
    if (one_req) {
        if (tid == 0) {
            sm.pass_req[0] = rq0;
            sm.n_pass = 1;
        }
        if (tid < 128 && rq >= 0) atomicMax(&sm.pass_j1[0], row_jmax + 1);
    } else {
        if (tid == 0) {
            // distinct requests in order of first appearance; a run of equal requests costs one compare
            int n = 0, prev = -1, prev_k = -1;
            for (int i = 0; i < 128; ++i) {
                const int r = sm.row_req[i];
                int k = -1;
                if (r >= 0) {
                    if (r == prev) {
                        k = prev_k;
                    } else {
                        k = 0;
                        while (k < n && sm.pass_req[k] != r) ++k;
                        if (k == n) sm.pass_req[n++] = r;
                    }
                    prev = r;
                    prev_k = k;
                }
                sm.row_pass[i] = k;
            }
            sm.n_pass = n;
        }
        __syncthreads();
        if (tid < 128 && sm.row_pass[tid] >= 0) atomicMax(&sm.pass_j1[sm.row_pass[tid]], row_jmax + 1);
    }
    __syncthreads();
    const int n_pass = sm.n_pass;
    const int j_end_chunk = min(j0 + kChunk, max_blocks);
    // blocks [j0, pass_end(k)) hold candidates of pass k's rows
    auto pass_end = [&](int k) { return min(j_end_chunk, max(j0, sm.pass_j1[k])); };
    int total = 0;
    for (int k = 0; k < n_pass; ++k) total += pass_end(k) - j0;

    // blocks past a row's request's candidates are -inf (all of the chunk for a row without a valid
    // request; with a single request, the scores of an invalid row are left as they are)
    auto fill_neg_inf = [&]() {
        if (tid < 64) return;
        const int e = tid - 64;                          // 128 epilogue threads
        if (one_req) {
            const int from = pass_end(0);
            if (from >= j_end_chunk) return;
            for (int i = 0; i < 128 && row0 + i < n_rows; ++i) {
                float *o = scores + (size_t(row0 + i) * G + g) * max_blocks;
                for (int j = from + e; j < j_end_chunk; j += 128) o[j] = -INFINITY;
            }
            return;
        }
        for (int i = 0; i < 128; ++i) {
            const int grow = row0 + i;
            if (grow >= n_rows) break;
            const int k = sm.row_pass[i];
            const int from = k >= 0 ? pass_end(k) : j0;
            float *o = scores + (size_t(grow) * G + g) * max_blocks;
            for (int j = from + e; j < j_end_chunk; j += 128) o[j] = -INFINITY;
        }
    };
    // fused top-k: this chunk's candidate list of row i, kListLen keys (0 = none)
    auto list_of = [&](int i) { return lists + ((size_t(row0 + i) * G + g) * n_chunks + chunk) * kListLen; };
    if (total <= 0) {
        if (FUSED) {
            if (tid < 128 && row0 + tid < n_rows)
                for (int i = 0; i < kListLen; ++i) list_of(tid)[i] = 0ull;
            return;
        }
        fill_neg_inf();
        return;
    }

    if (tid == 0) {
        mbar_init(&sm.a_full, 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&sm.acc_full[a], 1);
            mbar_init(&sm.acc_empty[a], 4);
        }
        mbar_init(&sm.drain, 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&sm.tmem_base, 256);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;

    if (warp == 0) {
        if (lane == 0) {
            tma_prefetch_desc(&amap);
            tma_prefetch_desc(&bmap);
            mbar_arrive_expect_tx(&sm.a_full, Smem::kTileBytes);
            tma_load_3d(sm.a, &amap, &sm.a_full, 0, g, row0);
            int issued = 0, it = 0;          // blocks over all passes
            bool ok = true;
            for (int pk = 0; ok && pk < n_pass; ++pk) {
                const int req = sm.pass_req[pk], nb = pass_end(pk) - j0;
                for (int jj = 0; jj < nb; ++jj, ++it) {
                    const int s = it % kStages;
                    if (it >= kStages && !mbar_wait(&sm.empty[s], ((it / kStages) - 1) & 1, err, &sm.abort)) {
                        ok = false;
                        break;
                    }
                    int page = block_table[size_t(req) * max_blocks + j0 + jj];
                    if (page < 0 || page >= n_pages) {
                        raise_flag(err, MSA_FLAG_BOUNDS);
                        page = 0;
                    }
                    mbar_arrive_expect_tx(&sm.full[s], Smem::kTileBytes);
                    tma_load_4d(sm.b[s], &bmap, &sm.full[s], 0, g, 0, page);
                    issued = it + 1;
                }
            }
            // on abort: let every issued copy land before the CTA can exit
            if (sm.abort) {
                for (int jj = max(0, issued - kStages); jj < issued; ++jj)
                    mbar_wait(&sm.full[jj % kStages], (jj / kStages) & 1, err, nullptr);
                mbar_wait(&sm.a_full, 0, err, nullptr);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t a_addr = smem_u32(sm.a);
            bool ok = mbar_wait(&sm.a_full, 0, err, &sm.abort);
            for (int jj = 0; ok && jj < total; ++jj) {   // blocks over all passes
                const int s = jj % kStages;
                const int acc = jj & 1;
                if (!mbar_wait(&sm.full[s], (jj / kStages) & 1, err, &sm.abort)) break;
                if (jj >= 2 && !mbar_wait(&sm.acc_empty[acc], ((jj >> 1) - 1) & 1, err, &sm.abort)) break;
                tc_fence_after();
                const uint32_t b_addr = smem_u32(sm.b[s]);
#pragma unroll
                for (int k = 0; k < DI / 16; ++k) {
                    const uint64_t ad = make_smem_desc(a_addr + k * 32, 16, kSbo, kSw);
                    const uint64_t bd = make_smem_desc(b_addr + k * 32, 16, kSbo, kSw);
                    mma_bf16(tmem + uint32_t(acc * 128), ad, bd, kIdesc, k > 0 ? 1u : 0u);
                }
                mma_commit(&sm.empty[s]);
                mma_commit(&sm.acc_full[acc]);
            }
            // all issued MMAs complete before TMEM can be released
            mma_commit(&sm.drain);
            mbar_wait(&sm.drain, 0, err, nullptr);
        }
    } else {
        // epilogue: thread = accumulator row (TMEM lane quadrant = warp % 4)
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const int grow = row0 + row;
        const int p = grow < n_rows ? q_pos[grow] : -1;
        const uint32_t lane_addr = tmem + (uint32_t(quad * 32) << 16);
        bool ok = true;
        int it = 0;                                      // blocks over all passes
        const int own = p >> 7;                          // the row's own block (forced, not ranked)
        // fused top-k: the chunk's best candidates, best first, as (order-preserving score bits, block);
        // a row meets its blocks in increasing block order, so on equal scores the entry already in the
        // list ranks first and a strict compare of the score bits alone gives the (score desc, block asc)
        // order of the 64-bit sort keys, which are built only when the list is written out
        uint32_t lst_s[kListLen];                        // 0 = empty (every real score maps above 0)
        int32_t lst_j[kListLen];
#pragma unroll
        for (int i = 0; i < kListLen; ++i) {
            lst_s[i] = 0u;
            lst_j[i] = 0;
        }
        for (int pk = 0; ok && pk < n_pass; ++pk) {
        const int req = sm.pass_req[pk], nblk = pass_end(pk) - j0;
        for (int jj = 0; jj < nblk; ++jj, ++it) {
            const int acc = it & 1;
            ok = __all_sync(0xffffffffu, mbar_wait(&sm.acc_full[acc], (it >> 1) & 1, err, &sm.abort));
            if (!ok) break;
            tc_fence_after();
            const int lim = p - (j0 + jj) * 128;     // columns c <= lim are visible
            // block max in four independent chains of 3-input maxima (one dependent chain would
            // leave the epilogue waiting on instruction latency)
            float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int c0 = 0; c0 < 128; c0 += 64) {   // two 32-column TMEM loads per wait
                uint32_t v[2][32];
                tmem_ld32(lane_addr + uint32_t(acc * 128 + c0), v[0]);
                tmem_ld32(lane_addr + uint32_t(acc * 128 + c0 + 32), v[1]);
                tmem_ld_wait();
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int c1 = c0 + 32 * hh;
                    if (lim < c1 + 31) {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (c1 + i > lim) v[hh][i] = __float_as_uint(-INFINITY);
                    }
#pragma unroll
                    for (int i = 0; i < 32; i += 8)
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            mx[k] = fmax3(mx[k], __uint_as_float(v[hh][i + k]), __uint_as_float(v[hh][i + 4 + k]));
                }
            }
            const float best = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.acc_empty[acc]);
            if (FUSED) {
                const int jb = j0 + jj;
                if (jb < own && (one_req || sm.row_req[row] == req)) {
                    uint32_t ks = uint32_t(topk_key(best, jb, err) >> 32);
                    if (ks > lst_s[kListLen - 1]) {
                        // sorted insertion without a dependency chain: the entries below the new one
                        // (gt[i], a suffix of the list) move down one slot and the first of them takes
                        // the new entry; the worst one drops out
                        bool gt[kListLen];
#pragma unroll
                        for (int i = 0; i < kListLen; ++i) gt[i] = ks > lst_s[i];
#pragma unroll
                        for (int i = kListLen - 1; i >= 1; --i) {
                            lst_s[i] = gt[i] ? (gt[i - 1] ? lst_s[i - 1] : ks) : lst_s[i];
                            lst_j[i] = gt[i] ? (gt[i - 1] ? lst_j[i - 1] : jb) : lst_j[i];
                        }
                        lst_s[0] = gt[0] ? ks : lst_s[0];
                        lst_j[0] = gt[0] ? jb : lst_j[0];
                    }
                }
                continue;
            }
            sm.sc[row][jj & 31] = best;
            if ((jj & 31) == 31 || jj == nblk - 1) {
                // the warp writes back its own 32 rows, one coalesced 128-byte segment per row
                __syncwarp();
                const int base = jj & ~31;
                const int ncols = jj - base + 1;
                for (int i = 0; i < 32; ++i) {
                    const int r = quad * 32 + i;
                    const int gr = row0 + r;
                    if (gr < n_rows && lane < ncols && (one_req || sm.row_req[r] == req))   // this pass's rows
                        scores[(size_t(gr) * G + g) * max_blocks + j0 + base + lane] = sm.sc[r][lane];
                }
                __syncwarp();
            }
        }
        }
        if (FUSED && grow < n_rows) {
            uint64_t *o = list_of(row);
#pragma unroll
            for (int i = 0; i < kListLen; ++i)
                o[i] = lst_s[i] ? (uint64_t(lst_s[i]) << 32) | uint64_t(~uint32_t(lst_j[i])) : 0ull;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (!FUSED) fill_neg_inf();
    if (warp == 1) tmem_dealloc(tmem, 256);
}

template <int DI, bool FUSED>
cudaError_t launch_di(const void *q_idx, const void *kidx, const int32_t *bt, const int32_t *q_req,
                      const int32_t *q_pos, int n_rows, int n_req, int n_pages, const Shape &s, float *scores,
                      uint64_t *lists, int32_t *err, cudaStream_t st) {
    alignas(64) CUtensorMap am, bm;
    const char *why = nullptr;
    {
        const uint64_t dims[3] = {uint64_t(DI), uint64_t(s.G), uint64_t(n_rows)};
        const uint64_t strides[2] = {uint64_t(DI) * 2, uint64_t(s.G) * DI * 2};
        const uint32_t box[3] = {uint32_t(DI), 1u, 128u};
        if (!encode_tensor_map(&am, 3, q_idx, dims, strides, box, DI * 2, &why)) return cudaErrorInvalidValue;
    }
    {
        const uint64_t dims[4] = {uint64_t(DI), uint64_t(s.G), 128ull, uint64_t(n_pages)};
        const uint64_t strides[3] = {uint64_t(DI) * 2, uint64_t(s.G) * DI * 2, 128ull * s.G * DI * 2};
        const uint32_t box[4] = {uint32_t(DI), 1u, 128u, 1u};
        if (!encode_tensor_map(&bm, 4, kidx, dims, strides, box, DI * 2, &why)) return cudaErrorInvalidValue;
    }
    const int n_tiles = (n_rows + 127) / 128;
    const int n_chunks = (s.max_blocks + kChunk - 1) / kChunk;
    const size_t smem = sizeof(ScoreSmem<DI>) + 1024;
    cudaError_t e =
        cudaFuncSetAttribute(k_score_prefill<DI, FUSED>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    const long long gx = 1LL * n_tiles * n_chunks;
    if (gx > 0x7fffffffLL || s.G > 65535) return cudaErrorInvalidConfiguration;
    dim3 grid(unsigned(gx), unsigned(s.G));
    k_score_prefill<DI, FUSED><<<grid, kThreads, smem, st>>>(am, bm, bt, q_req, q_pos, n_rows, n_req, n_pages,
                                                             s.G, s.max_blocks, n_chunks, scores, lists, err);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_score_prefill(const void *q_idx, const void *kidx, const int32_t *block_table,
                                 const int32_t *q_req, const int32_t *q_pos, int n_rows, int n_req,
                                 int n_pages, const Shape &s, float *scores, uint64_t *lists, int32_t *err,
                                 cudaStream_t st) {
    if (n_rows <= 0) return cudaSuccess;
#define MSA_SP_CASE(DD)                                                                                          \
    if (s.Di == DD)                                                                                              \
        return lists ? launch_di<DD, true>(q_idx, kidx, block_table, q_req, q_pos, n_rows, n_req, n_pages, s,    \
                                           scores, lists, err, st)                                               \
                     : launch_di<DD, false>(q_idx, kidx, block_table, q_req, q_pos, n_rows, n_req, n_pages, s,   \
                                            scores, lists, err, st);
    MSA_SP_CASE(64) MSA_SP_CASE(32)
#undef MSA_SP_CASE
    return cudaErrorNotSupported;
}

int score_prefill_chunks(int max_blocks) { return (max_blocks + kChunk - 1) / kChunk; }

}  // namespace msa
