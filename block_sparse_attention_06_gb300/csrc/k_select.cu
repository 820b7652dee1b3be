// Selection bookkeeping: top-k blocks per (row, group), decode page tables and
// the {q, kv block} -> {kv block, q} inversion.
//
// "Together AI 解析如何高效服务 MiniMax M3…": 架构/特性 (the K most relevant blocks
// per KV group), 将 MSA 与分页注意力集成 (page tables per flattened (request,
// group) row), KV 块主序稀疏注意力 (the mapping is reorganised from {q, kv block}
// to {kv block, q}), 未来工作 (top-k and the remap are small kernels of their own).
#include "msa_device.cuh"
#include "msa_internal.h"

namespace msa {
namespace {

// ------------------------------------------------------------------ top-k

__device__ __forceinline__ uint64_t max_u64(uint64_t a, uint64_t b) { return a > b ? a : b; }

// Largest of a lane's keys that is below `bound` (0 when none): four independent
// max chains, so the dependent depth is PER/4 + 2 instead of PER.
template <int PER>
__device__ __forceinline__ uint64_t lane_max_below(const uint64_t (&keys)[PER], uint64_t bound) {
    uint64_t part[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const uint64_t k = keys[i] < bound ? keys[i] : 0ull;
        part[i & 3] = max_u64(part[i & 3], k);
    }
    return max_u64(max_u64(part[0], part[1]), max_u64(part[2], part[3]));
}

// The n best keys (n <= 32) among a warp's candidate keys, best first: lane i < n
// receives the i-th best key, every other lane 0.  A key of 0 is "no candidate";
// when fewer than n candidates exist the missing ranks are 0 too.  Every lane
// keeps its best key not yet taken; a round takes the warp maximum of those
// (two 32-bit warp reductions: score word, then block word among the lanes that
// hold that score) and only the lane it came from moves to its next key.  Keys
// are unique (the block id is inside), so equal scores are ordered by block id
// and nothing is taken twice.
template <int PER>
__device__ __forceinline__ uint64_t warp_top_n(const uint64_t (&keys)[PER], int n) {
    const int lane = threadIdx.x & 31;
    uint64_t local = lane_max_below<PER>(keys, ~0ull);
    uint64_t mine = 0;
    for (int round = 0; round < n; ++round) {
        const uint32_t hi = uint32_t(local >> 32);
        const uint32_t mhi = __reduce_max_sync(0xffffffffu, hi);
        const uint32_t mlo = __reduce_max_sync(0xffffffffu, hi == mhi ? uint32_t(local) : 0u);
        const uint64_t best = (uint64_t(mhi) << 32) | mlo;
        if (lane == round) mine = best;
        if (best != 0ull && local == best) local = lane_max_below<PER>(keys, best);
    }
    return mine;
}

// Position of this lane's block id among the ids held by lanes 0 .. n-1
// (ascending order); only meaningful for lanes < n.
__device__ __forceinline__ int rank_ascending(int id, int n) {
    int rank = 0;
#pragma unroll
    for (int l = 0; l < 32; ++l) {
        const int other = __shfl_sync(0xffffffffu, id, l);
        rank += (l < n && other < id) ? 1 : 0;
    }
    return rank;
}

// Bitonic sort of one key per lane, descending: lane i ends with the i-th largest of
// the warp's 32 keys (five merge levels, fifteen exchange steps).
__device__ __forceinline__ uint64_t warp_sort_desc(uint64_t k) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1)
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            const uint64_t o = __shfl_xor_sync(0xffffffffu, k, stride);
            // blocks of `size` alternate direction; the last level (size 32) runs descending
            const bool keep_max = ((lane & size) == 0) == ((lane & stride) == 0);
            k = keep_max ? max_u64(k, o) : (k < o ? k : o);
        }
    return k;
}

// CTA-wide top-n: every warp reduces its own keys to its n best, sorted best
// first, then warp 0 merges those NW sorted lists: lane w holds the head of warp
// w's list, each round takes the warp maximum of the heads and only the lane it
// came from moves on.  Returns, in warp 0, the lane's key as warp_top_n does;
// other warps return 0.  `stage` holds NT keys of shared memory.
template <int NT, int PER>
__device__ __forceinline__ uint64_t cta_top_n(const uint64_t (&keys)[PER], int n, uint64_t *stage) {
    constexpr int NW = NT / 32;
    static_assert(NW <= 32, "one list per lane of warp 0");
    const int tid = threadIdx.x, lane = tid & 31;
    if constexpr (PER == 1) {
        const uint64_t k = warp_sort_desc(keys[0]);
        stage[tid] = lane < n ? k : 0ull;
    } else {
        stage[tid] = warp_top_n<PER>(keys, n);
    }
    __syncthreads();
    uint64_t mine = 0;
    if (tid < 32) {
        int pos = 0;
        uint64_t head = lane < NW ? stage[lane * 32] : 0ull;
        for (int round = 0; round < n; ++round) {
            const uint32_t hi = uint32_t(head >> 32);
            const uint32_t mhi = __reduce_max_sync(0xffffffffu, hi);
            const uint32_t mlo = __reduce_max_sync(0xffffffffu, hi == mhi ? uint32_t(head) : 0u);
            const uint64_t best = (uint64_t(mhi) << 32) | mlo;
            if (lane == round) mine = best;
            if (best != 0ull && head == best) {
                ++pos;
                head = pos < n ? stage[lane * 32 + pos] : 0ull;
            }
        }
    }
    return mine;
}

// One warp per (row, group); keys of candidates j = lane + 32 * i live in registers.
template <int PER>
__global__ void __launch_bounds__(256) k_topk_warp(const float *__restrict__ scores,
                                                   const int32_t *__restrict__ q_pos, int n_rows,
                                                   int G, int max_blocks, int topk,
                                                   int32_t *__restrict__ sel, int32_t *err) {
    const int item = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (item >= n_rows * G) return;
    const int r = item / G;
    int32_t *out = sel + size_t(item) * topk;
    const int p = q_pos[r];
    if (p < 0 || (p >> 7) >= max_blocks || (p >> 7) >= 32 * PER) {
        for (int i = lane; i < topk; i += 32) out[i] = -1;
        if (lane == 0) raise_flag(err, MSA_FLAG_BOUNDS);
        return;
    }
    const int own = p >> 7;
    const int k_eff = min(topk, own + 1);
    const float *s = scores + size_t(item) * max_blocks;
    uint64_t keys[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int j = lane + 32 * i;
        keys[i] = j < own ? topk_key(s[j], j, err) : 0ull;
    }
    const int mine = int(~uint32_t(warp_top_n<PER>(keys, k_eff - 1)));
    const int rank = rank_ascending(mine, k_eff - 1);
    if (lane < k_eff - 1) out[rank] = mine;
    if (lane == 0) out[k_eff - 1] = own;
    for (int i = k_eff + lane; i < topk; i += 32) out[i] = -1;
}

// Top-k fused into prefill scoring, second half: one warp per (row, group) merges the
// candidate lists that the scoring CTAs kept for the row's block chunks (the best
// kSelectListLen keys of each chunk, 0 = none) into the selection, with the same
// rule and output as k_topk_warp.  The lists hold every candidate that can make
// the row's top k - 1, so the selection is the one k_topk_warp makes from the
// scores.
// The inversion's first pass for one selected block j of (row q, group g): set bit q
// of key (g * n_req + q_req[q]) * max_blocks + j in the per-key row bitmap.  A block
// listed twice for one (row, group), or a request id out of range, raises
// MSA_FLAG_BOUNDS.
__device__ __forceinline__ void inv_mark_one(uint32_t *__restrict__ bitmap, size_t words,
                                             const int32_t *__restrict__ q_req, int n_req, int max_blocks, int q,
                                             int g, int j, int32_t *err) {
    const int req = q_req[q];
    if (j < 0 || j >= max_blocks || req < 0 || req >= n_req) {
        raise_flag(err, MSA_FLAG_BOUNDS);
        return;
    }
    const size_t key = (size_t(g) * n_req + req) * max_blocks + j;
    const uint32_t bit = 1u << (q & 31);
    const uint32_t old = atomicOr(bitmap + key * words + (q >> 5), bit);
    if (old & bit) raise_flag(err, MSA_FLAG_BOUNDS);
}

// Merge of the chunks' candidate lists into the selection, one warp per (row,
// group).  With mark.bitmap set it also marks the inversion bitmap for every
// selected block (the inversion's first pass, fused here).
template <int PER>
__global__ void __launch_bounds__(256) k_topk_merge(const uint64_t *__restrict__ lists,
                                                    const int32_t *__restrict__ q_pos, int n_rows, int G,
                                                    int max_blocks, int n_cand, int topk,
                                                    int32_t *__restrict__ sel, InvMark mark, int32_t *err) {
    const int item = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (item >= n_rows * G) return;
    const int r = item / G;
    int32_t *out = sel + size_t(item) * topk;
    const int p = q_pos[r];
    if (p < 0 || (p >> 7) >= max_blocks) {
        for (int i = lane; i < topk; i += 32) out[i] = -1;
        if (lane == 0) raise_flag(err, MSA_FLAG_BOUNDS);
        return;
    }
    const int own = p >> 7;
    const int k_eff = min(topk, own + 1);
    const uint64_t *l = lists + size_t(item) * n_cand;
    uint64_t keys[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int c = lane + 32 * i;
        keys[i] = c < n_cand ? l[c] : 0ull;
    }
    const int mine = int(~uint32_t(warp_top_n<PER>(keys, k_eff - 1)));
    const int rank = rank_ascending(mine, k_eff - 1);
    if (lane < k_eff - 1) out[rank] = mine;
    if (lane == 0) out[k_eff - 1] = own;
    for (int i = k_eff + lane; i < topk; i += 32) out[i] = -1;
    if (mark.bitmap) {
        const int g = item - r * G;
        if (lane < k_eff - 1)
            inv_mark_one(mark.bitmap, mark.words, mark.q_req, mark.n_req, max_blocks, r, g, mine, err);
        if (lane == 0) inv_mark_one(mark.bitmap, mark.words, mark.q_req, mark.n_req, max_blocks, r, g, own, err);
    }
}

// The same merge with one thread per (row, group), for rows of at most NC chunks.  Each chunk's
// list is sorted best first, so the best k - 1 of the row are the first k - 1 keys of a k-way
// merge of the lists: every step takes the largest of the NC list heads and moves that list on.
// A thread keeps the next kMergeWin keys of every list in registers and reloads one key per step,
// which arrives while the list's other kMergeWin - 1 keys are taken, so a step seldom waits on
// memory.  The chosen ids are then put in ascending order by a sorting network; a missing
// candidate (key 0) gives id -1, which sorts first, as in k_topk_merge.
constexpr int kMergeWin = 4;

__device__ __forceinline__ void cmp_swap(int &a, int &b) {
    const int lo = min(a, b), hi = max(a, b);
    a = lo;
    b = hi;
}

template <int NC>
__global__ void __launch_bounds__(256) k_topk_merge_heads(const uint64_t *__restrict__ lists,
                                                          const int32_t *__restrict__ q_pos, int n_rows, int G,
                                                          int max_blocks, int topk, int32_t *__restrict__ sel,
                                                          InvMark mark, int32_t *err) {
    constexpr int L = kSelectListLen;
    constexpr int W = kMergeWin;
    static_assert(L + 1 == 16, "the sorting network orders 16 ids");
    static_assert(W <= L, "the window lies inside a list");
    const int item = blockIdx.x * blockDim.x + threadIdx.x;
    if (item >= n_rows * G) return;
    const int r = item / G;
    int32_t *out = sel + size_t(item) * topk;
    const int p = q_pos[r];
    if (p < 0 || (p >> 7) >= max_blocks) {
        for (int i = 0; i < topk; ++i) out[i] = -1;
        raise_flag(err, MSA_FLAG_BOUNDS);
        return;
    }
    const int own = p >> 7;
    const int k_eff = min(topk, own + 1);
    const int n = k_eff - 1;                        // non-own blocks to choose, <= L
    const uint64_t *l = lists + size_t(item) * NC * L;
    uint64_t win[NC][W];                            // win[c][0] is the head of list c
    int nxt[NC];                                    // list index of the key after the window
#pragma unroll
    for (int c = 0; c < NC; ++c) {
#pragma unroll
        for (int k = 0; k < W; ++k) win[c][k] = l[c * L + k];
        nxt[c] = W;
    }
    int id[16];
#pragma unroll
    for (int t = 0; t < 16; ++t) id[t] = INT_MAX;   // past n: sorts last, never written
#pragma unroll
    for (int t = 0; t < L; ++t) {
        if (t >= n) break;
        uint64_t best = win[0][0];
        int cb = 0;
#pragma unroll
        for (int c = 1; c < NC; ++c)
            if (win[c][0] > best) {
                best = win[c][0];
                cb = c;
            }
        id[t] = best ? int(~uint32_t(best)) : -1;
        if (best) {
            // one load for the list the key came from, then its window moves on by one
            int at = nxt[0];
#pragma unroll
            for (int c = 1; c < NC; ++c) at = c == cb ? nxt[c] : at;
            const uint64_t fresh = at < L ? l[cb * L + at] : 0ull;
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                const bool take = c == cb;
#pragma unroll
                for (int k = 0; k < W - 1; ++k) win[c][k] = take ? win[c][k + 1] : win[c][k];
                win[c][W - 1] = take ? fresh : win[c][W - 1];
                nxt[c] += take ? 1 : 0;
            }
        }
    }
    // Batcher's odd-even merge sort of 16 ids, ascending
#pragma unroll
    for (int k = 2; k <= 16; k <<= 1)
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1)
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int m = i ^ j;
                if (m > i) {
                    if ((i & k) == 0) cmp_swap(id[i], id[m]);
                    else cmp_swap(id[m], id[i]);
                }
            }
#pragma unroll
    for (int t = 0; t < 16; ++t)
        if (t < n) out[t] = id[t];
    out[n] = own;
    for (int i = k_eff; i < topk; ++i) out[i] = -1;
    if (mark.bitmap) {
        const int g = item - r * G;
#pragma unroll
        for (int t = 0; t < 16; ++t)
            if (t < n) inv_mark_one(mark.bitmap, mark.words, mark.q_req, mark.n_req, max_blocks, r, g, id[t], err);
        inv_mark_one(mark.bitmap, mark.words, mark.q_req, mark.n_req, max_blocks, r, g, own, err);
    }
}

// One CTA of NT threads per (row, group) for long contexts: each warp keeps its
// own best k-1, then warp 0 picks the best k-1 of those.
template <int NT, int PER>
__global__ void __launch_bounds__(NT) k_topk_cta(const float *__restrict__ scores,
                                                 const int32_t *__restrict__ q_pos, int G,
                                                 int max_blocks, int topk, int32_t *__restrict__ sel,
                                                 int32_t *err) {
    __shared__ uint64_t stage[NT];
    const int item = blockIdx.x;
    const int tid = threadIdx.x;
    const int r = item / G;
    int32_t *out = sel + size_t(item) * topk;
    const int p = q_pos[r];
    if (p < 0 || (p >> 7) >= max_blocks || (p >> 7) >= NT * PER) {
        for (int i = tid; i < topk; i += NT) out[i] = -1;
        if (tid == 0) raise_flag(err, MSA_FLAG_BOUNDS);
        return;
    }
    const int own = p >> 7;
    const int k_eff = min(topk, own + 1);
    const float *s = scores + size_t(item) * max_blocks;
    uint64_t keys[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int j = tid + NT * i;
        keys[i] = j < own ? topk_key(s[j], j, err) : 0ull;
    }
    const uint64_t best = cta_top_n<NT, PER>(keys, k_eff - 1, stage);
    if (tid < 32) {
        const int mine = int(~uint32_t(best));
        const int rank = rank_ascending(mine, k_eff - 1);
        if (tid < k_eff - 1) out[rank] = mine;
        if (tid == 0) out[k_eff - 1] = own;
        for (int i = k_eff + tid; i < topk; i += 32) out[i] = -1;
    }
}

// ------------------------------------------------------------------ decode selection (fused)
//
// After the decode index scan, one launch turns a request's block scores into
// its selection, its page tables and its row lengths ("Together AI 解析如何高效
// 服务 MiniMax M3…", 将 MSA 与分页注意力集成: page tables per flattened (request,
// group) row; 未来工作: the small top-k kernel fused with its neighbours).  Lane
// i < k_eff of the row's warp owns slot i of the ascending selection.

// Write the selection, page table and row length of row `item` (one warp).
// `best` holds, in lanes 0 .. k_eff-2, the chosen non-own keys.
__device__ __forceinline__ void emit_decode_row(uint64_t best, int item, int b, int L, int own, int k_eff,
                                                int topk, int max_blocks, int n_pages,
                                                const int32_t *__restrict__ block_table, int32_t *__restrict__ sel,
                                                int32_t *__restrict__ pt, int32_t *__restrict__ row_len,
                                                int32_t *err) {
    const int lane = threadIdx.x & 31;
    int id = int(~uint32_t(best));
    int slot = rank_ascending(id, k_eff - 1);
    if (lane == k_eff - 1) {   // the own block is the largest id: last slot
        id = own;
        slot = k_eff - 1;
    }
    int tok = 0;
    if (lane < k_eff) {
        int page = -1;
        if (id < 0 || id >= max_blocks) {
            raise_flag(err, MSA_FLAG_BOUNDS);
        } else {
            page = block_table[size_t(b) * max_blocks + id];
            if (page < 0 || page >= n_pages) {
                raise_flag(err, MSA_FLAG_BOUNDS);
                page = -1;
            } else {
                tok = max(0, min(128, L - id * 128));
            }
        }
        sel[size_t(item) * topk + slot] = id;
        pt[size_t(item) * topk + slot] = page;
    }
    for (int i = k_eff + lane; i < topk; i += 32) {
        sel[size_t(item) * topk + i] = -1;
        pt[size_t(item) * topk + i] = -1;
    }
    tok = warp_sum_i(tok);
    if (lane == 0) row_len[item] = tok;
}

// One CTA of NT threads per (request, group) row, PER candidates per thread.
template <int NT, int PER>
__global__ void __launch_bounds__(NT) k_decode_select_cta(
    const float *__restrict__ scores, const int32_t *__restrict__ seq_lens,
    const int32_t *__restrict__ block_table, int B, int G, int max_blocks, int topk, int n_pages,
    int32_t *__restrict__ sel, int32_t *__restrict__ pt, int32_t *__restrict__ row_len,
    int32_t *__restrict__ counters, int32_t *err) {
    __shared__ uint64_t stage[NT];
    const int item = blockIdx.x;
    const int tid = threadIdx.x;
    const int b = item / G;
    // seq_lens and the block table are inputs of the step, not results of the scan: read them
    // (the block table's row into L2) while the scan still runs
    const int L = seq_lens[b];
    const int p = L - 1;
    const bool bad = p < 0 || (p >> 7) >= max_blocks || (p >> 7) >= NT * PER;
    if (!bad) {
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int j = tid + NT * i;
            if (j <= (p >> 7) && (j & 31) == 0) prefetch_l2(block_table + size_t(b) * max_blocks + j);
        }
    }
    pdl_wait();
    pdl_trigger();
    if (counters && tid == 0) counters[item] = 0;
    if (bad) {
        for (int i = tid; i < topk; i += NT) {
            sel[size_t(item) * topk + i] = -1;
            pt[size_t(item) * topk + i] = -1;
        }
        if (tid == 0) {
            row_len[item] = 0;
            raise_flag(err, MSA_FLAG_BOUNDS);
        }
        return;
    }
    const int own = p >> 7;
    const int k_eff = min(topk, own + 1);
    const float *s = scores + size_t(item) * max_blocks;
    uint64_t keys[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int j = tid + NT * i;
        keys[i] = j < own ? topk_key(s[j], j, err) : 0ull;
    }
    const uint64_t best = cta_top_n<NT, PER>(keys, k_eff - 1, stage);
    if (tid < 32)
        emit_decode_row(best, item, b, L, own, k_eff, topk, max_blocks, n_pages, block_table, sel, pt, row_len,
                        err);
}

// ------------------------------------------------------------------ decode page table

__global__ void k_page_table(const int32_t *__restrict__ sel, const int32_t *__restrict__ block_table,
                             const int32_t *__restrict__ seq_lens, int B, int G, int topk,
                             int max_blocks, int n_pages, int32_t *__restrict__ pt,
                             int32_t *__restrict__ row_len, int32_t *err) {
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= B * G) return;
    const int b = r / G;
    const int L = seq_lens[b];
    int len = 0;
    for (int s = 0; s < topk; ++s) {
        const int j = sel[size_t(r) * topk + s];
        int page = -1;
        if (j >= 0) {
            if (j >= max_blocks) {
                raise_flag(err, MSA_FLAG_BOUNDS);
            } else {
                page = block_table[size_t(b) * max_blocks + j];
                if (page < 0 || page >= n_pages) {
                    raise_flag(err, MSA_FLAG_BOUNDS);
                    page = -1;
                } else {
                    len += max(0, min(128, L - j * 128));
                }
            }
        }
        pt[size_t(r) * topk + s] = page;
    }
    row_len[r] = len;
}

// ------------------------------------------------------------------ inversion
//
// Stable counting sort through a per-key bitmap over query rows: mark bits with
// atomicOr (order-free), count per key, scan, then emit each key's rows in
// ascending order.  Deterministic for any schedule.

struct InvLayout {
    size_t n_keys, words, bitmap_off, prefix_off, cnt_off, bytes;
};

// Workspace: the per-key row bitmap, the per-key exclusive prefix count of its words, the per-key count.
__host__ __device__ inline InvLayout inv_layout(int n_rows, int n_req, int G, int max_blocks) {
    InvLayout l;
    l.n_keys = size_t(G) * n_req * max_blocks;
    l.words = (size_t(n_rows) + 31) / 32;
    l.bitmap_off = 0;
    const size_t bm = (l.n_keys * l.words * 4 + 255) & ~size_t(255);
    l.prefix_off = bm;
    l.cnt_off = l.prefix_off + bm;
    l.bytes = l.cnt_off + ((l.n_keys * 4 + 255) & ~size_t(255));
    return l;
}

__global__ void k_inv_mark(const int32_t *__restrict__ sel, const int32_t *__restrict__ q_req, int n_rows,
                           int n_req, int G, int topk, int max_blocks, uint32_t *__restrict__ bitmap,
                           size_t words, int32_t *err) {
    const size_t e = size_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (e >= size_t(n_rows) * G * topk) return;
    const int j = sel[e];
    if (j < 0) return;
    const int q = int(e / (size_t(G) * topk));
    const int g = int((e / topk) % G);
    inv_mark_one(bitmap, words, q_req, n_req, max_blocks, q, g, j, err);
}

// One warp per key: the rows that selected the key (set bits), counted per bitmap word into an
// exclusive prefix over the key's words, and in total.
__global__ void k_inv_count(const uint32_t *__restrict__ bitmap, size_t words, size_t n_keys,
                            int32_t *__restrict__ prefix, int32_t *__restrict__ cnt) {
    const size_t key = (size_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (key >= n_keys) return;
    const uint32_t *row = bitmap + key * words;
    int32_t *pre = prefix + key * words;
    int base = 0;
    for (size_t w0 = 0; w0 < words; w0 += 32) {
        const int c = (w0 + lane < words) ? __popc(row[w0 + lane]) : 0;
        int x = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (w0 + lane < words) pre[w0 + lane] = base + x - c;
        base += __shfl_sync(0xffffffffu, x, 31);
    }
    if (lane == 0) cnt[key] = base;
}

// Exclusive scan of n counts into off[0..n] with one CTA of 1024 threads.
__global__ void __launch_bounds__(1024) k_inv_scan(const int32_t *__restrict__ cnt, size_t n,
                                                   int32_t *__restrict__ off) {
    __shared__ int32_t wsum[32];
    __shared__ int32_t carry_s;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) carry_s = 0;
    __syncthreads();
    for (size_t base = 0; base < n; base += 1024) {
        const size_t i = base + tid;
        const int32_t v = i < n ? cnt[i] : 0;
        int32_t x = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) wsum[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int32_t w = wsum[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int32_t y = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += y;
            }
            wsum[lane] = w;   // inclusive over warps
        }
        __syncthreads();
        const int32_t carry = carry_s;
        const int32_t excl = carry + (warp ? wsum[warp - 1] : 0) + x - v;
        if (i < n) off[i] = excl;
        __syncthreads();
        if (tid == 1023) carry_s = excl + v;
        __syncthreads();
    }
    if (tid == 0) off[n] = carry_s;
}

// One thread per (row q, group g, slot): its place among the rows that selected the same key is
// the key's CSR offset, the set bits of the key's bitmap in the words before q's word, and those
// of q's word below bit q (rows ascending: the order is stable in q and does not depend on the
// schedule).  Empty or rejected slots get ent_pos -1.
__global__ void k_inv_emit(const uint32_t *__restrict__ bitmap, const int32_t *__restrict__ prefix, size_t words,
                           const int32_t *__restrict__ off, const int32_t *__restrict__ sel,
                           const int32_t *__restrict__ q_req, int n_rows, int n_req, int G, int topk,
                           int max_blocks, int32_t *__restrict__ ent, int32_t *__restrict__ ent_pos) {
    const size_t e = size_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (e >= size_t(n_rows) * G * topk) return;
    const int j = sel[e];
    const int q = int(e / (size_t(G) * topk));
    const int g = int((e / topk) % G);
    const int slot = int(e % topk);
    const int req = q_req[q];
    if (j < 0 || j >= max_blocks || req < 0 || req >= n_req) {   // bounds were flagged by k_inv_mark
        ent_pos[e] = -1;
        return;
    }
    const size_t key = (size_t(g) * n_req + req) * max_blocks + j;
    const size_t w = key * words + (q >> 5);
    const int pos = off[key] + prefix[w] + __popc(bitmap[w] & ((1u << (q & 31)) - 1u));
    ent[pos] = q * topk + slot;
    ent_pos[e] = pos;
}

}  // namespace

cudaError_t launch_topk_merge(const uint64_t *lists, const int32_t *q_pos, int n_rows, const Shape &s,
                              int n_chunks, int32_t *sel, const InvMark &mark, int32_t *err, cudaStream_t st) {
    if (n_rows <= 0) return cudaSuccess;
    const int n_cand = n_chunks * kSelectListLen;
    const long long warps = 1LL * n_rows * s.G;
    if (n_chunks <= 8) {
        const unsigned tblocks = unsigned((warps + 255) / 256);
#define MSA_TMH_CASE(NC)                                                                                   \
    if (n_chunks == NC) {                                                                                  \
        k_topk_merge_heads<NC><<<tblocks, 256, 0, st>>>(lists, q_pos, n_rows, s.G, s.max_blocks, s.topk, sel, \
                                                        mark, err);                                        \
        return cudaGetLastError();                                                                         \
    }
        MSA_TMH_CASE(1) MSA_TMH_CASE(2) MSA_TMH_CASE(3) MSA_TMH_CASE(4)
        MSA_TMH_CASE(5) MSA_TMH_CASE(6) MSA_TMH_CASE(7) MSA_TMH_CASE(8)
#undef MSA_TMH_CASE
    }
    const unsigned blocks = unsigned((warps + 7) / 8);
#define MSA_TM_CASE(PP)                                                                                     \
    if (n_cand <= 32 * PP) {                                                                                \
        k_topk_merge<PP><<<blocks, 256, 0, st>>>(lists, q_pos, n_rows, s.G, s.max_blocks, n_cand, s.topk, sel, \
                                                 mark, err);                                                \
        return cudaGetLastError();                                                                          \
    }
    MSA_TM_CASE(1) MSA_TM_CASE(2) MSA_TM_CASE(3) MSA_TM_CASE(4) MSA_TM_CASE(8) MSA_TM_CASE(16) MSA_TM_CASE(32)
#undef MSA_TM_CASE
    return cudaErrorNotSupported;
}

cudaError_t launch_topk(const float *scores, const int32_t *q_pos, int n_rows, const Shape &s,
                        int32_t *sel, int32_t *err, cudaStream_t st) {
    const int items = n_rows * s.G;
    if (items <= 0) return cudaSuccess;
    const int mb = s.max_blocks;
    if (mb <= 1024) {
        // keys per lane in steps of 4: no lane holds more empty slots than it must
        const unsigned grid = unsigned((items + 7) / 8);
        const int per = (mb + 31) / 32;
#define MSA_TOPK_WARP(P) \
    k_topk_warp<P><<<grid, 256, 0, st>>>(scores, q_pos, n_rows, s.G, mb, s.topk, sel, err)
        if (per <= 4) MSA_TOPK_WARP(4);
        else if (per <= 8) MSA_TOPK_WARP(8);
        else if (per <= 12) MSA_TOPK_WARP(12);
        else if (per <= 16) MSA_TOPK_WARP(16);
        else if (per <= 20) MSA_TOPK_WARP(20);
        else if (per <= 24) MSA_TOPK_WARP(24);
        else if (per <= 28) MSA_TOPK_WARP(28);
        else MSA_TOPK_WARP(32);
#undef MSA_TOPK_WARP
    } else if (mb <= 8192) {
        k_topk_cta<256, 32><<<unsigned(items), 256, 0, st>>>(scores, q_pos, s.G, mb, s.topk, sel, err);
    } else if (mb <= 16384) {
        k_topk_cta<512, 32><<<unsigned(items), 512, 0, st>>>(scores, q_pos, s.G, mb, s.topk, sel, err);
    } else {
        return cudaErrorNotSupported;
    }
    return cudaGetLastError();
}

cudaError_t launch_page_table(const int32_t *sel, const int32_t *block_table, const int32_t *seq_lens,
                              int B, int n_pages, const Shape &s, int32_t *pt, int32_t *row_len,
                              int32_t *err, cudaStream_t st) {
    const int rows = B * s.G;
    if (rows <= 0) return cudaSuccess;
    k_page_table<<<unsigned((rows + 127) / 128), 128, 0, st>>>(sel, block_table, seq_lens, B, s.G, s.topk,
                                                                s.max_blocks, n_pages, pt, row_len, err);
    return cudaGetLastError();
}

cudaError_t launch_decode_select(const float *scores, const int32_t *seq_lens, const int32_t *block_table,
                                 int B, int n_pages, const Shape &s, int32_t *sel, int32_t *pt,
                                 int32_t *row_len, int32_t *counters, int32_t *err, cudaStream_t st,
                                 bool pdl) {
    const int items = B * s.G;
    if (items <= 0) return cudaSuccess;
    const int mb = s.max_blocks;
#define MSA_DSEL_ARGS scores, seq_lens, block_table, B, s.G, mb, s.topk, n_pages, sel, pt, row_len, counters, err
    // a CTA per row, one candidate per thread up to 1,024 blocks: each warp then sorts its 32 keys
    // with a bitonic network, where a warp holding 16 candidates per lane would rescan them in every
    // one of the top-k's rounds; past 1,024 blocks 512 threads with several candidates each did
    // better than 1,024 (decode1m: 328 against 334 us per step)
#define MSA_DSEL_CTA(NT, PER)                                                                             \
    if (mb <= (NT) * (PER))                                                                               \
        return launch_kernel(k_decode_select_cta<NT, PER>, dim3(unsigned(items)), dim3(NT), 0, st, pdl,   \
                             MSA_DSEL_ARGS);
    MSA_DSEL_CTA(128, 1) MSA_DSEL_CTA(256, 1) MSA_DSEL_CTA(512, 1) MSA_DSEL_CTA(1024, 1)
    MSA_DSEL_CTA(512, 4) MSA_DSEL_CTA(512, 8) MSA_DSEL_CTA(512, 16) MSA_DSEL_CTA(512, 32)
#undef MSA_DSEL_CTA
#undef MSA_DSEL_ARGS
    return cudaErrorNotSupported;
}

size_t invert_workspace_bytes(int n_rows, int n_req, const Shape &s) {
    return inv_layout(n_rows, n_req, s.G, s.max_blocks).bytes;
}

InvMark invert_clear(const int32_t *q_req, int n_rows, int n_req, const Shape &s, void *ws, cudaStream_t st,
                     cudaError_t *e) {
    const InvLayout l = inv_layout(n_rows, n_req, s.G, s.max_blocks);
    InvMark m{reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(ws) + l.bitmap_off), l.words, q_req, n_req};
    *e = cudaMemsetAsync(m.bitmap, 0, l.n_keys * l.words * 4, st);
    return m;
}

cudaError_t launch_invert(const int32_t *sel, const int32_t *q_req, int n_rows, int n_req,
                          const Shape &s, int32_t *blk_off, int32_t *blk_ent, int32_t *ent_pos, void *ws,
                          int32_t *err, cudaStream_t st) {
    cudaError_t e;
    const InvMark m = invert_clear(q_req, n_rows, n_req, s, ws, st, &e);
    if (e != cudaSuccess) return e;
    const size_t n_ent = size_t(n_rows) * s.G * s.topk;
    if (n_ent > 0) {
        k_inv_mark<<<unsigned((n_ent + 255) / 256), 256, 0, st>>>(sel, q_req, n_rows, n_req, s.G, s.topk,
                                                                   s.max_blocks, m.bitmap, m.words, err);
    }
    return launch_invert_finish(sel, q_req, n_rows, n_req, s, blk_off, blk_ent, ent_pos, ws, err, st);
}

cudaError_t launch_invert_finish(const int32_t *sel, const int32_t *q_req, int n_rows, int n_req, const Shape &s,
                                 int32_t *blk_off, int32_t *blk_ent, int32_t *ent_pos, void *ws, int32_t *err,
                                 cudaStream_t st) {
    const InvLayout l = inv_layout(n_rows, n_req, s.G, s.max_blocks);
    uint8_t *w = static_cast<uint8_t *>(ws);
    uint32_t *bitmap = reinterpret_cast<uint32_t *>(w + l.bitmap_off);
    int32_t *prefix = reinterpret_cast<int32_t *>(w + l.prefix_off);
    int32_t *cnt = reinterpret_cast<int32_t *>(w + l.cnt_off);
    const size_t n_ent = size_t(n_rows) * s.G * s.topk;
    const unsigned kgrid = unsigned((l.n_keys + 7) / 8);
    k_inv_count<<<kgrid, 256, 0, st>>>(bitmap, l.words, l.n_keys, prefix, cnt);
    k_inv_scan<<<1, 1024, 0, st>>>(cnt, l.n_keys, blk_off);
    if (n_ent > 0)
        k_inv_emit<<<unsigned((n_ent + 255) / 256), 256, 0, st>>>(bitmap, prefix, l.words, blk_off, sel, q_req,
                                                                   n_rows, n_req, s.G, s.topk, s.max_blocks,
                                                                   blk_ent, ent_pos);
    return cudaGetLastError();
}

}  // namespace msa
