/*
 * msa.h -- C ABI of libmsa.so, the MiniMax Sparse Attention (MSA) hot path on
 * NVIDIA GB300 (sm_103a).
 *
 * Sources, cited by page title and section:
 *   [T-zh]  "Together AI 解析如何高效服务 MiniMax M3：1M token 上下文与多模态推理优化"
 *           (aihot.news) -- sections 架构/特性 (two-part MSA), KV 块主序稀疏注意力
 *           (block-major prefill + Log-Sum-Exp reduction), 将 MSA 与分页注意力集成
 *           (decode page tables, groups flattened into the batch), 解码索引评分内核优化
 *           (decode index scoring), 未来工作 (top-k / remap kernels).
 *   [T-ja]  "MiniMax-M3の効率的な推論サービス：100万トークンコンテキストとマルチモーダルを後悔なく実現"
 *           (news.chathome.org) -- the same material in summary.
 *   [NV-ja] "NVIDIA 加速インフラ上で MiniMax M3 を活用した長文脈推論とエージェントワークフローの展開"
 *           (news.ainew.jp) -- MSA paragraph after Table 1 (each KV block read once).
 *
 * Conventions for every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller, except where
 *     an entry point says that page-locked host memory is accepted (the host
 *     caches of msa_offload_gather, the source of msa_stage_from_host, out and
 *     lse of the decode attention); the library allocates no memory.  bf16 tensors are passed as `const void *` and hold
 *     IEEE bfloat16 bit patterns.  All tensors are dense, row-major, with the
 *     shapes written beside each argument.
 *   - Paged caches share one page pool of n_pages pages of page_size = 128
 *     tokens, token stride = G * width (the strided KV view of [T-zh
 *     将 MSA 与分页注意力集成]):  k_cache, v_cache bf16 [n_pages][128][G][D],
 *     kidx_cache bf16 [n_pages][128][G][Di] (same page ids as K/V).
 *   - block_table int32 [n_req][dims->max_blocks]: logical block -> page.
 *   - A query row has an absolute position q_pos and a request q_req.  Its
 *     candidate blocks are 0 .. q_pos/128; block q_pos/128 is its own block.
 *     Query head h belongs to KV group h / (Hq / G).
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream); calls return after host-side validation, never synchronise,
 *     and never throw.
 *   - Host-side validation failures return MSA_ERR_INVALID_ARG or
 *     MSA_ERR_UNSUPPORTED before anything is enqueued.  Errors the kernels
 *     detect (an out-of-range page or block id, a malformed selection, a wait
 *     that timed out) are OR-ed as flags into *err_word, a caller-owned device
 *     int32; the affected outputs are then unspecified.  msa_check() reads
 *     and clears that word.
 *   - Supported shapes: page_size == 128, Hq % G == 0, Hq / G in {4, 8},
 *     D in {64, 128}, Di in {32, 64}, 1 <= topk <= 32.  Others return
 *     MSA_ERR_UNSUPPORTED.
 */
#ifndef MSA_H_
#define MSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MSA_OK = 0,
    MSA_ERR_INVALID_ARG = 1,   /* null pointer, negative size, inconsistent dims     */
    MSA_ERR_UNSUPPORTED = 2,   /* a shape outside the supported set                  */
    MSA_ERR_CUDA = 3,          /* a CUDA runtime call failed (see msa_last_error)    */
    MSA_ERR_DEVICE_BOUNDS = 4, /* a kernel met an out-of-range index (err_word)      */
    MSA_ERR_TIMEOUT = 5,       /* a bounded device-side wait expired (err_word)      */
    MSA_ERR_WORKSPACE = 6,     /* workspace smaller than msa_workspace_bytes()       */
    MSA_ERR_DEVICE_UNSUPPORTED = 7 /* a kernel met a layout it cannot handle (err_word) */
} msa_status_t;

/* Bits of the device error word. */
#define MSA_FLAG_BOUNDS      0x1
#define MSA_FLAG_TIMEOUT     0x2
#define MSA_FLAG_UNSUPPORTED 0x4
#define MSA_FLAG_NAN         0x8

typedef struct {
    int32_t Hq;         /* query heads                                          */
    int32_t G;          /* KV groups (= KV heads)                               */
    int32_t D;          /* head dim of Q/K/V                                    */
    int32_t Di;         /* index-key dim (one index head per KV group)          */
    int32_t page_size;  /* tokens per page = per KV block; must be 128          */
    int32_t topk;       /* blocks kept per (row, group), own block included     */
    int32_t max_blocks; /* block_table row stride = last dim of the scores      */
    float sm_scale;     /* attention logit scale, normally 1/sqrt(D)            */
} msa_dims_t;

typedef void *msa_stream_t;

/* Phase selector of msa_index_score. */
#define MSA_PHASE_DECODE       0
#define MSA_PHASE_PREFILL      1
#define MSA_PHASE_DECODE_MULTI 2

/* Operation selector of msa_workspace_bytes. */
#define MSA_OP_INVERT  0
#define MSA_OP_DECODE  1
#define MSA_OP_PREFILL 2
#define MSA_OP_SELECT_PREFILL 3
#define MSA_OP_SELECT_INVERT_PREFILL 4

/*
 * msa_index_score -- block scores for every (row, group, candidate block).
 * [T-zh 解码索引评分内核优化]: the query-side index vector is compared with every
 * candidate key-side index vector and each 128-token KV block is reduced to one
 * score; one score per KV group ([T-zh 架构/特性]).  The reduction is the MAX of
 * the raw dot products over the block's tokens at positions <= q_pos.
 *
 *   q_idx       bf16 [n_rows][G][Di]
 *   kidx_cache  bf16 [n_pages][128][G][Di]
 *   block_table int32 [n_req][max_blocks]
 *   q_req, q_pos int32 [n_rows]
 *   scores      fp32 [n_rows][G][max_blocks]  out; -inf for blocks > q_pos/128
 *   phase       MSA_PHASE_DECODE: each row streams its own candidate pages
 *               (HBM-bound path, any rows).  MSA_PHASE_PREFILL: rows are
 *               scored 128 at a time on the tensor cores.  The rows of a chunk
 *               may belong to several requests (a ragged multi-request chunked
 *               prefill): a run of 128 consecutive rows that holds rows of m
 *               requests is scored m times, once against each request's pages,
 *               so this phase suits chunks of a few long requests; single-token
 *               (decode) rows belong on MSA_PHASE_DECODE.
 *               MSA_PHASE_DECODE_MULTI: several decode rows per request
 *               (speculative or multi-token decode) share one read of each
 *               candidate page: keys as the M side of bf16 tensor-core MMAs, the
 *               request's rows as N ([T-zh 解码索引评分内核优化], the AB-swapped
 *               formulation).  Rows must be grouped by request (q_req
 *               non-decreasing, else MSA_FLAG_UNSUPPORTED) with at most 16 rows
 *               per request (else MSA_FLAG_UNSUPPORTED); max_blocks <= 65535.
 * A page id outside [0, n_pages) or a q_pos/128 >= max_blocks raises
 * MSA_FLAG_BOUNDS.
 */
msa_status_t msa_index_score(const void *q_idx, const void *kidx_cache, const int32_t *block_table,
                             const int32_t *q_req, const int32_t *q_pos, int32_t n_rows,
                             int32_t n_req, int32_t n_pages, const msa_dims_t *dims, int32_t phase,
                             float *scores, int32_t *err_word, msa_stream_t stream);

/*
 * msa_select_prefill -- msa_index_score (MSA_PHASE_PREFILL) and msa_topk_blocks in
 * one pass, writing the same selection and no scores.  [T-zh 未来工作]: the small
 * top-k kernel is a fusion candidate.  Each scoring CTA keeps, per row, the best
 * topk - 1 candidates of its chunk of 128 blocks (the sort keys of
 * msa_topk_blocks, in registers); a merge kernel picks each row's selection from
 * the lists of all its chunks.
 *
 *   q_idx ... dims   as msa_index_score
 *   sel       int32 [n_rows][G][topk]  out, identical to msa_topk_blocks on the
 *             scores of msa_index_score
 *   workspace device scratch of msa_workspace_bytes(MSA_OP_SELECT_PREFILL, n_rows,
 *             n_req, dims) bytes, 16-byte aligned (the candidate lists)
 * Limits: topk <= 16 and max_blocks <= 8704 (MSA_ERR_UNSUPPORTED otherwise: use
 * the two calls).
 */
msa_status_t msa_select_prefill(const void *q_idx, const void *kidx_cache, const int32_t *block_table,
                                const int32_t *q_req, const int32_t *q_pos, int32_t n_rows, int32_t n_req,
                                int32_t n_pages, const msa_dims_t *dims, int32_t *sel, void *workspace,
                                size_t workspace_bytes, int32_t *err_word, msa_stream_t stream);

/*
 * msa_select_invert_prefill -- msa_select_prefill followed by
 * msa_invert_selection, with the same outputs as those two calls.  [T-zh 未来工作]:
 * the top-k kernel and the q-kv -> kv-q remap kernel are fusion candidates; here
 * the kernel that merges the candidate lists into the selection also marks each
 * selected (key, row) for the inversion, so the remap's first pass needs no
 * kernel of its own.
 *
 *   q_idx ... dims        as msa_select_prefill
 *   sel                   int32 [n_rows][G][topk]  out, as msa_select_prefill
 *   blk_off, blk_ent, ent_pos  out, as msa_invert_selection
 *   workspace  device scratch of msa_workspace_bytes(MSA_OP_SELECT_INVERT_PREFILL,
 *              n_rows, n_req, dims) bytes, 16-byte aligned (candidate lists, then
 *              the inversion's workspace)
 * Limits: those of msa_select_prefill and msa_invert_selection.
 */
msa_status_t msa_select_invert_prefill(const void *q_idx, const void *kidx_cache, const int32_t *block_table,
                                       const int32_t *q_req, const int32_t *q_pos, int32_t n_rows, int32_t n_req,
                                       int32_t n_pages, const msa_dims_t *dims, int32_t *sel, int32_t *blk_off,
                                       int32_t *blk_ent, int32_t *ent_pos, void *workspace, size_t workspace_bytes,
                                       int32_t *err_word, msa_stream_t stream);

/*
 * msa_topk_blocks -- per (row, group): the own block q_pos/128 is always kept;
 * the other candidates 0 .. q_pos/128 - 1 are ranked by (score descending,
 * block id ascending) and the best k_eff - 1 are kept, k_eff = min(topk,
 * q_pos/128 + 1).  [T-zh 架构/特性]: the K most relevant blocks per KV group;
 * [T-zh 解码索引评分内核优化]: only the top blocks go to attention.  -0.0 ranks
 * equal to +0.0; a NaN score raises MSA_FLAG_NAN and ranks as -inf.
 *
 *   scores fp32 [n_rows][G][max_blocks]
 *   q_pos  int32 [n_rows]
 *   sel    int32 [n_rows][G][topk]  out; ascending block ids, -1 padding
 * Candidate counts up to 16384 blocks (2M tokens) are supported.
 */
msa_status_t msa_topk_blocks(const float *scores, const int32_t *q_pos, int32_t n_rows,
                             const msa_dims_t *dims, int32_t *sel, int32_t *err_word,
                             msa_stream_t stream);

/*
 * msa_build_page_table -- decode page tables.  [T-zh 将 MSA 与分页注意力集成]: a page
 * table is built from the selected blocks and the KV-group dimension is
 * flattened into the batch, so row r = b * G + g has its own table.
 *
 *   sel         int32 [B][G][topk]   decode selection (row b at seq_lens[b] - 1)
 *   block_table int32 [B][max_blocks]
 *   seq_lens    int32 [B]            cached tokens incl. the new one
 *   page_table  int32 [B*G][topk]    out; physical page per slot, -1 padding
 *   row_len     int32 [B*G]          out; tokens the row attends (selected
 *                                    blocks clipped at seq_lens[b])
 */
msa_status_t msa_build_page_table(const int32_t *sel, const int32_t *block_table,
                                  const int32_t *seq_lens, int32_t B, int32_t n_pages,
                                  const msa_dims_t *dims, int32_t *page_table, int32_t *row_len,
                                  int32_t *err_word, msa_stream_t stream);

/*
 * msa_invert_selection -- {q, kv block} -> {kv block, q}.  [T-zh KV 块主序稀疏注意力]:
 * the mapping is reorganised so attention can loop over KV blocks outside and
 * queries inside.  Keys are key = (g * n_req + q_req[q]) * max_blocks + block;
 * the output is a CSR whose entries are q * topk + slot, ascending in q inside
 * each key (deterministic, a stable counting sort).  ent_pos is the inverse
 * map: the CSR position of each selected (row, group, slot), which is also the
 * row of that slot's partial in msa_sparse_attn_prefill's output.
 *
 *   sel      int32 [n_rows][G][topk]
 *   q_req    int32 [n_rows]
 *   blk_off  int32 [G * n_req * max_blocks + 1]  out
 *   blk_ent  int32 [n_rows * G * topk]           out (first blk_off[last] used)
 *   ent_pos  int32 [n_rows][G][topk]             out; blk_ent[ent_pos[q][g][s]] ==
 *                                                q * topk + s where sel[q][g][s] >= 0,
 *                                                -1 where sel < 0
 *   workspace device scratch of msa_workspace_bytes(MSA_OP_INVERT, ...) bytes
 */
msa_status_t msa_invert_selection(const int32_t *sel, const int32_t *q_req, int32_t n_rows,
                                  int32_t n_req, const msa_dims_t *dims, int32_t *blk_off,
                                  int32_t *blk_ent, int32_t *ent_pos, void *workspace,
                                  size_t workspace_bytes, int32_t *err_word, msa_stream_t stream);

/*
 * msa_sparse_attn_prefill -- KV-block-major sparse attention.  [T-zh KV 块主序稀疏注意力]
 * and [T-ja, KV block-major kernel paragraph]: for each (group, KV block) the
 * block's K and V are read once and every query that selected it attends it;
 * [NV-ja]: each KV cache block is read once with contiguous access.  For each
 * CSR entry i = (q, slot) of key (g, req, j) and each head hh < Hq/G of group
 * g, writes the softmax-normalised partial output over block j's tokens at
 * positions <= q_pos[q], and its log-sum-exp (natural log of the sum of exp of
 * the sm_scale-scaled logits), as partial i (CSR order).  Entries past
 * blk_off[last] are not written.
 *
 * Partial layout (o_part), HPG = Hq/G.  Entry i owns HPG * D bf16 at element
 * i * HPG * D, as D/8 column chunks of 8 bf16, chunk-major: the 8 values of
 * (entry i, head hh, columns 8c .. 8c+7) start at bf16 element
 *     i * HPG * D  +  (c * HPG + hh) * 8.
 * This is the order in which the kernel's epilogue stores a tile straight from
 * registers (one head row per lane: every store instruction writes whole 128-byte
 * lines).
 *
 *   q        bf16 [n_rows][Hq][D]
 *   k_cache, v_cache bf16 [n_pages][128][G][D]
 *   block_table int32 [n_req][max_blocks];  q_req, q_pos int32 [n_rows]
 *   blk_off, blk_ent  the CSR of msa_invert_selection (same n_req, dims)
 *   o_part   bf16 [n_rows * G * topk][D/8][Hq/G][8]  out (layout above)
 *   lse_part fp32 [n_rows * G * topk][Hq/G]     out
 *   workspace device scratch of msa_workspace_bytes(MSA_OP_PREFILL, n_rows,
 *            n_req, ...) bytes, 16-byte aligned: the work list (each key cut
 *            into chunks of at most 8 tiles of 128/(Hq/G) entries) that one
 *            persistent CTA per SM consumes; written by the call itself.
 */
msa_status_t msa_sparse_attn_prefill(const void *q, const void *k_cache, const void *v_cache,
                                     const int32_t *block_table, const int32_t *q_req,
                                     const int32_t *q_pos, const int32_t *blk_off,
                                     const int32_t *blk_ent, int32_t n_rows, int32_t n_req,
                                     int32_t n_pages, const msa_dims_t *dims, void *o_part,
                                     float *lse_part, void *workspace, size_t workspace_bytes,
                                     int32_t *err_word, msa_stream_t stream);

/*
 * msa_lse_merge -- Log-Sum-Exp reduction of per-block partials.  [T-zh KV
 * 块主序稀疏注意力]: the partial O of each KV block is rescaled and summed.  For
 * each (q, h), g = h / (Hq/G), hh = h % (Hq/G), over the slots s with
 * sel[q][g][s] >= 0, the partial O_s / lse_s being entry ent_pos[q][g][s], head hh
 * of o_part (in the layout of msa_sparse_attn_prefill) / lse_part:
 *   lse = m + log(sum_s exp(lse_s - m)),  m = max_s lse_s
 *   out = sum_s exp(lse_s - lse) * O_s
 * Slots with sel < 0 are never read.  An ent_pos outside [0, n_rows*G*topk)
 * raises MSA_FLAG_BOUNDS and that slot is skipped.
 *
 *   o_part   bf16 [n_rows * G * topk][D/8][Hq/G][8]
 *   lse_part fp32 [n_rows * G * topk][Hq/G]
 *   sel, ent_pos  int32 [n_rows][G][topk]
 *   out      bf16 [n_rows][Hq][D]  out;  lse fp32 [n_rows][Hq]  out
 */
msa_status_t msa_lse_merge(const void *o_part, const float *lse_part, const int32_t *sel,
                           const int32_t *ent_pos, int32_t n_rows, const msa_dims_t *dims, void *out,
                           float *lse, int32_t *err_word, msa_stream_t stream);

/*
 * msa_sparse_attn_decode -- decode attention over per-(request, group) page
 * tables ([T-zh 将 MSA 与分页注意力集成]): row r = b * G + g reads its row_len[r]
 * tokens from pages page_table[r][0], [1], ... in order (slot s holds tokens
 * s*128 .. s*128+127 of the row); the Hq/G heads of group g attend them.
 * The (row, slot) items are cut into one contiguous range per SM; the slots of a
 * row inside one range (a segment) share one online softmax and write one partial
 * to the workspace, at the segment's first slot.  The segment that completes a
 * row merges the row's partials (the same reduction as msa_lse_merge), counted
 * in pages on a per-row counter in the workspace that this call clears before
 * its kernel runs.
 *
 *   q          bf16 [B][Hq][D]
 *   page_table int32 [B*G][topk];  row_len int32 [B*G]
 *   out        bf16 [B][Hq][D]  out;  lse fp32 [B][Hq]  out: device memory or
 *              page-locked host memory, written directly over the host link
 *              (other host memory gives MSA_ERR_INVALID_ARG)
 *   workspace  device scratch of msa_workspace_bytes(MSA_OP_DECODE, B, ...) bytes
 */
msa_status_t msa_sparse_attn_decode(const void *q, const void *k_cache, const void *v_cache,
                                    const int32_t *page_table, const int32_t *row_len, int32_t B,
                                    int32_t n_pages, const msa_dims_t *dims, void *out, float *lse,
                                    void *workspace, size_t workspace_bytes, int32_t *err_word,
                                    msa_stream_t stream);

/*
 * msa_offload_gather -- K/V offload with the k-index kept on the GPU.  [T-zh 未来工作]:
 * the KV cache may sit in host memory while the k-index stays resident; only the
 * pages the selection picked are fetched.  The GPU reads the page-locked host
 * caches in place (zero copy over the host link) and writes each selected group
 * slice into a device pool, so msa_sparse_attn_decode runs on the pool unchanged.
 *
 *   host_k_cache, host_v_cache  bf16 [n_host_pages][128][G][D], page-locked host
 *                    memory (cudaHostAlloc / cudaHostRegister), 16-byte aligned;
 *                    caller-owned, only read
 *   page_table       int32 [B*G][topk] device, host page ids (msa_build_page_table
 *                    on the host block table), -1 padding
 *   pool_k, pool_v   bf16 [B*topk][128][G][D] device, out: pool page b*topk + s
 *                    holds, in group slice g, the slice g of host page
 *                    page_table[b*G + g][s]
 *   pool_page_table  int32 [B*G][topk] device, out: the pool page of each slot (-1
 *                    where page_table is -1); pass it with the pools and
 *                    n_pages = B*topk to msa_sparse_attn_decode
 * A host page id >= n_host_pages raises MSA_FLAG_BOUNDS and its slot is not
 * copied.  Host caches that are not page-locked give MSA_ERR_INVALID_ARG.
 */
msa_status_t msa_offload_gather(const void *host_k_cache, const void *host_v_cache, int32_t n_host_pages,
                                const int32_t *page_table, int32_t B, const msa_dims_t *dims, void *pool_k,
                                void *pool_v, int32_t *pool_page_table, int32_t *err_word, msa_stream_t stream);

/*
 * msa_stage_from_host -- copy a step's packed inputs from page-locked host memory
 * to device memory.  Not an MSA operation: the transport of a decode step's
 * per-step inputs (q, q_idx, seq_lens, block table; a few hundred KB), done by a
 * kernel whose 16-byte loads read the host buffer in place over the host link
 * instead of by a copy-engine transfer, whose fixed cost (about 10 us on a
 * Grace-Blackwell node) exceeds the transfer itself at this size.
 *   host_src  page-locked host memory (cudaHostAlloc, cudaMallocHost or
 *             cudaHostRegister), 16-byte aligned
 *   dev_dst   device memory, 16-byte aligned
 *   bytes     a multiple of 16
 * Ordered on `stream` like a cudaMemcpyAsync; the host buffer must not change
 * until the copy has run.  Errors: MSA_ERR_INVALID_ARG for a source that is not
 * page-locked host memory, a destination that is not device memory, or a
 * pointer or size that is not a multiple of 16 bytes.
 */
msa_status_t msa_stage_from_host(const void *host_src, void *dev_dst, size_t bytes, msa_stream_t stream);

/*
 * msa_decode_step -- one whole decode step for B requests, each with one new
 * query token at position seq_lens[b] - 1: index scan (msa_index_score,
 * MSA_PHASE_DECODE, rows = requests), top-k (msa_topk_blocks), page tables
 * (msa_build_page_table) and paged sparse attention (msa_sparse_attn_decode),
 * with the same results as those four calls.  [T-zh 解码索引评分内核优化,
 * 将 MSA 与分页注意力集成]; [T-zh 未来工作]: the small top-k and page-table kernels
 * are fused into one.  Three kernels run back to back with programmatic
 * dependent launch, so each starts while the previous one drains; the scan is
 * launched that way too and reads nothing before the kernel ahead of it on the
 * stream has completed.
 *
 *   q           bf16 [B][Hq][D];  q_idx bf16 [B][G][Di]
 *   k_cache, v_cache bf16 [n_pages][128][G][D];  kidx_cache bf16 [n_pages][128][G][Di]
 *   block_table int32 [B][max_blocks];  seq_lens int32 [B] (cached tokens incl. the new one)
 *   scores      fp32 [B][G][max_blocks]  out
 *   sel         int32 [B][G][topk]       out
 *   page_table  int32 [B*G][topk], row_len int32 [B*G]  out
 *   out         bf16 [B][Hq][D], lse fp32 [B][Hq]      out: device memory or
 *               page-locked host memory, which the attention kernel then writes
 *               directly over the host link (no separate copy of the results)
 *   workspace   msa_workspace_bytes(MSA_OP_DECODE, B, 0, dims) bytes
 * Limits: B*G <= 65535, max_blocks <= 16384; caches 16-byte aligned.  out or lse
 * in other host memory gives MSA_ERR_INVALID_ARG.
 */
msa_status_t msa_decode_step(const void *q, const void *q_idx, const void *k_cache, const void *v_cache,
                             const void *kidx_cache, const int32_t *block_table, const int32_t *seq_lens, int32_t B,
                             int32_t n_pages, const msa_dims_t *dims, float *scores, int32_t *sel,
                             int32_t *page_table, int32_t *row_len, void *out, float *lse, void *workspace,
                             size_t workspace_bytes, int32_t *err_word, msa_stream_t stream);

/*
 * msa_sparse_attn_decode_noalloc -- the same computation as msa_sparse_attn_decode
 * for callers that cannot allocate device memory.  The pages have no counterpart
 * to it; it exists for callers like a serving engine that has reserved almost all
 * HBM for its paged KV pool and routes every allocation through its own
 * allocator, or a plugin host that forbids libraries from calling cudaMalloc.
 * Such a caller cannot provide a workspace either, so the segment partials
 * go to a fixed 16 MiB device array inside the library instead.
 *
 *   Arguments, layouts and outputs: as msa_sparse_attn_decode, minus the workspace.
 *   Limit: msa_workspace_bytes(MSA_OP_DECODE, B, 0, dims) must not exceed 16 MiB
 *   (for example B <= 31 requests at G = 8, topk = 16, Hq/G = 8, D = 128); larger
 *   calls return MSA_ERR_WORKSPACE and enqueue nothing.
 *   Allocation: none -- no cudaMalloc, cudaFree or allocating library routine.
 *   The array is static device memory that a GPU holds from the library's first
 *   use on it until the process exits.  With CUDA's default lazy module loading
 *   that first use is this entry point's first call on the device: it looks up
 *   the array's device address (cudaGetSymbolAddress, with that device current),
 *   which loads the module and reserves the 16 MiB.  Make that first call before
 *   any stream capture and before reserving the rest of device memory for a KV
 *   pool; if the reservation fails the call returns MSA_ERR_CUDA and says so.
 *   The address is kept per device: do not call this entry point on a device
 *   again after cudaDeviceReset.
 *   Sharing: all calls use the same array and find in it what the previous call
 *   left.  Calls whose kernels overlap on the GPU race on it, so the caller must
 *   serialise them (one stream, or events between streams).
 */
msa_status_t msa_sparse_attn_decode_noalloc(const void *q, const void *k_cache, const void *v_cache,
                                            const int32_t *page_table, const int32_t *row_len, int32_t B,
                                            int32_t n_pages, const msa_dims_t *dims, void *out, float *lse,
                                            int32_t *err_word, msa_stream_t stream);

/*
 * msa_workspace_bytes -- device scratch needed by an operation:
 *   MSA_OP_INVERT: n_rows query rows, n_req requests;
 *   MSA_OP_DECODE: n_rows = B decode requests (n_req ignored);
 *   MSA_OP_PREFILL: n_rows query rows, n_req requests.
 * Returns 0 for invalid arguments.
 */
size_t msa_workspace_bytes(int32_t op, int32_t n_rows, int32_t n_req, const msa_dims_t *dims);

/*
 * msa_check -- synchronise `stream`, read the device error word, reset it to 0,
 * and map it to a status (MSA_OK when no flag is set; bounds before NaN before
 * timeout before unsupported).
 */
msa_status_t msa_check(int32_t *err_word, msa_stream_t stream);

/* Human-readable name of a status. */
const char *msa_status_str(msa_status_t status);

/* Detail of the last MSA_ERR_* returned on this thread (static storage). */
const char *msa_last_error(void);

/* Library version: major * 10000 + minor * 100 + patch. */
int32_t msa_version(void);

/*
 * msa_selftest_timeout -- exercises the device error path that every bounded
 * wait of the library shares, without any fault: one thread waits on an
 * mbarrier that nothing arrives on, gives up after the wait limit (2 s), raises
 * MSA_FLAG_TIMEOUT in err_word and returns.  msa_check(err_word) then reports
 * MSA_ERR_TIMEOUT and clears the word; the stream stays usable.
 *
 *   err_word  int32 device word, caller-owned
 */
msa_status_t msa_selftest_timeout(int32_t *err_word, msa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MSA_H_ */
