/*
 * MSA ORACLE -- test infrastructure, not product code.
 *
 * A plain, slow, single-threaded CPU restatement of what MiniMax Sparse
 * Attention (MSA) computes, in double precision on bf16 inputs.  Only the test
 * suite, the package smoke check and the benchmark's CPU-baseline leg load it.
 * It shares no code, header or table with the CUDA library.
 *
 * Sources (web pages; cited by title and section):
 *   [T-zh]  "Together AI 解析如何高效服务 MiniMax M3：1M token 上下文与多模态推理优化"
 *           (aihot.news), sections 架构/特性, KV 块主序稀疏注意力,
 *           将 MSA 与分页注意力集成, 解码索引评分内核优化, 未来工作.
 *   [T-ja]  "MiniMax-M3の効率的な推論サービス：100万トークンコンテキストとマルチモーダルを後悔なく実現"
 *           (news.chathome.org), the MSA, KV-block-major kernel, paged-attention
 *           and decode index-scoring paragraphs.
 *   [NV-ja] "NVIDIA 加速インフラ上で MiniMax M3 を活用した長文脈推論とエージェントワークフローの展開"
 *           (news.ainew.jp), the MSA paragraph after Table 1.
 *
 * Readings where the pages are silent (each one is listed with its reason in
 * the design notes of the repository):
 *   - block score = MAX over the block's causally visible tokens of the raw
 *     dot product q_idx . k_idx (no scale, no activation);
 *   - a row at absolute position p has candidate blocks 0 .. floor(p/page);
 *     its own block floor(p/page) is always selected and counts inside k;
 *   - the other candidates are ranked by (score descending, block ascending),
 *     k_eff = min(k, n_cand), the selection is written in ascending block
 *     order and padded with -1;
 *   - attention logits are scaled by sm_scale (1/sqrt(D)); lse is the natural
 *     log of the sum of exp of the scaled logits;
 *   - the LSE merge is the standard one: lse = m + log sum_s exp(lse_s - m),
 *     O = sum_s exp(lse_s - lse) * O_s, with each O_s normalised in its block.
 *
 * Parity pins for every function live in the CPU test suite (brute force on
 * tiny inputs, library routines on special cases, closed forms, invariants,
 * and a hand-worked fixture).
 *
 * Return value of every entry point: 0 on success, a negative number when an
 * index (page id, block id, request id) falls outside its array.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static double bf16_value(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Candidate blocks of a row at absolute position p: 0 .. p / page. */
static int32_t n_candidates(int32_t p, int32_t page)
{
    return p / page + 1;
}

/*
 * Block scores.  [T-zh 解码索引评分内核优化]: each query's query-side index vector
 * is compared with every candidate key-side index vector and each 128-token KV
 * block is reduced to one score; [T-zh 架构/特性]: one selection per KV group.
 *
 * q_idx       [n_rows][G][Di] bf16
 * kidx        [n_pages][page][G][Di] bf16
 * block_table [n_req][bt_stride] int32
 * scores      [n_rows][G][max_blocks] double; -inf for non-candidates
 */
int oracle_block_scores(const uint16_t *q_idx, const uint16_t *kidx,
                        const int32_t *block_table, int32_t bt_stride,
                        const int32_t *q_req, const int32_t *q_pos, int32_t n_rows,
                        int32_t n_req, int32_t G, int32_t Di, int32_t page,
                        int32_t n_pages, int32_t max_blocks, double *scores)
{
    for (int32_t r = 0; r < n_rows; ++r) {
        int32_t req = q_req[r];
        int32_t p = q_pos[r];
        if (req < 0 || req >= n_req || p < 0) return -1;
        int32_t n_cand = n_candidates(p, page);
        if (n_cand > max_blocks || n_cand > bt_stride) return -2;
        for (int32_t g = 0; g < G; ++g) {
            double *out = scores + ((size_t)r * G + g) * max_blocks;
            for (int32_t j = 0; j < max_blocks; ++j) out[j] = -INFINITY;
            const uint16_t *qv = q_idx + ((size_t)r * G + g) * Di;
            for (int32_t j = 0; j < n_cand; ++j) {
                int32_t pg = block_table[(size_t)req * bt_stride + j];
                if (pg < 0 || pg >= n_pages) return -3;
                double best = -INFINITY;
                for (int32_t t = 0; t < page; ++t) {
                    if ((int64_t)j * page + t > p) break;      /* causal */
                    const uint16_t *kv = kidx + (((size_t)pg * page + t) * G + g) * Di;
                    double dot = 0.0;
                    for (int32_t d = 0; d < Di; ++d) dot += bf16_value(qv[d]) * bf16_value(kv[d]);
                    if (dot > best) best = dot;
                }
                out[j] = best;
            }
        }
    }
    return 0;
}

/*
 * Top-k block selection per (row, group).  [T-zh 架构/特性]: the score part
 * picks the K most relevant blocks per KV group; [T-zh 解码索引评分内核优化]: only
 * the top blocks are kept for the attention kernel.
 *
 * scores [n_rows][G][max_blocks] double (only candidates are read)
 * sel    [n_rows][G][topk] int32, ascending block ids, -1 padding
 */
int oracle_topk(const double *scores, const int32_t *q_pos, int32_t n_rows, int32_t G,
                int32_t page, int32_t max_blocks, int32_t topk, int32_t *sel)
{
    unsigned char *taken = (unsigned char *)malloc((size_t)max_blocks + 1);
    int32_t *pick = (int32_t *)malloc(sizeof(int32_t) * ((size_t)topk + 1));
    if (!taken || !pick) { free(taken); free(pick); return -9; }
    int rc = 0;
    for (int32_t r = 0; r < n_rows && rc == 0; ++r) {
        int32_t n_cand = n_candidates(q_pos[r], page);
        if (q_pos[r] < 0 || n_cand > max_blocks) { rc = -2; break; }
        int32_t own = n_cand - 1;
        int32_t k_eff = n_cand < topk ? n_cand : topk;
        for (int32_t g = 0; g < G; ++g) {
            const double *s = scores + ((size_t)r * G + g) * max_blocks;
            memset(taken, 0, (size_t)max_blocks + 1);
            int32_t n_pick = 0;
            /* k_eff - 1 rounds: best remaining non-own candidate, lower id on ties */
            for (int32_t round = 0; round < k_eff - 1; ++round) {
                int32_t best = -1;
                for (int32_t j = 0; j < own; ++j) {
                    if (taken[j]) continue;
                    if (best < 0 || s[j] > s[best]) best = j;   /* strict: keeps lower j on ties */
                }
                taken[best] = 1;
                pick[n_pick++] = best;
            }
            pick[n_pick++] = own;                                  /* own block always kept */
            /* ascending block order (insertion sort) */
            for (int32_t a = 1; a < n_pick; ++a) {
                int32_t v = pick[a], b = a - 1;
                while (b >= 0 && pick[b] > v) { pick[b + 1] = pick[b]; --b; }
                pick[b + 1] = v;
            }
            int32_t *o = sel + ((size_t)r * G + g) * topk;
            for (int32_t i = 0; i < topk; ++i) o[i] = i < n_pick ? pick[i] : -1;
        }
    }
    free(taken);
    free(pick);
    return rc;
}

/*
 * Decode page table.  [T-zh 将 MSA 与分页注意力集成]: build a page table from the
 * selected blocks and flatten the KV-group dimension into the batch, so row
 * r = b * G + g has its own table.
 *
 * sel      [B][G][topk]  (decode: one row per request, position seq_lens[b]-1)
 * pt       [B*G][topk]   physical page per slot, -1 padding
 * row_len  [B*G]         tokens the row attends: selected blocks, clipped at seq_len
 */
int oracle_page_table(const int32_t *sel, const int32_t *block_table, int32_t bt_stride,
                      const int32_t *seq_lens, int32_t B, int32_t G, int32_t topk,
                      int32_t page, int32_t *pt, int32_t *row_len)
{
    for (int32_t b = 0; b < B; ++b) {
        for (int32_t g = 0; g < G; ++g) {
            int32_t r = b * G + g;
            int32_t len = 0;
            for (int32_t s = 0; s < topk; ++s) {
                int32_t j = sel[((size_t)b * G + g) * topk + s];
                if (j < 0) { pt[(size_t)r * topk + s] = -1; continue; }
                if (j >= bt_stride) return -2;
                pt[(size_t)r * topk + s] = block_table[(size_t)b * bt_stride + j];
                int32_t vis = seq_lens[b] - j * page;            /* tokens of block j that exist */
                if (vis > page) vis = page;
                if (vis < 0) vis = 0;
                len += vis;
            }
            row_len[r] = len;
        }
    }
    return 0;
}

/*
 * {q, kv block} -> {kv block, q} inversion.  [T-zh KV 块主序稀疏注意力]: the
 * mapping is reorganised so the attention kernel can loop over KV blocks outside
 * and queries inside.  Stable counting sort: key = (g * n_req + req) * max_blocks
 * + block; inside one key, entries keep ascending row order.
 *
 * sel      [n_rows][G][topk]
 * blk_off  [G * n_req * max_blocks + 1]  CSR offsets
 * blk_ent  [sum of valid slots]          entry = row * topk + slot
 */
int oracle_invert(const int32_t *sel, const int32_t *q_req, int32_t n_rows, int32_t n_req,
                  int32_t G, int32_t topk, int32_t max_blocks, int32_t *blk_off, int32_t *blk_ent)
{
    size_t n_keys = (size_t)G * n_req * max_blocks;
    int32_t *cursor = (int32_t *)calloc(n_keys + 1, sizeof(int32_t));
    if (!cursor) return -9;
    for (size_t i = 0; i <= n_keys; ++i) blk_off[i] = 0;
    for (int32_t q = 0; q < n_rows; ++q) {
        if (q_req[q] < 0 || q_req[q] >= n_req) { free(cursor); return -1; }
        for (int32_t g = 0; g < G; ++g)
            for (int32_t s = 0; s < topk; ++s) {
                int32_t j = sel[((size_t)q * G + g) * topk + s];
                if (j < 0) continue;
                if (j >= max_blocks) { free(cursor); return -2; }
                blk_off[((size_t)g * n_req + q_req[q]) * max_blocks + j + 1] += 1;
            }
    }
    for (size_t i = 0; i < n_keys; ++i) blk_off[i + 1] += blk_off[i];
    for (size_t i = 0; i < n_keys; ++i) cursor[i] = blk_off[i];
    for (int32_t q = 0; q < n_rows; ++q)
        for (int32_t g = 0; g < G; ++g)
            for (int32_t s = 0; s < topk; ++s) {
                int32_t j = sel[((size_t)q * G + g) * topk + s];
                if (j < 0) continue;
                size_t key = ((size_t)g * n_req + q_req[q]) * max_blocks + j;
                blk_ent[cursor[key]++] = q * topk + s;
            }
    free(cursor);
    return 0;
}

/* Softmax over n logits in one pass: returns lse, writes normalised weights. */
static double softmax_weights(const double *logit, int32_t n, double *w)
{
    double m = -INFINITY;
    for (int32_t i = 0; i < n; ++i) if (logit[i] > m) m = logit[i];
    double sum = 0.0;
    for (int32_t i = 0; i < n; ++i) { w[i] = exp(logit[i] - m); sum += w[i]; }
    for (int32_t i = 0; i < n; ++i) w[i] /= sum;
    return m + log(sum);
}

/*
 * Exact attention of each query head over the tokens of its group's selected
 * blocks.  [T-zh 架构/特性]: dense attention between the query token and the
 * selected blocks; [NV-ja, MSA paragraph]: no KV compression.  Head h belongs
 * to group h / (Hq / G).  Tokens past the row's position are masked (causal).
 *
 * q [n_rows][Hq][D]; k_cache, v_cache [n_pages][page][G][D]
 * sel [n_rows][G][topk]; out [n_rows][Hq][D]; lse [n_rows][Hq]
 */
int oracle_attention(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                     const int32_t *block_table, int32_t bt_stride, const int32_t *q_req,
                     const int32_t *q_pos, const int32_t *sel, int32_t n_rows, int32_t n_req,
                     int32_t Hq, int32_t G, int32_t D, int32_t page, int32_t n_pages,
                     int32_t topk, double sm_scale, double *out, double *lse)
{
    int32_t hpg = Hq / G;
    size_t cap = (size_t)topk * page;
    double *logit = (double *)malloc(sizeof(double) * cap);
    double *w = (double *)malloc(sizeof(double) * cap);
    int32_t *tok_page = (int32_t *)malloc(sizeof(int32_t) * cap);
    int32_t *tok_slot = (int32_t *)malloc(sizeof(int32_t) * cap);
    if (!logit || !w || !tok_page || !tok_slot) { free(logit); free(w); free(tok_page); free(tok_slot); return -9; }
    int rc = 0;
    for (int32_t r = 0; r < n_rows && rc == 0; ++r) {
        int32_t req = q_req[r], p = q_pos[r];
        if (req < 0 || req >= n_req) { rc = -1; break; }
        for (int32_t h = 0; h < Hq && rc == 0; ++h) {
            int32_t g = h / hpg;
            int32_t n = 0;
            for (int32_t s = 0; s < topk; ++s) {
                int32_t j = sel[((size_t)r * G + g) * topk + s];
                if (j < 0) continue;
                if (j >= bt_stride) { rc = -2; break; }
                int32_t pg = block_table[(size_t)req * bt_stride + j];
                if (pg < 0 || pg >= n_pages) { rc = -3; break; }
                for (int32_t t = 0; t < page; ++t) {
                    if ((int64_t)j * page + t > p) break;
                    tok_page[n] = pg;
                    tok_slot[n] = t;
                    ++n;
                }
            }
            if (rc) break;
            const uint16_t *qh = q + ((size_t)r * Hq + h) * D;
            for (int32_t i = 0; i < n; ++i) {
                const uint16_t *kv = k_cache + (((size_t)tok_page[i] * page + tok_slot[i]) * G + g) * D;
                double dot = 0.0;
                for (int32_t d = 0; d < D; ++d) dot += bf16_value(qh[d]) * bf16_value(kv[d]);
                logit[i] = dot * sm_scale;
            }
            double *o = out + ((size_t)r * Hq + h) * D;
            for (int32_t d = 0; d < D; ++d) o[d] = 0.0;
            if (n == 0) { lse[(size_t)r * Hq + h] = -INFINITY; continue; }
            lse[(size_t)r * Hq + h] = softmax_weights(logit, n, w);
            for (int32_t i = 0; i < n; ++i) {
                const uint16_t *vv = v_cache + (((size_t)tok_page[i] * page + tok_slot[i]) * G + g) * D;
                for (int32_t d = 0; d < D; ++d) o[d] += w[i] * bf16_value(vv[d]);
            }
        }
    }
    free(logit); free(w); free(tok_page); free(tok_slot);
    return rc;
}

/*
 * Per-block partial outputs.  [T-zh KV 块主序稀疏注意力]: with the KV-block-major
 * loop only a partial O per KV block is computed; each partial here is the
 * softmax-normalised output over that block's visible tokens plus its lse.
 *
 * o_part   [n_rows][topk][Hq][D]   (slot-major, heads inside)
 * lse_part [n_rows][topk][Hq]      -inf (and O = 0) for an empty slot
 */
int oracle_block_partials(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                          const int32_t *block_table, int32_t bt_stride, const int32_t *q_req,
                          const int32_t *q_pos, const int32_t *sel, int32_t n_rows, int32_t n_req,
                          int32_t Hq, int32_t G, int32_t D, int32_t page, int32_t n_pages,
                          int32_t topk, double sm_scale, double *o_part, double *lse_part)
{
    int32_t hpg = Hq / G;
    double *logit = (double *)malloc(sizeof(double) * (size_t)page);
    double *w = (double *)malloc(sizeof(double) * (size_t)page);
    if (!logit || !w) { free(logit); free(w); return -9; }
    int rc = 0;
    for (int32_t r = 0; r < n_rows && rc == 0; ++r) {
        int32_t req = q_req[r], p = q_pos[r];
        if (req < 0 || req >= n_req) { rc = -1; break; }
        for (int32_t s = 0; s < topk && rc == 0; ++s) {
            for (int32_t h = 0; h < Hq; ++h) {
                int32_t g = h / hpg;
                int32_t j = sel[((size_t)r * G + g) * topk + s];
                double *o = o_part + (((size_t)r * topk + s) * Hq + h) * D;
                double *l = lse_part + ((size_t)r * topk + s) * Hq + h;
                for (int32_t d = 0; d < D; ++d) o[d] = 0.0;
                if (j < 0) { *l = -INFINITY; continue; }
                if (j >= bt_stride) { rc = -2; break; }
                int32_t pg = block_table[(size_t)req * bt_stride + j];
                if (pg < 0 || pg >= n_pages) { rc = -3; break; }
                int32_t n = 0;
                const uint16_t *qh = q + ((size_t)r * Hq + h) * D;
                for (int32_t t = 0; t < page; ++t) {
                    if ((int64_t)j * page + t > p) break;
                    const uint16_t *kv = k_cache + (((size_t)pg * page + t) * G + g) * D;
                    double dot = 0.0;
                    for (int32_t d = 0; d < D; ++d) dot += bf16_value(qh[d]) * bf16_value(kv[d]);
                    logit[n++] = dot * sm_scale;
                }
                if (n == 0) { *l = -INFINITY; continue; }
                *l = softmax_weights(logit, n, w);
                for (int32_t t = 0; t < n; ++t) {
                    const uint16_t *vv = v_cache + (((size_t)pg * page + t) * G + g) * D;
                    for (int32_t d = 0; d < D; ++d) o[d] += w[t] * bf16_value(vv[d]);
                }
            }
        }
    }
    free(logit); free(w);
    return rc;
}

/*
 * Log-Sum-Exp merge of per-block partials.  [T-zh KV 块主序稀疏注意力]: a final
 * reduction based on Log-Sum-Exp rescales the partial O outputs and sums them
 * (the page's own formula did not survive extraction; this is the standard one).
 * Slots whose lse is -inf are skipped.
 */
int oracle_lse_merge(const double *o_part, const double *lse_part, int32_t n_rows,
                     int32_t Hq, int32_t D, int32_t topk, double *out, double *lse)
{
    for (int32_t r = 0; r < n_rows; ++r) {
        for (int32_t h = 0; h < Hq; ++h) {
            double m = -INFINITY;
            for (int32_t s = 0; s < topk; ++s) {
                double l = lse_part[((size_t)r * topk + s) * Hq + h];
                if (l > m) m = l;
            }
            double *o = out + ((size_t)r * Hq + h) * D;
            for (int32_t d = 0; d < D; ++d) o[d] = 0.0;
            if (m == -INFINITY) { lse[(size_t)r * Hq + h] = -INFINITY; continue; }
            double sum = 0.0;
            for (int32_t s = 0; s < topk; ++s) {
                double l = lse_part[((size_t)r * topk + s) * Hq + h];
                if (l != -INFINITY) sum += exp(l - m);
            }
            double total = m + log(sum);
            lse[(size_t)r * Hq + h] = total;
            for (int32_t s = 0; s < topk; ++s) {
                double l = lse_part[((size_t)r * topk + s) * Hq + h];
                if (l == -INFINITY) continue;
                double wgt = exp(l - total);
                const double *os = o_part + (((size_t)r * topk + s) * Hq + h) * D;
                for (int32_t d = 0; d < D; ++d) o[d] += wgt * os[d];
            }
        }
    }
    return 0;
}

/*
 * Attention over a decode page table: what a stock GQA paged-attention kernel
 * computes once [T-zh 将 MSA 与分页注意力集成] has handed it one table per
 * flattened (request, group) row.  Row r = b * G + g reads its row_len[r] tokens
 * from pages pt[r][0], pt[r][1], ... in order; heads of group g attend them.
 *
 * q [B][Hq][D]; pt [B*G][topk]; row_len [B*G]; out [B][Hq][D]; lse [B][Hq]
 */
int oracle_paged_attention(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                           const int32_t *pt, const int32_t *row_len, int32_t B, int32_t Hq,
                           int32_t G, int32_t D, int32_t page, int32_t n_pages, int32_t topk,
                           double sm_scale, double *out, double *lse)
{
    int32_t hpg = Hq / G;
    size_t cap = (size_t)topk * page;
    double *logit = (double *)malloc(sizeof(double) * cap);
    double *w = (double *)malloc(sizeof(double) * cap);
    if (!logit || !w) { free(logit); free(w); return -9; }
    int rc = 0;
    for (int32_t b = 0; b < B && rc == 0; ++b) {
        for (int32_t h = 0; h < Hq && rc == 0; ++h) {
            int32_t g = h / hpg;
            int32_t r = b * G + g;
            int32_t n = row_len[r];
            if (n < 0 || (size_t)n > cap) { rc = -2; break; }
            const uint16_t *qh = q + ((size_t)b * Hq + h) * D;
            for (int32_t i = 0; i < n; ++i) {
                int32_t pg = pt[(size_t)r * topk + i / page];
                if (pg < 0 || pg >= n_pages) { rc = -3; break; }
                const uint16_t *kv = k_cache + (((size_t)pg * page + i % page) * G + g) * D;
                double dot = 0.0;
                for (int32_t d = 0; d < D; ++d) dot += bf16_value(qh[d]) * bf16_value(kv[d]);
                logit[i] = dot * sm_scale;
            }
            if (rc) break;
            double *o = out + ((size_t)b * Hq + h) * D;
            for (int32_t d = 0; d < D; ++d) o[d] = 0.0;
            if (n == 0) { lse[(size_t)b * Hq + h] = -INFINITY; continue; }
            lse[(size_t)b * Hq + h] = softmax_weights(logit, n, w);
            for (int32_t i = 0; i < n; ++i) {
                int32_t pg = pt[(size_t)r * topk + i / page];
                const uint16_t *vv = v_cache + (((size_t)pg * page + i % page) * G + g) * D;
                for (int32_t d = 0; d < D; ++d) o[d] += w[i] * bf16_value(vv[d]);
            }
        }
    }
    free(logit); free(w);
    return rc;
}
