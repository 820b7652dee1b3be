// Host-side launchers shared between the C-ABI layer and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "msa.h"

#include <utility>

namespace msa {

// Launch `kernel` on `st`; with pdl == true the launch carries programmatic
// stream serialisation, so it may overlap the tail of the previous kernel on the
// stream (the kernel must call pdl_wait() before reading that kernel's output).
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool pdl,
                          Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

struct Shape {
    int Hq, G, D, Di, topk, max_blocks, hpg;
    float sm_scale;
};

cudaError_t launch_score_decode(const void *q_idx, const void *kidx, const int32_t *block_table,
                                const int32_t *q_req, const int32_t *q_pos, int n_rows, int n_req,
                                int n_pages, const Shape &s, float *scores, int32_t *err,
                                cudaStream_t st);

// `bytes` (a multiple of 16) from page-locked host memory (its device mapping) to device memory.
cudaError_t launch_stage_from_host(const void *src, void *dst, size_t bytes, cudaStream_t st);
// Selected K/V pages from host memory into a device pool (zero-copy gather).
cudaError_t launch_offload_gather(const void *host_k, const void *host_v, const int32_t *page_table, int B,
                                  int n_host_pages, const Shape &s, void *pool_k, void *pool_v,
                                  int32_t *pool_page_table, int32_t *err, cudaStream_t st);
// Multi-token decode scoring: rows grouped by request (q_req non-decreasing, <= 16 rows each).
cudaError_t launch_score_decode_mt(const void *q_idx, const void *kidx, const int32_t *block_table,
                                   const int32_t *q_req, const int32_t *q_pos, int n_rows, int n_req, int n_pages,
                                   const Shape &s, float *scores, int32_t *err, cudaStream_t st);
cudaError_t launch_score_prefill(const void *q_idx, const void *kidx, const int32_t *block_table,
                                 const int32_t *q_req, const int32_t *q_pos, int n_rows, int n_req,
                                 int n_pages, const Shape &s, float *scores, uint64_t *lists, int32_t *err,
                                 cudaStream_t st);
// Prefill scoring with top-k fused: block chunks per row (candidate lists per (row, group, chunk)),
// candidates kept per list, and the merge of the lists into the selection.
int score_prefill_chunks(int max_blocks);
constexpr int kSelectListLen = 15;
// Target of the inversion's first pass (bit q of key k at bitmap[k * words + q / 32]);
// bitmap == nullptr means "do not mark".
struct InvMark {
    uint32_t *bitmap;
    size_t words;
    const int32_t *q_req;
    int n_req;
};
cudaError_t launch_topk_merge(const uint64_t *lists, const int32_t *q_pos, int n_rows, const Shape &s,
                              int n_chunks, int32_t *sel, const InvMark &mark, int32_t *err, cudaStream_t st);

cudaError_t launch_topk(const float *scores, const int32_t *q_pos, int n_rows, const Shape &s,
                        int32_t *sel, int32_t *err, cudaStream_t st);

cudaError_t launch_page_table(const int32_t *sel, const int32_t *block_table, const int32_t *seq_lens,
                              int B, int n_pages, const Shape &s, int32_t *pt, int32_t *row_len,
                              int32_t *err, cudaStream_t st);

size_t invert_workspace_bytes(int n_rows, int n_req, const Shape &s);
cudaError_t launch_invert(const int32_t *sel, const int32_t *q_req, int n_rows, int n_req,
                          const Shape &s, int32_t *blk_off, int32_t *blk_ent, int32_t *ent_pos, void *ws,
                          int32_t *err, cudaStream_t st);
// The inversion in two halves around a caller that marks the bitmap itself:
// invert_clear zeroes the bitmap in the inversion workspace and returns the mark
// target; launch_invert_finish counts, scans and emits from the marked bitmap.
InvMark invert_clear(const int32_t *q_req, int n_rows, int n_req, const Shape &s, void *ws, cudaStream_t st,
                     cudaError_t *e);
cudaError_t launch_invert_finish(const int32_t *sel, const int32_t *q_req, int n_rows, int n_req, const Shape &s,
                                 int32_t *blk_off, int32_t *blk_ent, int32_t *ent_pos, void *ws, int32_t *err,
                                 cudaStream_t st);

// Block-major prefill attention: a plan kernel writes the chunk work list into
// the workspace, then one persistent CTA per SM consumes it.
size_t prefill_workspace_bytes(int n_rows, int n_req, const Shape &s);
cudaError_t launch_attn_prefill(const void *q, const void *k_cache, const void *v_cache,
                                const int32_t *block_table, const int32_t *q_req,
                                const int32_t *q_pos, const int32_t *blk_off,
                                const int32_t *blk_ent, int n_rows, int n_req, int n_pages,
                                const Shape &s, void *o_part, float *lse_part, void *ws,
                                int32_t *err, cudaStream_t st);

cudaError_t launch_lse_merge(const void *o_part, const float *lse_part, const int32_t *sel,
                             const int32_t *ent_pos, int n_rows, const Shape &s, void *out, float *lse,
                             int32_t *err, cudaStream_t st);

// Decode workspace: segment partials (one per run of a row's pages inside one
// CTA's range, at the run's first slot), their lse, and one merge counter per
// (request, group) row.  The counters must be zero when the attention kernel
// starts; launch_attn_decode clears them itself unless counters_zeroed is set
// (the fused decode step clears them in its select kernel).
size_t decode_workspace_bytes(int B, const Shape &s);
int32_t *decode_ws_counters(void *ws, int B, const Shape &s);
cudaError_t launch_attn_decode(const void *q, const void *k_cache, const void *v_cache,
                               const int32_t *pt, const int32_t *row_len, int B, int n_pages,
                               const Shape &s, void *out, float *lse, void *ws, int32_t *err,
                               cudaStream_t st, bool counters_zeroed = false, bool pdl = false);

// Decode selection in one launch after the index scan: top-k per (request,
// group), page table and row lengths; also zeroes `counters` (B*G entries,
// may be null).  Launched with programmatic serialisation after the scan.
cudaError_t launch_decode_select(const float *scores, const int32_t *seq_lens, const int32_t *block_table,
                                 int B, int n_pages, const Shape &s, int32_t *sel, int32_t *pt,
                                 int32_t *row_len, int32_t *counters, int32_t *err, cudaStream_t st,
                                 bool pdl);

// Decode index scan whose rows are the B requests themselves (row b is request
// b at position seq_lens[b] - 1).
cudaError_t launch_score_decode_seq(const void *q_idx, const void *kidx, const int32_t *block_table,
                                    const int32_t *seq_lens, int B, int n_pages, const Shape &s,
                                    float *scores, int32_t *err, cudaStream_t st, bool pdl = false);

// Tensor-map creation through the driver entry point (no libcuda link dependency).
bool encode_tensor_map(void *map, int rank, const void *base, const uint64_t *dims,
                       const uint64_t *strides_bytes, const uint32_t *box, int swizzle_bytes,
                       const char **why);

int sm_count();

// One thread waits on an mbarrier that nothing arrives on (the device timeout path).
cudaError_t launch_selftest_timeout(int32_t *err, cudaStream_t st);

// Record the detail string that msa_last_error() returns on this thread.
void set_last_error(const char *msg);

}  // namespace msa
