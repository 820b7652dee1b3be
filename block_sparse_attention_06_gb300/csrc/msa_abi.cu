// The exported C ABI (include/msa.h): argument validation on the host, then
// kernel launches on the caller's stream.  Nothing here allocates device memory.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "msa.h"
#include "msa_internal.h"

namespace msa {

namespace {

thread_local char g_last_error[512] = "";

msa_status_t fail(msa_status_t st, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
msa_status_t fail(msa_status_t st, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return st;
}

msa_status_t cuda_fail(cudaError_t e, const char *where) {
    if (e == cudaErrorNotSupported)
        return fail(MSA_ERR_UNSUPPORTED, "%s: shape not supported by the kernels", where);
    return fail(MSA_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// Validate the dims a given operation depends on and fill the internal shape.
msa_status_t check_dims(const msa_dims_t *d, bool need_attn, bool need_index, Shape *s, const char *who) {
    if (!d) return fail(MSA_ERR_INVALID_ARG, "%s: dims is NULL", who);
    if (d->Hq <= 0 || d->G <= 0 || d->D <= 0 || d->Di <= 0 || d->topk <= 0 || d->max_blocks <= 0)
        return fail(MSA_ERR_INVALID_ARG, "%s: non-positive dimension", who);
    if (d->Hq % d->G != 0) return fail(MSA_ERR_INVALID_ARG, "%s: Hq %% G != 0", who);
    if (d->page_size != 128) return fail(MSA_ERR_UNSUPPORTED, "%s: page_size must be 128", who);
    if (d->topk > 32) return fail(MSA_ERR_UNSUPPORTED, "%s: topk > 32", who);
    const int hpg = d->Hq / d->G;
    if (need_attn) {
        if (hpg != 4 && hpg != 8) return fail(MSA_ERR_UNSUPPORTED, "%s: Hq/G must be 4 or 8", who);
        if (d->D != 64 && d->D != 128) return fail(MSA_ERR_UNSUPPORTED, "%s: D must be 64 or 128", who);
        if (!(d->sm_scale > 0.f)) return fail(MSA_ERR_INVALID_ARG, "%s: sm_scale must be > 0", who);
    }
    if (need_index) {
        if (d->Di != 32 && d->Di != 64) return fail(MSA_ERR_UNSUPPORTED, "%s: Di must be 32 or 64", who);
        if (d->G > 16 || (d->G & (d->G - 1)) != 0)
            return fail(MSA_ERR_UNSUPPORTED, "%s: G must be a power of two <= 16", who);
    }
    s->Hq = d->Hq;
    s->G = d->G;
    s->D = d->D;
    s->Di = d->Di;
    s->topk = d->topk;
    s->max_blocks = d->max_blocks;
    s->hpg = hpg;
    s->sm_scale = d->sm_scale;
    return MSA_OK;
}

#define MSA_REQUIRE(cond, ...)                                   \
    do {                                                         \
        if (!(cond)) return fail(MSA_ERR_INVALID_ARG, __VA_ARGS__); \
    } while (0)

}  // namespace

bool encode_tensor_map(void *map, int rank, const void *base, const uint64_t *dims, const uint64_t *strides_bytes,
                       const uint32_t *box, int swizzle_bytes, const char **why) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) {
        *why = "cuTensorMapEncodeTiled unavailable";
        return false;
    }
    cuuint64_t gd[5];
    cuuint64_t gs[4];
    cuuint32_t bx[5], es[5];
    for (int i = 0; i < rank; ++i) {
        gd[i] = dims[i];
        bx[i] = box[i];
        es[i] = 1;
    }
    for (int i = 0; i < rank - 1; ++i) gs[i] = strides_bytes[i];
    CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_NONE;
    if (swizzle_bytes == 128) sw = CU_TENSOR_MAP_SWIZZLE_128B;
    else if (swizzle_bytes == 64) sw = CU_TENSOR_MAP_SWIZZLE_64B;
    else if (swizzle_bytes == 32) sw = CU_TENSOR_MAP_SWIZZLE_32B;
    CUresult r = fn(static_cast<CUtensorMap *>(map), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, cuuint32_t(rank),
                    const_cast<void *>(base), gd, gs, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        *why = "cuTensorMapEncodeTiled rejected the layout";
        return false;
    }
    return true;
}

void set_last_error(const char *msg) { snprintf(g_last_error, sizeof g_last_error, "%s", msg); }

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
    return n;
}

}  // namespace msa

using namespace msa;

extern "C" {

msa_status_t msa_index_score(const void *q_idx, const void *kidx_cache, const int32_t *block_table,
                             const int32_t *q_req, const int32_t *q_pos, int32_t n_rows, int32_t n_req,
                             int32_t n_pages, const msa_dims_t *dims, int32_t phase, float *scores,
                             int32_t *err_word, msa_stream_t stream) {
    Shape s;
    msa_status_t st = check_dims(dims, false, true, &s, "msa_index_score");
    if (st != MSA_OK) return st;
    MSA_REQUIRE(n_rows >= 0 && n_req > 0 && n_pages > 0, "msa_index_score: bad sizes");
    if (n_rows == 0) return MSA_OK;
    MSA_REQUIRE(q_idx && kidx_cache && block_table && q_req && q_pos && scores && err_word,
                "msa_index_score: NULL pointer");
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (phase == MSA_PHASE_DECODE)
        e = launch_score_decode(q_idx, kidx_cache, block_table, q_req, q_pos, n_rows, n_req, n_pages, s, scores,
                                err_word, cs);
    else if (phase == MSA_PHASE_PREFILL)
        e = launch_score_prefill(q_idx, kidx_cache, block_table, q_req, q_pos, n_rows, n_req, n_pages, s, scores,
                                 nullptr, err_word, cs);
    else if (phase == MSA_PHASE_DECODE_MULTI)
        e = launch_score_decode_mt(q_idx, kidx_cache, block_table, q_req, q_pos, n_rows, n_req, n_pages, s, scores,
                                   err_word, cs);
    else
        return fail(MSA_ERR_INVALID_ARG, "msa_index_score: unknown phase %d", phase);
    return e == cudaSuccess ? MSA_OK : cuda_fail(e, "msa_index_score");
}

// Candidate lists of the fused prefill selection, 256-byte rounded.
static size_t select_lists_bytes(int n_rows, const Shape &s) {
    const size_t b = size_t(n_rows) * s.G * score_prefill_chunks(s.max_blocks) * kSelectListLen * sizeof(uint64_t);
    return (b + 255) & ~size_t(255);
}

// Checks shared by msa_select_prefill and msa_select_invert_prefill.
static msa_status_t check_select_prefill(const msa_dims_t *dims, Shape *s, const char *who) {
    msa_status_t st = check_dims(dims, false, true, s, who);
    if (st != MSA_OK) return st;
    if (s->topk > kSelectListLen + 1) return fail(MSA_ERR_UNSUPPORTED, "%s: topk > %d", who, kSelectListLen + 1);
    if (score_prefill_chunks(s->max_blocks) * kSelectListLen > 1024)
        return fail(MSA_ERR_UNSUPPORTED, "%s: max_blocks > %d", who, 1024 / kSelectListLen * 128);
    return MSA_OK;
}

msa_status_t msa_select_prefill(const void *q_idx, const void *kidx_cache, const int32_t *block_table,
                                const int32_t *q_req, const int32_t *q_pos, int32_t n_rows, int32_t n_req,
                                int32_t n_pages, const msa_dims_t *dims, int32_t *sel, void *workspace,
                                size_t workspace_bytes, int32_t *err_word, msa_stream_t stream) {
    Shape s;
    msa_status_t st = check_select_prefill(dims, &s, "msa_select_prefill");
    if (st != MSA_OK) return st;
    MSA_REQUIRE(n_rows >= 0 && n_req > 0 && n_pages > 0, "msa_select_prefill: bad sizes");
    if (n_rows == 0) return MSA_OK;
    MSA_REQUIRE(q_idx && kidx_cache && block_table && q_req && q_pos && sel && workspace && err_word,
                "msa_select_prefill: NULL pointer");
    const int n_chunks = score_prefill_chunks(s.max_blocks);
    const size_t need = size_t(n_rows) * s.G * n_chunks * kSelectListLen * sizeof(uint64_t);
    if (workspace_bytes < need)
        return fail(MSA_ERR_WORKSPACE, "msa_select_prefill: workspace of %zu bytes, %zu needed", workspace_bytes,
                    need);
    if (reinterpret_cast<uintptr_t>(workspace) & 15u)
        return fail(MSA_ERR_INVALID_ARG, "msa_select_prefill: workspace must be 16-byte aligned");
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    uint64_t *lists = static_cast<uint64_t *>(workspace);
    cudaError_t e = launch_score_prefill(q_idx, kidx_cache, block_table, q_req, q_pos, n_rows, n_req, n_pages, s,
                                         nullptr, lists, err_word, cs);
    if (e == cudaSuccess) e = launch_topk_merge(lists, q_pos, n_rows, s, n_chunks, sel, InvMark{}, err_word, cs);
    return e == cudaSuccess ? MSA_OK : cuda_fail(e, "msa_select_prefill");
}

msa_status_t msa_select_invert_prefill(const void *q_idx, const void *kidx_cache, const int32_t *block_table,
                                       const int32_t *q_req, const int32_t *q_pos, int32_t n_rows, int32_t n_req,
                                       int32_t n_pages, const msa_dims_t *dims, int32_t *sel, int32_t *blk_off,
                                       int32_t *blk_ent, int32_t *ent_pos, void *workspace, size_t workspace_bytes,
                                       int32_t *err_word, msa_stream_t stream) {
    Shape s;
    msa_status_t st = check_select_prefill(dims, &s, "msa_select_invert_prefill");
    if (st != MSA_OK) return st;
    MSA_REQUIRE(n_rows >= 0 && n_req > 0 && n_pages > 0, "msa_select_invert_prefill: bad sizes");
    MSA_REQUIRE(blk_off && err_word, "msa_select_invert_prefill: NULL pointer");
    MSA_REQUIRE(n_rows == 0 || (q_idx && kidx_cache && block_table && q_req && q_pos && sel && blk_ent && ent_pos),
                "msa_select_invert_prefill: NULL pointer");
    if (1.0 * n_rows * s.G * s.topk > 2147483647.0)
        return fail(MSA_ERR_UNSUPPORTED, "msa_select_invert_prefill: more than 2^31 entries");
    MSA_REQUIRE(workspace, "msa_select_invert_prefill: NULL workspace");
    if (reinterpret_cast<uintptr_t>(workspace) & 15u)
        return fail(MSA_ERR_INVALID_ARG, "msa_select_invert_prefill: workspace must be 16-byte aligned");
    const size_t lists_bytes = select_lists_bytes(n_rows, s);
    const size_t need = lists_bytes + invert_workspace_bytes(n_rows, n_req, s);
    if (workspace_bytes < need)
        return fail(MSA_ERR_WORKSPACE, "msa_select_invert_prefill: workspace of %zu bytes, %zu needed",
                    workspace_bytes, need);
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    void *inv_ws = static_cast<uint8_t *>(workspace) + lists_bytes;
    cudaError_t e;
    const InvMark mark = invert_clear(q_req, n_rows, n_req, s, inv_ws, cs, &e);
    if (e == cudaSuccess && n_rows > 0) {
        uint64_t *lists = static_cast<uint64_t *>(workspace);
        e = launch_score_prefill(q_idx, kidx_cache, block_table, q_req, q_pos, n_rows, n_req, n_pages, s, nullptr,
                                 lists, err_word, cs);
        if (e == cudaSuccess)
            e = launch_topk_merge(lists, q_pos, n_rows, s, score_prefill_chunks(s.max_blocks), sel, mark, err_word,
                                  cs);
    }
    if (e == cudaSuccess)
        e = launch_invert_finish(sel, q_req, n_rows, n_req, s, blk_off, blk_ent, ent_pos, inv_ws, err_word, cs);
    return e == cudaSuccess ? MSA_OK : cuda_fail(e, "msa_select_invert_prefill");
}

msa_status_t msa_topk_blocks(const float *scores, const int32_t *q_pos, int32_t n_rows, const msa_dims_t *dims,
                             int32_t *sel, int32_t *err_word, msa_stream_t stream) {
    Shape s;
    msa_status_t st = check_dims(dims, false, false, &s, "msa_topk_blocks");
    if (st != MSA_OK) return st;
    MSA_REQUIRE(n_rows >= 0, "msa_topk_blocks: n_rows < 0");
    if (n_rows == 0) return MSA_OK;
    MSA_REQUIRE(scores && q_pos && sel && err_word, "msa_topk_blocks: NULL pointer");
    if (s.max_blocks > 16384) return fail(MSA_ERR_UNSUPPORTED, "msa_topk_blocks: max_blocks > 16384");
    cudaError_t e = launch_topk(scores, q_pos, n_rows, s, sel, err_word, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MSA_OK : cuda_fail(e, "msa_topk_blocks");
}

msa_status_t msa_build_page_table(const int32_t *sel, const int32_t *block_table, const int32_t *seq_lens, int32_t B,
                                  int32_t n_pages, const msa_dims_t *dims, int32_t *page_table, int32_t *row_len,
                                  int32_t *err_word, msa_stream_t stream) {
    Shape s;
    msa_status_t st = check_dims(dims, false, false, &s, "msa_build_page_table");
    if (st != MSA_OK) return st;
    MSA_REQUIRE(B >= 0 && n_pages > 0, "msa_build_page_table: bad sizes");
    if (B == 0) return MSA_OK;
    MSA_REQUIRE(sel && block_table && seq_lens && page_table && row_len && err_word,
                "msa_build_page_table: NULL pointer");
    cudaError_t e = launch_page_table(sel, block_table, seq_lens, B, n_pages, s, page_table, row_len, err_word,
                                      static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MSA_OK : cuda_fail(e, "msa_build_page_table");
}

msa_status_t msa_invert_selection(const int32_t *sel, const int32_t *q_req, int32_t n_rows, int32_t n_req,
                                  const msa_dims_t *dims, int32_t *blk_off, int32_t *blk_ent, int32_t *ent_pos,
                                  void *workspace, size_t workspace_bytes, int32_t *err_word,
                                  msa_stream_t stream) {
    Shape s;
    msa_status_t st = check_dims(dims, false, false, &s, "msa_invert_selection");
    if (st != MSA_OK) return st;
    MSA_REQUIRE(n_rows >= 0 && n_req > 0, "msa_invert_selection: bad sizes");
    MSA_REQUIRE(sel || n_rows == 0, "msa_invert_selection: NULL sel");
    MSA_REQUIRE(q_req || n_rows == 0, "msa_invert_selection: NULL q_req");
    MSA_REQUIRE(blk_off && err_word, "msa_invert_selection: NULL pointer");
    MSA_REQUIRE(blk_ent || n_rows == 0, "msa_invert_selection: NULL blk_ent");
    MSA_REQUIRE(ent_pos || n_rows == 0, "msa_invert_selection: NULL ent_pos");
    if (1.0 * n_rows * s.G * s.topk > 2147483647.0)
        return fail(MSA_ERR_UNSUPPORTED, "msa_invert_selection: more than 2^31 entries");
    const size_t need = invert_workspace_bytes(n_rows, n_req, s);
    if (!workspace || workspace_bytes < need)
        return fail(MSA_ERR_WORKSPACE, "msa_invert_selection: workspace needs %zu bytes", need);
    cudaError_t e = launch_invert(sel, q_req, n_rows, n_req, s, blk_off, blk_ent, ent_pos, workspace, err_word,
                                  static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MSA_OK : cuda_fail(e, "msa_invert_selection");
}

msa_status_t msa_sparse_attn_prefill(const void *q, const void *k_cache, const void *v_cache,
                                     const int32_t *block_table, const int32_t *q_req, const int32_t *q_pos,
                                     const int32_t *blk_off, const int32_t *blk_ent, int32_t n_rows, int32_t n_req,
                                     int32_t n_pages, const msa_dims_t *dims, void *o_part, float *lse_part,
                                     void *workspace, size_t workspace_bytes, int32_t *err_word,
                                     msa_stream_t stream) {
    Shape s;
    msa_status_t st = check_dims(dims, true, false, &s, "msa_sparse_attn_prefill");
    if (st != MSA_OK) return st;
    MSA_REQUIRE(n_rows >= 0 && n_req > 0 && n_pages > 0, "msa_sparse_attn_prefill: bad sizes");
    if (n_rows == 0) return MSA_OK;
    MSA_REQUIRE(q && k_cache && v_cache && block_table && q_req && q_pos && blk_off && blk_ent && o_part &&
                    lse_part && err_word,
                "msa_sparse_attn_prefill: NULL pointer");
    if (1.0 * n_rows * s.G * s.topk > 2147483647.0)
        return fail(MSA_ERR_UNSUPPORTED, "msa_sparse_attn_prefill: more than 2^31 entries");
    const size_t need = prefill_workspace_bytes(n_rows, n_req, s);
    if (!workspace || workspace_bytes < need)
        return fail(MSA_ERR_WORKSPACE, "msa_sparse_attn_prefill: workspace needs %zu bytes", need);
    if (reinterpret_cast<uintptr_t>(workspace) & 15u)
        return fail(MSA_ERR_INVALID_ARG, "msa_sparse_attn_prefill: workspace must be 16-byte aligned");
    cudaError_t e = launch_attn_prefill(q, k_cache, v_cache, block_table, q_req, q_pos, blk_off, blk_ent, n_rows,
                                        n_req, n_pages, s, o_part, lse_part, workspace, err_word,
                                        static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MSA_OK : cuda_fail(e, "msa_sparse_attn_prefill");
}

msa_status_t msa_lse_merge(const void *o_part, const float *lse_part, const int32_t *sel, const int32_t *ent_pos,
                           int32_t n_rows, const msa_dims_t *dims, void *out, float *lse, int32_t *err_word,
                           msa_stream_t stream) {
    Shape s;
    msa_status_t st = check_dims(dims, false, false, &s, "msa_lse_merge");
    if (st != MSA_OK) return st;
    if (s.D != 64 && s.D != 128) return fail(MSA_ERR_UNSUPPORTED, "msa_lse_merge: D must be 64 or 128");
    MSA_REQUIRE(n_rows >= 0, "msa_lse_merge: n_rows < 0");
    if (n_rows == 0) return MSA_OK;
    MSA_REQUIRE(o_part && lse_part && sel && ent_pos && out && lse && err_word, "msa_lse_merge: NULL pointer");
    if (1.0 * n_rows * s.G * s.topk > 2147483647.0)
        return fail(MSA_ERR_UNSUPPORTED, "msa_lse_merge: more than 2^31 entries");
    cudaError_t e = launch_lse_merge(o_part, lse_part, sel, ent_pos, n_rows, s, out, lse, err_word,
                                     static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MSA_OK : cuda_fail(e, "msa_lse_merge");
}

// The device address of page-locked host memory (cudaHostAlloc, cudaMallocHost or
// cudaHostRegister), or nullptr for anything else.  Pageable memory is addressable by the GPU
// on some systems (address translation over the host link) but not on all, and the driver's
// host-pointer lookup accepts it there, so the memory type is checked instead.
static void *pinned_device_ptr(const void *p) {
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

// Decode results (out, lse) may live in device memory or in page-locked host memory; in the
// latter case the attention kernel writes them straight into it over the host link.  *dev gets
// the address the kernel writes through; anything else is refused.
static msa_status_t result_ptr(void *p, void **dev, const char *who) {
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return fail(MSA_ERR_INVALID_ARG, "%s: out and lse must be device or page-locked host memory", who);
    }
    if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) {
        *dev = p;
        return MSA_OK;
    }
    if (a.type == cudaMemoryTypeHost && a.devicePointer) {
        *dev = a.devicePointer;
        return MSA_OK;
    }
    return fail(MSA_ERR_INVALID_ARG, "%s: out and lse must be device or page-locked host memory", who);
}

msa_status_t msa_sparse_attn_decode(const void *q, const void *k_cache, const void *v_cache,
                                    const int32_t *page_table, const int32_t *row_len, int32_t B, int32_t n_pages,
                                    const msa_dims_t *dims, void *out, float *lse, void *workspace,
                                    size_t workspace_bytes, int32_t *err_word, msa_stream_t stream) {
    Shape s;
    msa_status_t st = check_dims(dims, true, false, &s, "msa_sparse_attn_decode");
    if (st != MSA_OK) return st;
    MSA_REQUIRE(B >= 0 && n_pages > 0, "msa_sparse_attn_decode: bad sizes");
    if (B == 0) return MSA_OK;
    MSA_REQUIRE(q && k_cache && v_cache && page_table && row_len && out && lse && err_word,
                "msa_sparse_attn_decode: NULL pointer");
    if (1LL * B * s.G > 65535) return fail(MSA_ERR_UNSUPPORTED, "msa_sparse_attn_decode: B*G > 65535");
    const size_t need = decode_workspace_bytes(B, s);
    if (!workspace || workspace_bytes < need)
        return fail(MSA_ERR_WORKSPACE, "msa_sparse_attn_decode: workspace needs %zu bytes", need);
    if ((reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache)) & 15u)
        return fail(MSA_ERR_INVALID_ARG, "msa_sparse_attn_decode: caches must be 16-byte aligned");
    void *out_d = nullptr, *lse_d = nullptr;
    if ((st = result_ptr(out, &out_d, "msa_sparse_attn_decode")) != MSA_OK) return st;
    if ((st = result_ptr(lse, &lse_d, "msa_sparse_attn_decode")) != MSA_OK) return st;
    cudaError_t e = launch_attn_decode(q, k_cache, v_cache, page_table, row_len, B, n_pages, s, out_d,
                                       static_cast<float *>(lse_d), workspace, err_word,
                                       static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MSA_OK : cuda_fail(e, "msa_sparse_attn_decode");
}

msa_status_t msa_offload_gather(const void *host_k_cache, const void *host_v_cache, int32_t n_host_pages,
                                const int32_t *page_table, int32_t B, const msa_dims_t *dims, void *pool_k,
                                void *pool_v, int32_t *pool_page_table, int32_t *err_word, msa_stream_t stream) {
    Shape s;
    msa_status_t st = check_dims(dims, true, false, &s, "msa_offload_gather");
    if (st != MSA_OK) return st;
    MSA_REQUIRE(B >= 0 && n_host_pages > 0, "msa_offload_gather: bad sizes");
    if (B == 0) return MSA_OK;
    MSA_REQUIRE(host_k_cache && host_v_cache && page_table && pool_k && pool_v && pool_page_table && err_word,
                "msa_offload_gather: NULL pointer");
    if ((reinterpret_cast<uintptr_t>(host_k_cache) | reinterpret_cast<uintptr_t>(host_v_cache) |
         reinterpret_cast<uintptr_t>(pool_k) | reinterpret_cast<uintptr_t>(pool_v)) & 15u)
        return fail(MSA_ERR_INVALID_ARG, "msa_offload_gather: caches and pools must be 16-byte aligned");
    // the GPU reads the host caches in place: they must be page-locked and mapped
    void *dk = pinned_device_ptr(host_k_cache), *dv = pinned_device_ptr(host_v_cache);
    if (!dk || !dv) return fail(MSA_ERR_INVALID_ARG, "msa_offload_gather: host caches must be page-locked host memory");
    cudaError_t e = launch_offload_gather(dk, dv, page_table, B, n_host_pages, s, pool_k, pool_v, pool_page_table,
                                          err_word, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MSA_OK : cuda_fail(e, "msa_offload_gather");
}

msa_status_t msa_stage_from_host(const void *host_src, void *dev_dst, size_t bytes, msa_stream_t stream) {
    if (bytes == 0) return MSA_OK;
    MSA_REQUIRE(host_src && dev_dst, "msa_stage_from_host: NULL pointer");
    if (((reinterpret_cast<uintptr_t>(host_src) | reinterpret_cast<uintptr_t>(dev_dst)) & 15u) || (bytes & 15u))
        return fail(MSA_ERR_INVALID_ARG, "msa_stage_from_host: pointers and size must be multiples of 16 bytes");
    // the kernel reads the host buffer in place: it must be page-locked and mapped
    void *src = pinned_device_ptr(host_src);
    if (!src) return fail(MSA_ERR_INVALID_ARG, "msa_stage_from_host: the source must be page-locked host memory");
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, dev_dst) != cudaSuccess ||
        (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged)) {
        cudaGetLastError();
        return fail(MSA_ERR_INVALID_ARG, "msa_stage_from_host: the destination must be device memory");
    }
    const cudaError_t e = launch_stage_from_host(src, dev_dst, bytes, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MSA_OK : cuda_fail(e, "msa_stage_from_host");
}

msa_status_t msa_decode_step(const void *q, const void *q_idx, const void *k_cache, const void *v_cache,
                             const void *kidx_cache, const int32_t *block_table, const int32_t *seq_lens, int32_t B,
                             int32_t n_pages, const msa_dims_t *dims, float *scores, int32_t *sel,
                             int32_t *page_table, int32_t *row_len, void *out, float *lse, void *workspace,
                             size_t workspace_bytes, int32_t *err_word, msa_stream_t stream) {
    Shape s;
    msa_status_t st = check_dims(dims, true, true, &s, "msa_decode_step");
    if (st != MSA_OK) return st;
    MSA_REQUIRE(B >= 0 && n_pages > 0, "msa_decode_step: bad sizes");
    if (B == 0) return MSA_OK;
    MSA_REQUIRE(q && q_idx && k_cache && v_cache && kidx_cache && block_table && seq_lens && scores && sel &&
                    page_table && row_len && out && lse && err_word,
                "msa_decode_step: NULL pointer");
    if (1LL * B * s.G > 65535) return fail(MSA_ERR_UNSUPPORTED, "msa_decode_step: B*G > 65535");
    if (s.max_blocks > 16384) return fail(MSA_ERR_UNSUPPORTED, "msa_decode_step: max_blocks > 16384");
    const size_t need = decode_workspace_bytes(B, s);
    if (!workspace || workspace_bytes < need)
        return fail(MSA_ERR_WORKSPACE, "msa_decode_step: workspace needs %zu bytes", need);
    if ((reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache)) & 15u)
        return fail(MSA_ERR_INVALID_ARG, "msa_decode_step: caches must be 16-byte aligned");
    void *out_d = nullptr, *lse_d = nullptr;
    if ((st = result_ptr(out, &out_d, "msa_decode_step")) != MSA_OK) return st;
    if ((st = result_ptr(lse, &lse_d, "msa_decode_step")) != MSA_OK) return st;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    // the scan may start while the kernel before it on the stream (say, the one staging this step's
    // inputs) drains; it reads nothing until that kernel completes
    cudaError_t e = launch_score_decode_seq(q_idx, kidx_cache, block_table, seq_lens, B, n_pages, s, scores,
                                            err_word, cs, true);
    if (e != cudaSuccess) return cuda_fail(e, "msa_decode_step (index scan)");
    int32_t *counters = decode_ws_counters(workspace, B, s);
    e = launch_decode_select(scores, seq_lens, block_table, B, n_pages, s, sel, page_table, row_len, counters,
                             err_word, cs, true);
    if (e != cudaSuccess) return cuda_fail(e, "msa_decode_step (selection)");
    e = launch_attn_decode(q, k_cache, v_cache, page_table, row_len, B, n_pages, s, out_d, static_cast<float *>(lse_d),
                           workspace, err_word, cs, true, true);
    return e == cudaSuccess ? MSA_OK : cuda_fail(e, "msa_decode_step (attention)");
}

size_t msa_workspace_bytes(int32_t op, int32_t n_rows, int32_t n_req, const msa_dims_t *dims) {
    Shape s;
    if (n_rows < 0) return 0;
    if (op == MSA_OP_INVERT) {
        if (check_dims(dims, false, false, &s, "msa_workspace_bytes") != MSA_OK || n_req <= 0) return 0;
        return invert_workspace_bytes(n_rows, n_req, s);
    }
    if (op == MSA_OP_DECODE) {
        if (check_dims(dims, true, false, &s, "msa_workspace_bytes") != MSA_OK) return 0;
        return decode_workspace_bytes(n_rows, s);
    }
    if (op == MSA_OP_PREFILL) {
        if (check_dims(dims, true, false, &s, "msa_workspace_bytes") != MSA_OK || n_req <= 0) return 0;
        return prefill_workspace_bytes(n_rows, n_req, s);
    }
    if (op == MSA_OP_SELECT_PREFILL) {
        if (check_dims(dims, false, true, &s, "msa_workspace_bytes") != MSA_OK) return 0;
        return size_t(n_rows) * s.G * score_prefill_chunks(s.max_blocks) * kSelectListLen * sizeof(uint64_t);
    }
    if (op == MSA_OP_SELECT_INVERT_PREFILL) {
        if (check_dims(dims, false, true, &s, "msa_workspace_bytes") != MSA_OK || n_req <= 0) return 0;
        return select_lists_bytes(n_rows, s) + invert_workspace_bytes(n_rows, n_req, s);
    }
    return 0;
}

msa_status_t msa_check(int32_t *err_word, msa_stream_t stream) {
    if (!err_word) return fail(MSA_ERR_INVALID_ARG, "msa_check: NULL err_word");
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    int32_t h = 0;
    cudaError_t e = cudaMemcpyAsync(&h, err_word, sizeof h, cudaMemcpyDeviceToHost, cs);
    if (e == cudaSuccess) e = cudaStreamSynchronize(cs);
    if (e == cudaSuccess) e = cudaMemsetAsync(err_word, 0, sizeof h, cs);
    if (e != cudaSuccess) return cuda_fail(e, "msa_check");
    if (h & MSA_FLAG_BOUNDS) return fail(MSA_ERR_DEVICE_BOUNDS, "device: index out of range (word 0x%x)", h);
    if (h & MSA_FLAG_NAN) return fail(MSA_ERR_DEVICE_BOUNDS, "device: NaN block score (word 0x%x)", h);
    if (h & MSA_FLAG_TIMEOUT) return fail(MSA_ERR_TIMEOUT, "device: bounded wait expired (word 0x%x)", h);
    if (h & MSA_FLAG_UNSUPPORTED)
        return fail(MSA_ERR_DEVICE_UNSUPPORTED, "device: unsupported layout (word 0x%x)", h);
    return MSA_OK;
}

const char *msa_status_str(msa_status_t status) {
    switch (status) {
        case MSA_OK: return "MSA_OK";
        case MSA_ERR_INVALID_ARG: return "MSA_ERR_INVALID_ARG";
        case MSA_ERR_UNSUPPORTED: return "MSA_ERR_UNSUPPORTED";
        case MSA_ERR_CUDA: return "MSA_ERR_CUDA";
        case MSA_ERR_DEVICE_BOUNDS: return "MSA_ERR_DEVICE_BOUNDS";
        case MSA_ERR_TIMEOUT: return "MSA_ERR_TIMEOUT";
        case MSA_ERR_WORKSPACE: return "MSA_ERR_WORKSPACE";
        case MSA_ERR_DEVICE_UNSUPPORTED: return "MSA_ERR_DEVICE_UNSUPPORTED";
    }
    return "MSA_ERR_UNKNOWN";
}

const char *msa_last_error(void) { return g_last_error; }

int32_t msa_version(void) { return 300; }

msa_status_t msa_selftest_timeout(int32_t *err_word, msa_stream_t stream) {
    MSA_REQUIRE(err_word, "msa_selftest_timeout: NULL err_word");
    const cudaError_t e = launch_selftest_timeout(err_word, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MSA_OK : cuda_fail(e, "msa_selftest_timeout");
}

}  // extern "C"
