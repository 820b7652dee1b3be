// msa_sparse_attn_decode_noalloc: the decode attention entry point for callers
// that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at all.  One example is a serving engine
// that reserves nearly all HBM for its paged KV pool at start-up and routes every
// later allocation through its own allocator.  Another is a plugin host that
// forbids libraries from calling the CUDA allocator: cudaMalloc can synchronise
// the device and fails once the pool is reserved.  Such callers also cannot hand
// us a workspace.  This variant therefore keeps the segment partials in a
// file-scope device array of fixed size instead of a caller-provided workspace.
//
// The array exists once per GPU that uses the library and stays allocated until
// the process exits.  With CUDA's lazy module loading (the default), the device
// memory behind it is reserved when the library's module is first loaded on a
// device, which is this entry point's first call there (the address lookup
// below), not when the library is opened.  A caller that reserves nearly all HBM
// for its own pool must therefore make that first call before it reserves the
// pool; otherwise the lookup can fail for lack of memory, and the call returns
// MSA_ERR_CUDA saying so.
//
// The address is looked up once per device and kept.  After cudaDeviceReset the
// module is loaded again, possibly at another address, so a process that resets
// a device must not call this entry point on it again.
//
// Every call uses the same array, so calls whose kernels overlap on the GPU (for
// example on two streams) race on it and must be serialised by the caller.  The
// array keeps what the previous call left in it.  Only the per-row merge
// counters have to start at zero, and msa_sparse_attn_decode clears them on the
// stream before its kernel runs; the partials and their lse are written before
// they are read.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "msa.h"
#include "msa_internal.h"

namespace {

constexpr size_t kScratchBytes = size_t(16) << 20;   // 16 MiB

static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once per
// device (with that device current) and cached.  The host-side symbol is only a
// stand-in and must never be passed to a kernel.
cudaError_t scratch_on_current_device(void **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

msa_status_t fail(msa_status_t st, const char *msg) {
    msa::set_last_error(msg);
    return st;
}

}  // namespace

extern "C" {

msa_status_t msa_sparse_attn_decode_noalloc(const void *q, const void *k_cache, const void *v_cache,
                                            const int32_t *page_table, const int32_t *row_len, int32_t B,
                                            int32_t n_pages, const msa_dims_t *dims, void *out, float *lse,
                                            int32_t *err_word, msa_stream_t stream) {
    if (!dims) return fail(MSA_ERR_INVALID_ARG, "msa_sparse_attn_decode_noalloc: dims is NULL");
    if (B < 0 || n_pages <= 0) return fail(MSA_ERR_INVALID_ARG, "msa_sparse_attn_decode_noalloc: bad sizes");
    if (B == 0) return MSA_OK;
    const size_t need = msa_workspace_bytes(MSA_OP_DECODE, B, 0, dims);
    if (need == 0)
        return fail(MSA_ERR_UNSUPPORTED, "msa_sparse_attn_decode_noalloc: dims rejected (see msa_sparse_attn_decode)");
    if (need > kScratchBytes)
        return fail(MSA_ERR_WORKSPACE,
                    "msa_sparse_attn_decode_noalloc: B * G * topk partials need more than the 16 MiB static "
                    "scratch; use msa_sparse_attn_decode with a workspace");
    void *scratch = nullptr;
    cudaError_t e = scratch_on_current_device(&scratch);
    if (e != cudaSuccess) {
        char msg[384];
        snprintf(msg, sizeof msg,
                 "msa_sparse_attn_decode_noalloc: cudaGetSymbolAddress: %s (the first call on a device loads the "
                 "library's module and its 16 MiB scratch array; make it before reserving the rest of device "
                 "memory)",
                 cudaGetErrorString(e));
        return fail(MSA_ERR_CUDA, msg);
    }
    return msa_sparse_attn_decode(q, k_cache, v_cache, page_table, row_len, B, n_pages, dims, out, lse, scratch,
                                  kScratchBytes, err_word, stream);
}

}  // extern "C"
