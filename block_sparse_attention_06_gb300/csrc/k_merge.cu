// Log-Sum-Exp merge of per-block partial outputs (prefill).
//
// "Together AI 解析如何高效服务 MiniMax M3…", section KV 块主序稀疏注意力: because the
// block-major kernel only produces a partial O per KV block, a final reduction
// based on Log-Sum-Exp rescales the partial outputs and sums them.  One CTA per
// query row reads that row's [topk][Hq][D] bf16 partials as one contiguous
// stream (16-byte loads, coalesced across heads), so the kernel runs at HBM rate.
#include "msa_device.cuh"
#include "msa_internal.h"

namespace msa {
namespace {

template <int D>
__global__ void __launch_bounds__(256) k_lse_merge(const uint16_t *__restrict__ o_part,
                                                   const float *__restrict__ lse_part,
                                                   const int32_t *__restrict__ sel, int Hq, int G,
                                                   int topk, uint16_t *__restrict__ out,
                                                   float *__restrict__ lse) {
    extern __shared__ float w_s[];   // [topk][Hq] weights exp(lse_s - lse), 0 for empty slots
    const int q = blockIdx.x;
    const int tid = threadIdx.x;
    const int hpg = Hq / G;
    for (int h = tid; h < Hq; h += blockDim.x) {
        const int g = h / hpg;
        const int32_t *sq = sel + (size_t(q) * G + g) * topk;
        const float *lq = lse_part + size_t(q) * topk * Hq + h;
        float m = -INFINITY;
        for (int s = 0; s < topk; ++s)
            if (sq[s] >= 0) m = fmaxf(m, lq[size_t(s) * Hq]);
        float tot = -INFINITY;
        if (m != -INFINITY) {
            float sum = 0.f;
            for (int s = 0; s < topk; ++s)
                if (sq[s] >= 0) sum += __expf(lq[size_t(s) * Hq] - m);
            tot = m + __logf(sum);
        }
        for (int s = 0; s < topk; ++s)
            w_s[s * Hq + h] = (sq[s] >= 0 && tot != -INFINITY) ? __expf(lq[size_t(s) * Hq] - tot) : 0.f;
        lse[size_t(q) * Hq + h] = tot;
    }
    __syncthreads();
    const int chunks = Hq * (D / 8);
    const uint16_t *op = o_part + size_t(q) * topk * Hq * D;
    for (int c = tid; c < chunks; c += blockDim.x) {
        const int h = c / (D / 8);
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int s = 0; s < topk; ++s) {
            const float w = w_s[s * Hq + h];
            if (w == 0.f) continue;   // empty slot: its partial was never written
            const uint4 v = *reinterpret_cast<const uint4 *>(op + size_t(s) * Hq * D + size_t(c) * 8);
            acc[0] = fmaf(w, bf16_lo(v.x), acc[0]);
            acc[1] = fmaf(w, bf16_hi(v.x), acc[1]);
            acc[2] = fmaf(w, bf16_lo(v.y), acc[2]);
            acc[3] = fmaf(w, bf16_hi(v.y), acc[3]);
            acc[4] = fmaf(w, bf16_lo(v.z), acc[4]);
            acc[5] = fmaf(w, bf16_hi(v.z), acc[5]);
            acc[6] = fmaf(w, bf16_lo(v.w), acc[6]);
            acc[7] = fmaf(w, bf16_hi(v.w), acc[7]);
        }
        uint4 r;
        r.x = pack_bf16x2(acc[0], acc[1]);
        r.y = pack_bf16x2(acc[2], acc[3]);
        r.z = pack_bf16x2(acc[4], acc[5]);
        r.w = pack_bf16x2(acc[6], acc[7]);
        *reinterpret_cast<uint4 *>(out + size_t(q) * Hq * D + size_t(c) * 8) = r;
    }
}

}  // namespace

cudaError_t launch_lse_merge(const void *o_part, const float *lse_part, const int32_t *sel, int n_rows,
                             const Shape &s, void *out, float *lse, int32_t *err, cudaStream_t st) {
    (void)err;
    if (n_rows <= 0) return cudaSuccess;
    const size_t smem = size_t(s.topk) * s.Hq * sizeof(float);
    if (smem > 48 * 1024) return cudaErrorNotSupported;
    if (s.D == 128)
        k_lse_merge<128><<<unsigned(n_rows), 256, smem, st>>>(static_cast<const uint16_t *>(o_part), lse_part, sel,
                                                            s.Hq, s.G, s.topk, static_cast<uint16_t *>(out), lse);
    else if (s.D == 64)
        k_lse_merge<64><<<unsigned(n_rows), 256, smem, st>>>(static_cast<const uint16_t *>(o_part), lse_part, sel,
                                                           s.Hq, s.G, s.topk, static_cast<uint16_t *>(out), lse);
    else
        return cudaErrorNotSupported;
    return cudaGetLastError();
}

}  // namespace msa
