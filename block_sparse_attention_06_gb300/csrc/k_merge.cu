// Log-Sum-Exp merge of per-block partial outputs (prefill).
//
// "Together AI 解析如何高效服务 MiniMax M3…", section KV 块主序稀疏注意力: because the
// block-major kernel only produces a partial O per KV block, a final reduction
// based on Log-Sum-Exp rescales the partial outputs and sums them.  The partials
// are stored in CSR-entry order (the order in which the block-major kernel
// produces them); ent_pos maps each (row, group, slot) to its entry.  One CTA
// per query row gathers that row's G * topk partial blocks (HPG heads x D bf16,
// contiguous) with 16-byte loads, coalesced across a block's heads.
#include "msa_device.cuh"
#include "msa_internal.h"

namespace msa {
namespace {

template <int D>
__global__ void __launch_bounds__(256) k_lse_merge(const uint16_t *__restrict__ o_part,
                                                   const float *__restrict__ lse_part,
                                                   const int32_t *__restrict__ sel,
                                                   const int32_t *__restrict__ ent_pos, int Hq, int G,
                                                   int topk, long long n_ent, uint16_t *__restrict__ out,
                                                   float *__restrict__ lse, int32_t *err) {
    extern __shared__ float sh[];   // w_s [topk][Hq] weights exp(lse_s - lse) (0 for empty slots),
                                    // then pos_s [G][topk] entry of each (group, slot), -1 if empty
    float *w_s = sh;
    int32_t *pos_s = reinterpret_cast<int32_t *>(sh + topk * Hq);
    const int q = blockIdx.x;
    const int tid = threadIdx.x;
    const int hpg = Hq / G;
    for (int i = tid; i < G * topk; i += blockDim.x) {
        const size_t at = size_t(q) * G * topk + i;
        int p = -1;
        if (sel[at] >= 0) {
            p = ent_pos[at];
            if (p < 0 || p >= n_ent) {
                raise_flag(err, MSA_FLAG_BOUNDS);
                p = -1;
            }
        }
        pos_s[i] = p;
    }
    __syncthreads();
    for (int h = tid; h < Hq; h += blockDim.x) {
        const int g = h / hpg, hh = h - g * hpg;
        const int32_t *ps = pos_s + g * topk;
        float m = -INFINITY;
        for (int s = 0; s < topk; ++s)
            if (ps[s] >= 0) m = fmaxf(m, lse_part[size_t(ps[s]) * hpg + hh]);
        float tot = -INFINITY;
        if (m != -INFINITY) {
            float sum = 0.f;
            for (int s = 0; s < topk; ++s)
                if (ps[s] >= 0) sum += __expf(lse_part[size_t(ps[s]) * hpg + hh] - m);
            tot = m + __logf(sum);
        }
        for (int s = 0; s < topk; ++s)
            w_s[s * Hq + h] = (ps[s] >= 0 && tot != -INFINITY) ? __expf(lse_part[size_t(ps[s]) * hpg + hh] - tot)
                                                               : 0.f;
        lse[size_t(q) * Hq + h] = tot;
    }
    __syncthreads();
    const int chunks = Hq * (D / 8);
    for (int c = tid; c < chunks; c += blockDim.x) {
        const int h = c / (D / 8);
        const int g = h / hpg, hh = h - g * hpg;
        const int col = (c - h * (D / 8)) * 8;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int s = 0; s < topk; ++s) {
            const float w = w_s[s * Hq + h];
            if (w == 0.f) continue;   // empty slot: its partial was never written
            const uint4 v = *reinterpret_cast<const uint4 *>(
                o_part + (size_t(pos_s[g * topk + s]) * hpg + hh) * D + col);
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

cudaError_t launch_lse_merge(const void *o_part, const float *lse_part, const int32_t *sel, const int32_t *ent_pos,
                             int n_rows, const Shape &s, void *out, float *lse, int32_t *err, cudaStream_t st) {
    if (n_rows <= 0) return cudaSuccess;
    const size_t smem = size_t(s.topk) * s.Hq * sizeof(float) + size_t(s.G) * s.topk * sizeof(int32_t);
    if (smem > 48 * 1024) return cudaErrorNotSupported;
    const long long n_ent = 1LL * n_rows * s.G * s.topk;
    if (s.D == 128)
        k_lse_merge<128><<<unsigned(n_rows), 256, smem, st>>>(static_cast<const uint16_t *>(o_part), lse_part, sel,
                                                            ent_pos, s.Hq, s.G, s.topk, n_ent,
                                                            static_cast<uint16_t *>(out), lse, err);
    else if (s.D == 64)
        k_lse_merge<64><<<unsigned(n_rows), 256, smem, st>>>(static_cast<const uint16_t *>(o_part), lse_part, sel,
                                                           ent_pos, s.Hq, s.G, s.topk, n_ent,
                                                           static_cast<uint16_t *>(out), lse, err);
    else
        return cudaErrorNotSupported;
    return cudaGetLastError();
}

}  // namespace msa
