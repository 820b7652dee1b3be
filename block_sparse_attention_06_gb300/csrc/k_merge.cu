// Log-Sum-Exp merge of per-block partial outputs (prefill).
//
// "Together AI 解析如何高效服务 MiniMax M3…", section KV 块主序稀疏注意力: because the
// block-major kernel only produces a partial O per KV block, a final reduction
// based on Log-Sum-Exp rescales the partial outputs and sums them.  The partials
// are stored in CSR-entry order (the order in which the block-major kernel
// produces them); ent_pos maps each (row, group, slot) to its entry.  Within an
// entry's HPG x D block the 16-byte column chunk is the outer index and the head
// the inner one.  One CTA per query row gathers that row's G * topk partial blocks
// with 16-byte loads; its threads take heads fastest, so a warp's loads for one
// slot are contiguous (HPG heads x 32/HPG chunks).
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
    extern __shared__ float sh[];   // w_s [topk][Hq]: each slot's lse, then its weight exp(lse_s - lse)
                                    // (0 for empty slots); pos_s [G][topk] entry of each (group, slot),
                                    // -1 if empty
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
    // every (slot, head) lse of the row into shared memory, all loads independent
    for (int i = tid; i < topk * Hq; i += blockDim.x) {
        const int s = i / Hq, h = i - (i / Hq) * Hq;
        const int g = h / hpg, hh = h - g * hpg;
        const int p = pos_s[g * topk + s];
        w_s[i] = p >= 0 ? lse_part[size_t(p) * hpg + hh] : -INFINITY;
    }
    __syncthreads();
    for (int h = tid; h < Hq; h += blockDim.x) {
        float m = -INFINITY;
        for (int s = 0; s < topk; ++s) m = fmaxf(m, w_s[s * Hq + h]);
        float tot = -INFINITY;
        if (m != -INFINITY) {
            float sum = 0.f;
            for (int s = 0; s < topk; ++s) {
                const float l = w_s[s * Hq + h];
                if (l != -INFINITY) sum += __expf(l - m);
            }
            tot = m + __logf(sum);
        }
        for (int s = 0; s < topk; ++s) {
            const float l = w_s[s * Hq + h];
            w_s[s * Hq + h] = (l != -INFINITY && tot != -INFINITY) ? __expf(l - tot) : 0.f;
        }
        lse[size_t(q) * Hq + h] = tot;
    }
    __syncthreads();
    const int chunks = Hq * (D / 8);
    for (int c = tid; c < chunks; c += blockDim.x) {
        const int hh = c % hpg, rest = c / hpg;
        const int cc = rest % (D / 8), g = rest / (D / 8);
        const int h = g * hpg + hh, col = cc * 8;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        // four slots' loads in flight at a time; an empty slot (weight 0, never written) reads
        // entry 0 instead and is left out by a select, so no stale value can reach the sum
        for (int s0 = 0; s0 < topk; s0 += 4) {
            uint4 v[4];
            float w[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int s = s0 + i;
                w[i] = s < topk ? w_s[s * Hq + h] : 0.f;
                const int p = (s < topk && w[i] != 0.f) ? pos_s[g * topk + s] : 0;
                v[i] = *reinterpret_cast<const uint4 *>(o_part + size_t(p) * hpg * D + (size_t(cc) * hpg + hh) * 8);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                if (w[i] == 0.f) continue;
                acc[0] = fmaf(w[i], bf16_lo(v[i].x), acc[0]);
                acc[1] = fmaf(w[i], bf16_hi(v[i].x), acc[1]);
                acc[2] = fmaf(w[i], bf16_lo(v[i].y), acc[2]);
                acc[3] = fmaf(w[i], bf16_hi(v[i].y), acc[3]);
                acc[4] = fmaf(w[i], bf16_lo(v[i].z), acc[4]);
                acc[5] = fmaf(w[i], bf16_hi(v[i].z), acc[5]);
                acc[6] = fmaf(w[i], bf16_lo(v[i].w), acc[6]);
                acc[7] = fmaf(w[i], bf16_hi(v[i].w), acc[7]);
            }
        }
        uint4 r;
        r.x = pack_bf16x2(acc[0], acc[1]);
        r.y = pack_bf16x2(acc[2], acc[3]);
        r.z = pack_bf16x2(acc[4], acc[5]);
        r.w = pack_bf16x2(acc[6], acc[7]);
        *reinterpret_cast<uint4 *>(out + (size_t(q) * Hq + h) * D + col) = r;
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
