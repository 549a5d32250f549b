// seam.cu -- seam-window advance.
//
// At reuse, the first w tokens of each internal segment are not taken from
// the cache: the linear layers compute the window's own transitions on the
// fly, advance the running state through it and emit each seam token's output
// for the full-attention layers above (aibase article on HYPIC, paragraph on
// the full-attention layers; README "PIC modes", seam width PIC_SEAM_SINK,
// default 8).  One CTA per (seam, layer, head); thread j owns column j of
// the dk x dv state in registers and produces o_t[j] = (S_t^T q_t)_j = q_t . col.
// The work is a read and a write of the state plus w tokens: memory-bound.
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"

namespace hypic {

static constexpr int kSeamChunk = 32;

template <int DK, int DV>
__global__ void __launch_bounds__(DK > DV ? DK : DV) seam_simt_kernel(SeamParams p) {
    extern __shared__ float sm[];
    float* qs = sm;                    // [kSeamChunk][DK]
    float* ks = qs + kSeamChunk * DK;  // [kSeamChunk][DK]
    float* vs = ks + kSeamChunk * DK;  // [kSeamChunk][DV]
    float* gs = vs + kSeamChunk * DV;  // [kSeamChunk][DK] (GLA, KDA)
    float* as = gs + kSeamChunk * DK;  // [kSeamChunk]
    float* bs = as + kSeamChunk;       // [kSeamChunk]
    const int LH = p.n_layers * p.n_heads;
    const int r = blockIdx.x / LH, lh = blockIdx.x % LH;
    const int layer = lh / p.n_heads, head = lh % p.n_heads;
    const int c = threadIdx.x;
    const int fam = p.family;
    const int64_t obj = (int64_t)r * LH + lh;
    const float gm = (fam == kRETNET && p.gamma) ? p.gamma[(int64_t)layer * p.n_heads + head] : 1.f;
    float col[DK];
#pragma unroll
    for (int i = 0; i < DK; ++i) col[i] = (p.state_in && c < DV) ? p.state_in[(obj * DK + i) * DV + c] : 0.f;
    const int64_t t_begin = p.cu_seam[r], t_end = p.cu_seam[r + 1];
    for (int64_t t0 = t_begin; t0 < t_end; t0 += kSeamChunk) {
        const int n = (int)((t_end - t0) < kSeamChunk ? (t_end - t0) : kSeamChunk);
        __syncthreads();
        stage_rows<DK>(qs, p.q, p.in_dtype, layer, t0, n, head, p.n_tokens, p.n_heads);
        stage_rows<DK>(ks, p.k, p.in_dtype, layer, t0, n, head, p.n_tokens, p.n_heads);
        stage_rows<DV>(vs, p.v, p.in_dtype, layer, t0, n, head, p.n_tokens, p.n_heads);
        if (fam == kGLA || fam == kKDA) stage_rows<DK>(gs, p.g, kF32, layer, t0, n, head, p.n_tokens, p.n_heads);
        if (fam == kGDN || fam == kMAMBA2) stage_gate(as, p.alpha, layer, t0, n, head, p.n_tokens, p.n_heads, 1.f);
        if (fam == kGDN || fam == kKDA) stage_gate(bs, p.beta, layer, t0, n, head, p.n_tokens, p.n_heads, 1.f);
        __syncthreads();
        if (c < DV) {
            for (int t = 0; t < n; ++t) {
                const float* kt = ks + t * DK;
                const float* qt = qs + t * DK;
                const float vj = vs[t * DV + c];
                if (fam == kGDN || fam == kKDA) {  // KDA: the per-channel gate first, then a = 1
                    if (fam == kKDA) {
                        const float* gt = gs + t * DK;
#pragma unroll
                        for (int i = 0; i < DK; ++i) col[i] *= gt[i];
                    }
                    float u0 = 0.f, u1 = 0.f;
#pragma unroll
                    for (int i = 0; i < DK; i += 2) {
                        u0 = fmaf(kt[i], col[i], u0);
                        u1 = fmaf(kt[i + 1], col[i + 1], u1);
                    }
                    const float a = fam == kKDA ? 1.f : as[t], b = bs[t];
                    const float w = b * (vj - a * (u0 + u1));
#pragma unroll
                    for (int i = 0; i < DK; ++i) col[i] = fmaf(kt[i], w, a * col[i]);
                } else if (fam == kGLA) {
                    const float* gt = gs + t * DK;
#pragma unroll
                    for (int i = 0; i < DK; ++i) col[i] = fmaf(kt[i], vj, gt[i] * col[i]);
                } else {  // RetNet (gamma), Mamba2 (a_t), vanilla (1)
                    const float d = fam == kMAMBA2 ? as[t] : gm;
#pragma unroll
                    for (int i = 0; i < DK; ++i) col[i] = fmaf(kt[i], vj, d * col[i]);
                }
                float o0 = 0.f, o1 = 0.f;
#pragma unroll
                for (int i = 0; i < DK; i += 2) {
                    o0 = fmaf(qt[i], col[i], o0);
                    o1 = fmaf(qt[i + 1], col[i + 1], o1);
                }
                p.o_out[tok_row(layer, t0 + t, head, p.n_tokens, p.n_heads) * DV + c] = o0 + o1;
            }
        }
    }
    if (c < DV) {
        float* so = p.state_out + obj * DK * DV;
#pragma unroll
        for (int i = 0; i < DK; ++i) so[i * DV + c] = col[i];
    }
}

template <int DK, int DV>
static cudaError_t launch_seam_dims(const SeamParams& p, cudaStream_t s) {
    const int64_t grid = (int64_t)p.n_seams * p.n_layers * p.n_heads;
    if (grid == 0) return cudaSuccess;
    const size_t smem = sizeof(float) * (kSeamChunk * (3 * DK + DV) + 2 * kSeamChunk);
    auto kern = seam_simt_kernel<DK, DV>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)grid, DK > DV ? DK : DV, smem, s>>>(p);
    return cudaGetLastError();
}

template <int DK>
static cudaError_t launch_seam_dv(const SeamParams& p, cudaStream_t s) {
    switch (p.dv) {
        case 16: return launch_seam_dims<DK, 16>(p, s);
        case 32: return launch_seam_dims<DK, 32>(p, s);
        case 64: return launch_seam_dims<DK, 64>(p, s);
        case 128: return launch_seam_dims<DK, 128>(p, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_seam(const SeamParams& p, unsigned* /*err*/, cudaStream_t s) {
    switch (p.dk) {
        case 16: return launch_seam_dv<16>(p, s);
        case 32: return launch_seam_dv<32>(p, s);
        case 64: return launch_seam_dv<64>(p, s);
        case 128: return launch_seam_dv<128>(p, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace hypic
