// build_simt.cu -- work plan and the CUDA-core build of the cached pair
// (T_C, S(C|0)) for every family.
//
// The cached pair of a segment C is T_C, the ordered product of C's per-token
// transitions, and S(C|0), the state after C's tokens from a zero start (aibase
// article on HYPIC, paragraph on the linear layers).  This path runs the token
// recurrence itself, one CTA per (segment, layer, head), one thread per column
// of [T | S] with that column in registers: the column update of a token
// needs only the token's key, value and gates (broadcast from shared memory)
// and the column itself, so no thread ever talks to another inside the loop.
#include <cuda_runtime.h>
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace hypic {

static constexpr int kChunk = 64;  // tokens staged in shared memory at a time

size_t build_workspace_bytes(int n_seg) {
    size_t order = ((size_t)n_seg * sizeof(int32_t) + 255) & ~(size_t)255;
    return order + 256;
}

// ------------------------------------------------------------------ plan --
// Longest-body-first order of the segments (ties: lower index first), by rank:
// the rank of segment s is the number of segments that come before it.  Each
// CTA ranks 64 segments, four threads per segment counting over every fourth
// segment of a tile of body lengths staged in shared memory; the four counts
// are summed by shuffles.  Block 0 also zeroes the work counter.
constexpr int kPlanSegs = 64, kPlanThreads = 256, kPlanTile = 1024;

__device__ __forceinline__ int body_len(const int32_t* cu, const int32_t* skip, int s) {
    return cu[s + 1] - cu[s] - (skip ? skip[s] : 0);
}

__global__ void __launch_bounds__(kPlanThreads) build_plan_kernel(const int32_t* __restrict__ cu,
                                                                  const int32_t* __restrict__ skip, int n_seg,
                                                                  int32_t* __restrict__ order,
                                                                  unsigned* __restrict__ counter) {
    __shared__ int len[kPlanTile];
    const int tid = threadIdx.x, part = tid & 3;
    const int s = blockIdx.x * kPlanSegs + (tid >> 2);
    const int ls = s < n_seg ? body_len(cu, skip, s) : 0;
    int rank = 0;
    for (int j0 = 0; j0 < n_seg; j0 += kPlanTile) {
        const int m = n_seg - j0 < kPlanTile ? n_seg - j0 : kPlanTile;
        for (int e = tid; e < m; e += kPlanThreads) len[e] = body_len(cu, skip, j0 + e);
        __syncthreads();
        for (int e = part; e < m; e += 4) {
            const int lj = len[e];
            rank += (lj > ls) || (lj == ls && j0 + e < s);
        }
        __syncthreads();
    }
    rank += __shfl_xor_sync(0xffffffffu, rank, 1);
    rank += __shfl_xor_sync(0xffffffffu, rank, 2);
    if (part == 0 && s < n_seg) order[rank] = s;
    if (blockIdx.x == 0 && tid == 0) counter[0] = 0u;
}

cudaError_t launch_build_plan(const BuildParams& p, void* workspace, cudaStream_t s) {
    int32_t* order = reinterpret_cast<int32_t*>(workspace);
    unsigned* counter = reinterpret_cast<unsigned*>(reinterpret_cast<char*>(workspace) +
                                                    build_workspace_bytes(p.n_seg) - 256);
    if (p.n_seg > 0)
        build_plan_kernel<<<(p.n_seg + kPlanSegs - 1) / kPlanSegs, kPlanThreads, 0, s>>>(p.cu, p.skip, p.n_seg, order,
                                                                                          counter);
    return cudaGetLastError();
}

// ------------------------------------------------------ GDN, KDA (SIMT) --
// Thread c < DK owns column c of T (starts as e_c); thread DK + j owns column j
// of S (starts at 0).  Per token: u = k^T col, col <- a (col - b u k) + b v_j k
// (the write term only in the S columns).  KDA first scales the column by its
// per-channel gate, col_i <- a_t[i] col_i, then takes the same step with a = 1.  After every staged chunk the T
// columns are rescaled by a power of two so that their largest entry lies in
// [1, 2); the exponent is accumulated and stored with T (T_C = T_out 2^T_exp).
template <int DK, int DV>
__global__ void __launch_bounds__(DK + DV) gdn_build_simt_kernel(BuildParams p, const int32_t* __restrict__ order) {
    extern __shared__ float sm[];
    float* ks = sm;                    // [kChunk][DK]
    float* vs = ks + kChunk * DK;      // [kChunk][DV]
    float* as = vs + kChunk * DV;      // [kChunk]
    float* bs = as + kChunk;           // [kChunk]
    float* red = bs + kChunk;          // [32]
    float* gs = red + 32;              // [kChunk][DK] (KDA)
    const bool kda = p.family == kKDA;
    const int LH = p.n_layers * p.n_heads;
    const int seg = order[blockIdx.x / LH];
    const int lh = blockIdx.x % LH, layer = lh / p.n_heads, head = lh % p.n_heads;
    const int64_t b0 = (int64_t)p.cu[seg] + (p.skip ? p.skip[seg] : 0), b1 = p.cu[seg + 1];
    const int c = threadIdx.x;
    const bool isT = c < DK;
    float col[DK];
#pragma unroll
    for (int i = 0; i < DK; ++i) col[i] = (isT && i == c) ? 1.f : 0.f;
    int texp = 0;
    for (int64_t t0 = b0; t0 < b1; t0 += kChunk) {
        const int n = (int)((b1 - t0) < kChunk ? (b1 - t0) : kChunk);
        __syncthreads();
        stage_rows<DK>(ks, p.k, p.in_dtype, layer, t0, n, head, p.n_tokens, p.n_heads);
        stage_rows<DV>(vs, p.v, p.in_dtype, layer, t0, n, head, p.n_tokens, p.n_heads);
        if (kda)
            stage_rows<DK>(gs, p.g, kF32, layer, t0, n, head, p.n_tokens, p.n_heads);
        else
            stage_gate(as, p.alpha, layer, t0, n, head, p.n_tokens, p.n_heads, 1.f);
        stage_gate(bs, p.beta, layer, t0, n, head, p.n_tokens, p.n_heads, 1.f);
        __syncthreads();
        for (int t = 0; t < n; ++t) {
            const float4* kt = reinterpret_cast<const float4*>(ks + t * DK);
            float u0 = 0.f, u1 = 0.f, u2 = 0.f, u3 = 0.f;
            if (kda) {  // the per-channel gate applied to the column as the dot product reads it
                const float4* gt = reinterpret_cast<const float4*>(gs + t * DK);
#pragma unroll
                for (int i = 0; i < DK / 4; ++i) {
                    const float4 k4 = kt[i], g4 = gt[i];
                    col[4 * i] *= g4.x, col[4 * i + 1] *= g4.y, col[4 * i + 2] *= g4.z, col[4 * i + 3] *= g4.w;
                    u0 = fmaf(k4.x, col[4 * i], u0);
                    u1 = fmaf(k4.y, col[4 * i + 1], u1);
                    u2 = fmaf(k4.z, col[4 * i + 2], u2);
                    u3 = fmaf(k4.w, col[4 * i + 3], u3);
                }
            } else {
#pragma unroll
                for (int i = 0; i < DK / 4; ++i) {
                    const float4 k4 = kt[i];
                    u0 = fmaf(k4.x, col[4 * i], u0);
                    u1 = fmaf(k4.y, col[4 * i + 1], u1);
                    u2 = fmaf(k4.z, col[4 * i + 2], u2);
                    u3 = fmaf(k4.w, col[4 * i + 3], u3);
                }
            }
            const float u = (u0 + u1) + (u2 + u3);
            const float a = kda ? 1.f : as[t], b = bs[t];
            const float w = isT ? -a * b * u : b * (vs[t * DV + (c - DK)] - a * u);
            if (kda) {
#pragma unroll
                for (int i = 0; i < DK / 4; ++i) {
                    const float4 k4 = kt[i];
                    col[4 * i] = fmaf(k4.x, w, col[4 * i]);
                    col[4 * i + 1] = fmaf(k4.y, w, col[4 * i + 1]);
                    col[4 * i + 2] = fmaf(k4.z, w, col[4 * i + 2]);
                    col[4 * i + 3] = fmaf(k4.w, w, col[4 * i + 3]);
                }
            } else {
#pragma unroll
                for (int i = 0; i < DK / 4; ++i) {
                    const float4 k4 = kt[i];
                    col[4 * i] = fmaf(k4.x, w, a * col[4 * i]);
                    col[4 * i + 1] = fmaf(k4.y, w, a * col[4 * i + 1]);
                    col[4 * i + 2] = fmaf(k4.z, w, a * col[4 * i + 2]);
                    col[4 * i + 3] = fmaf(k4.w, w, a * col[4 * i + 3]);
                }
            }
        }
        float m = 0.f;
        if (isT)
#pragma unroll
            for (int i = 0; i < DK; ++i) m = fmaxf(m, fabsf(col[i]));
        m = block_max(m, red);
        if (m > 0.f && isfinite(m)) {
            const int e = ilogbf(m);
            if (e != 0) {
                if (isT)
#pragma unroll
                    for (int i = 0; i < DK; ++i) col[i] = ldexpf(col[i], -e);
                texp += e;
            }
        }
    }
    const int64_t obj = ((int64_t)seg * p.n_layers + layer) * p.n_heads + head;
    if (isT) {
        float* T = p.T_out + obj * DK * DK;
#pragma unroll
        for (int i = 0; i < DK; ++i) T[i * DK + c] = col[i];
        if (c == 0) p.T_exp[obj] = texp;
    } else {
        float* S = p.S_out + obj * DK * DV;
#pragma unroll
        for (int i = 0; i < DK; ++i) S[i * DV + (c - DK)] = col[i];
    }
}

// ------------------------------------------------- decay families (SIMT) --
// Thread j < DV owns column j of S.  RetNet: col <- g col + v_j k; Mamba2:
// col <- a_t col + v_j k; GLA: col_i <- g_t[i] col_i + v_j k_i; vanilla:
// col <- col + v_j k.  T: RetNet g^L, Mamba2 prod_t a_t (thread 0, in
// double), GLA prod_t g_t (thread i < DK keeps row i's product in double).
template <int DK, int DV>
__global__ void __launch_bounds__(DK > DV ? DK : DV) decay_build_simt_kernel(BuildParams p,
                                                                             const int32_t* __restrict__ order) {
    extern __shared__ float sm[];
    float* ks = sm;                // [kChunk][DK]
    float* vs = ks + kChunk * DK;  // [kChunk][DV]
    float* gs = vs + kChunk * DV;  // [kChunk][DK] (GLA)
    float* as = gs + kChunk * DK;  // [kChunk] (Mamba2)
    const int LH = p.n_layers * p.n_heads;
    const int seg = order[blockIdx.x / LH];
    const int lh = blockIdx.x % LH, layer = lh / p.n_heads, head = lh % p.n_heads;
    const int64_t b0 = (int64_t)p.cu[seg] + (p.skip ? p.skip[seg] : 0), b1 = p.cu[seg + 1];
    const int c = threadIdx.x;
    const int fam = p.family;
    const float gm = (fam == kRETNET && p.gamma) ? p.gamma[(int64_t)layer * p.n_heads + head] : 1.f;
    float col[DK];
#pragma unroll
    for (int i = 0; i < DK; ++i) col[i] = 0.f;
    double tprod = 1.0;
    for (int64_t t0 = b0; t0 < b1; t0 += kChunk) {
        const int n = (int)((b1 - t0) < kChunk ? (b1 - t0) : kChunk);
        __syncthreads();
        stage_rows<DK>(ks, p.k, p.in_dtype, layer, t0, n, head, p.n_tokens, p.n_heads);
        stage_rows<DV>(vs, p.v, p.in_dtype, layer, t0, n, head, p.n_tokens, p.n_heads);
        if (fam == kGLA) stage_rows<DK>(gs, p.g, kF32, layer, t0, n, head, p.n_tokens, p.n_heads);
        if (fam == kMAMBA2) stage_gate(as, p.alpha, layer, t0, n, head, p.n_tokens, p.n_heads, 1.f);
        __syncthreads();
        if (c < DV) {
            for (int t = 0; t < n; ++t) {
                const float4* kt = reinterpret_cast<const float4*>(ks + t * DK);
                const float vj = vs[t * DV + c];
                if (fam == kGLA) {
                    const float4* gt = reinterpret_cast<const float4*>(gs + t * DK);
#pragma unroll
                    for (int i = 0; i < DK / 4; ++i) {
                        const float4 k4 = kt[i], g4 = gt[i];
                        col[4 * i] = fmaf(k4.x, vj, g4.x * col[4 * i]);
                        col[4 * i + 1] = fmaf(k4.y, vj, g4.y * col[4 * i + 1]);
                        col[4 * i + 2] = fmaf(k4.z, vj, g4.z * col[4 * i + 2]);
                        col[4 * i + 3] = fmaf(k4.w, vj, g4.w * col[4 * i + 3]);
                    }
                } else {  // Mamba2 (a_t), RetNet (gamma), vanilla (1)
                    const float d = fam == kMAMBA2 ? as[t] : gm;
#pragma unroll
                    for (int i = 0; i < DK / 4; ++i) {
                        const float4 k4 = kt[i];
                        col[4 * i] = fmaf(k4.x, vj, d * col[4 * i]);
                        col[4 * i + 1] = fmaf(k4.y, vj, d * col[4 * i + 1]);
                        col[4 * i + 2] = fmaf(k4.z, vj, d * col[4 * i + 2]);
                        col[4 * i + 3] = fmaf(k4.w, vj, d * col[4 * i + 3]);
                    }
                }
            }
        }
        if (fam == kGLA && c < DK)
            for (int t = 0; t < n; ++t) tprod *= (double)gs[t * DK + c];
        if (fam == kMAMBA2 && c == 0)
            for (int t = 0; t < n; ++t) tprod *= (double)as[t];
    }
    const int64_t obj = ((int64_t)seg * p.n_layers + layer) * p.n_heads + head;
    if (c < DV) {
        float* S = p.S_out + obj * DK * DV;
#pragma unroll
        for (int i = 0; i < DK; ++i) S[i * DV + c] = col[i];
    }
    if (fam == kGLA && c < DK) p.T_out[obj * DK + c] = (float)tprod;
    if (fam == kRETNET && c == 0) p.T_out[obj] = (float)pow((double)gm, (double)(b1 - b0));
    if (fam == kMAMBA2 && c == 0) p.T_out[obj] = (float)tprod;
}

template <int DK, int DV>
static cudaError_t launch_simt_dims(const BuildParams& p, const int32_t* order, cudaStream_t s) {
    const int64_t grid = (int64_t)p.n_seg * p.n_layers * p.n_heads;
    if (grid == 0) return cudaSuccess;
    if (p.family == kGDN || p.family == kKDA) {
        const size_t smem = sizeof(float) * (kChunk * (DK + DV) + 2 * kChunk + 32 + (p.family == kKDA ? kChunk * DK : 0));
        auto kern = gdn_build_simt_kernel<DK, DV>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        kern<<<(unsigned)grid, DK + DV, smem, s>>>(p, order);
    } else {
        const size_t smem = sizeof(float) * (kChunk * (2 * DK + DV) + kChunk);
        auto kern = decay_build_simt_kernel<DK, DV>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        kern<<<(unsigned)grid, DK > DV ? DK : DV, smem, s>>>(p, order);
    }
    return cudaGetLastError();
}

template <int DK>
static cudaError_t launch_simt_dv(const BuildParams& p, const int32_t* order, cudaStream_t s) {
    switch (p.dv) {
        case 16: return launch_simt_dims<DK, 16>(p, order, s);
        case 32: return launch_simt_dims<DK, 32>(p, order, s);
        case 64: return launch_simt_dims<DK, 64>(p, order, s);
        case 128: return launch_simt_dims<DK, 128>(p, order, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_build_simt(const BuildParams& p, const void* workspace, unsigned* /*err*/, cudaStream_t s) {
    const int32_t* order = reinterpret_cast<const int32_t*>(workspace);
    switch (p.dk) {
        case 16: return launch_simt_dv<16>(p, order, s);
        case 32: return launch_simt_dv<32>(p, order, s);
        case 64: return launch_simt_dv<64>(p, order, s);
        case 128: return launch_simt_dv<128>(p, order, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace hypic
