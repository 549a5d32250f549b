// compose_simt.cu -- CUDA-core chain composition of cached pairs.
//
// Composition law of the aibase article on HYPIC (paragraph on the linear
// layers): S(C1.C2) = T(C2) S(C1) + S(C2).  Along a chain the running state is
// S <- T_p S + S_p for each pair p in order.  One CTA per (chain, layer,
// head), thread j owns column j of S in registers; T_p is staged in shared
// memory and read by all threads at the same address (broadcast).
#include <cuda_runtime.h>
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace hypic {

// GDN: dense T_p (dk x dk, stored as mantissa * 2^exp).  The new column is
// written to the thread's own column of a shared buffer and read back, which
// keeps only one column in registers.
template <int D>
__global__ void __launch_bounds__(D) compose_gdn_simt_kernel(ComposeParams p, unsigned* err) {
    extern __shared__ float sm[];
    float* Ts = sm;          // [D][D]
    float* Sn = Ts + D * D;  // [D][D], column c private to thread c
    const int LH = p.n_layers * p.n_heads;
    const int chain = blockIdx.x / LH, lh = blockIdx.x % LH;
    const int c = threadIdx.x;
    const int64_t obj = (int64_t)chain * LH + lh;
    float col[D];
#pragma unroll
    for (int i = 0; i < D; ++i) col[i] = p.S0 ? p.S0[(obj * D + i) * D + c] : 0.f;
    const int j0 = p.cu_chain[chain], j1 = p.cu_chain[chain + 1];
    for (int j = j0; j < j1; ++j) {
        const int pi = p.seg_idx[j];
        if (pi < 0 || pi >= p.n_pairs) {  // host validation makes this unreachable
            set_error(err, kErrBadIndex);
            break;
        }
        const int64_t pobj = (int64_t)pi * LH + lh;
        const float4* Tg = reinterpret_cast<const float4*>(p.T_tab + pobj * D * D);
        __syncthreads();
        for (int e = c; e < D * D / 4; e += D) reinterpret_cast<float4*>(Ts)[e] = Tg[e];
        __syncthreads();
        const int ex = p.T_exp_tab ? p.T_exp_tab[pobj] : 0;
        const float* Sp = p.S_tab + pobj * D * D;
        for (int i = 0; i < D; ++i) {
            const float* Ti = Ts + i * D;
            float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
            for (int m = 0; m < D; m += 4) {
                a0 = fmaf(Ti[m], col[m], a0);
                a1 = fmaf(Ti[m + 1], col[m + 1], a1);
                a2 = fmaf(Ti[m + 2], col[m + 2], a2);
                a3 = fmaf(Ti[m + 3], col[m + 3], a3);
            }
            Sn[i * D + c] = ldexpf((a0 + a1) + (a2 + a3), ex) + Sp[i * D + c];
        }
#pragma unroll
        for (int i = 0; i < D; ++i) col[i] = Sn[i * D + c];
    }
    float* out = p.S_out + obj * D * D;
#pragma unroll
    for (int i = 0; i < D; ++i) out[i * D + c] = col[i];
}

// RetNet (scalar T), GLA (row scaling by a dk-vector), vanilla (addition).
template <int DK, int DV>
__global__ void __launch_bounds__(DV) compose_decay_simt_kernel(ComposeParams p, unsigned* err) {
    const int LH = p.n_layers * p.n_heads;
    const int chain = blockIdx.x / LH, lh = blockIdx.x % LH;
    const int c = threadIdx.x;
    const int64_t obj = (int64_t)chain * LH + lh;
    float col[DK];
#pragma unroll
    for (int i = 0; i < DK; ++i) col[i] = p.S0 ? p.S0[(obj * DK + i) * DV + c] : 0.f;
    const int j0 = p.cu_chain[chain], j1 = p.cu_chain[chain + 1];
    for (int j = j0; j < j1; ++j) {
        const int pi = p.seg_idx[j];
        if (pi < 0 || pi >= p.n_pairs) {
            set_error(err, kErrBadIndex);
            break;
        }
        const int64_t pobj = (int64_t)pi * LH + lh;
        const float* Sp = p.S_tab + pobj * DK * DV;
        if (p.family == kRETNET || p.family == kMAMBA2) {
            const float t = p.T_tab[pobj];
#pragma unroll
            for (int i = 0; i < DK; ++i) col[i] = fmaf(t, col[i], Sp[i * DV + c]);
        } else if (p.family == kGLA) {
            const float* tv = p.T_tab + pobj * DK;
#pragma unroll
            for (int i = 0; i < DK; ++i) col[i] = fmaf(tv[i], col[i], Sp[i * DV + c]);
        } else {
#pragma unroll
            for (int i = 0; i < DK; ++i) col[i] += Sp[i * DV + c];
        }
    }
    float* out = p.S_out + obj * DK * DV;
#pragma unroll
    for (int i = 0; i < DK; ++i) out[i * DV + c] = col[i];
}

template <int DK, int DV>
static cudaError_t launch_compose_dims(const ComposeParams& p, unsigned* err, cudaStream_t s) {
    const int64_t grid = (int64_t)p.n_chains * p.n_layers * p.n_heads;
    if (grid == 0) return cudaSuccess;
    if (p.family == kGDN || p.family == kKDA) {
        if constexpr (DK == DV) {
            const size_t smem = sizeof(float) * 2 * DK * DK;
            auto kern = compose_gdn_simt_kernel<DK>;
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
            kern<<<(unsigned)grid, DK, smem, s>>>(p, err);
        } else {
            return cudaErrorInvalidValue;
        }
    } else {
        compose_decay_simt_kernel<DK, DV><<<(unsigned)grid, DV, 0, s>>>(p, err);
    }
    return cudaGetLastError();
}

template <int DK>
static cudaError_t launch_compose_dv(const ComposeParams& p, unsigned* err, cudaStream_t s) {
    switch (p.dv) {
        case 16: return launch_compose_dims<DK, 16>(p, err, s);
        case 32: return launch_compose_dims<DK, 32>(p, err, s);
        case 64: return launch_compose_dims<DK, 64>(p, err, s);
        case 128: return launch_compose_dims<DK, 128>(p, err, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_compose_simt(const ComposeParams& p, unsigned* err, cudaStream_t s) {
    switch (p.dk) {
        case 16: return launch_compose_dv<16>(p, err, s);
        case 32: return launch_compose_dv<32>(p, err, s);
        case 64: return launch_compose_dv<64>(p, err, s);
        case 128: return launch_compose_dv<128>(p, err, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace hypic
