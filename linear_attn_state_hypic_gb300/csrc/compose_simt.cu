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

// GDN, KDA: dense T_p (dk x dk, stored as mantissa * 2^exp).  The new column
// is written to the thread's own column of a shared buffer and read back,
// which keeps only one column in registers.  With T_out, threads D..2D-1 also
// carry the chain's own transition T_chain <- T_p T_chain (from I), one column
// each, renormalised by a power of two after every step (its exponent
// accumulated like the build's).
template <int D>
__global__ void __launch_bounds__(2 * D) compose_gdn_simt_kernel(ComposeParams p, unsigned* err) {
    extern __shared__ float sm[];
    float* Ts = sm;          // [D][D]
    float* Sn = Ts + D * D;  // [D][D], column c private to thread c
    float* Tn = Sn + D * D;  // [D][D] (T_chain, with T_out)
    float* red = Tn + (p.T_out ? D * D : 0);  // [8]
    const bool want_T = p.T_out != nullptr;
    const int LH = p.n_layers * p.n_heads;
    const int chain = blockIdx.x / LH, lh = blockIdx.x % LH;
    const bool isT = threadIdx.x >= D;
    const int c = isT ? threadIdx.x - D : threadIdx.x;
    const int64_t obj = (int64_t)chain * LH + lh;
    float col[D];
#pragma unroll
    for (int i = 0; i < D; ++i) col[i] = isT ? (i == c ? 1.f : 0.f) : p.S0 ? p.S0[(obj * D + i) * D + c] : 0.f;
    int texp = 0;
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
        for (int e = threadIdx.x; e < D * D / 4; e += blockDim.x) reinterpret_cast<float4*>(Ts)[e] = Tg[e];
        __syncthreads();
        const int ex = p.T_exp_tab ? p.T_exp_tab[pobj] : 0;
        const float* Sp = p.S_tab + pobj * D * D;
        constexpr int kRows = D < 16 ? D : 16;  // rows a batch: their S_p values loaded before any store
#pragma unroll 1
        for (int i0 = 0; i0 < D; i0 += kRows) {
            float spv[kRows];
#pragma unroll
            for (int r = 0; r < kRows; ++r) spv[r] = isT ? 0.f : Sp[(i0 + r) * D + c];
#pragma unroll
            for (int r = 0; r < kRows; ++r) {
                const int i = i0 + r;
                const float4* Ti = reinterpret_cast<const float4*>(Ts + i * D);
                float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
                for (int m = 0; m < D / 4; ++m) {
                    const float4 t4 = Ti[m];
                    a0 = fmaf(t4.x, col[4 * m], a0);
                    a1 = fmaf(t4.y, col[4 * m + 1], a1);
                    a2 = fmaf(t4.z, col[4 * m + 2], a2);
                    a3 = fmaf(t4.w, col[4 * m + 3], a3);
                }
                const float acc = (a0 + a1) + (a2 + a3);
                if (isT)
                    Tn[i * D + c] = acc;
                else
                    Sn[i * D + c] = ldexpf(acc, ex) + spv[r];
            }
        }
#pragma unroll
        for (int i = 0; i < D; ++i) col[i] = (isT ? Tn : Sn)[i * D + c];
        if (want_T) {
            float m = 0.f;
            if (isT)
#pragma unroll
                for (int i = 0; i < D; ++i) m = fmaxf(m, fabsf(col[i]));
            m = block_max(m, red);
            int e = (m > 0.f && isfinite(m)) ? ilogbf(m) : 0;
            if (isT && e != 0)
#pragma unroll
                for (int i = 0; i < D; ++i) col[i] = ldexpf(col[i], -e);
            texp += ex + e;
        }
    }
    if (isT) {
        float* To = p.T_out + obj * D * D;
#pragma unroll
        for (int i = 0; i < D; ++i) To[i * D + c] = col[i];
        if (c == 0) p.T_exp_out[obj] = texp;
    } else {
        float* out = p.S_out + obj * D * D;
#pragma unroll
        for (int i = 0; i < D; ++i) out[i * D + c] = col[i];
    }
}

// RetNet, Mamba2 (scalar T), GLA (row scaling by a dk-vector), vanilla
// (addition).  Thread c < DV owns column c of S; with T_out, the chain's own
// transition is the product of the T_p in double (thread 0 for a scalar,
// thread i < DK for entry i of GLA's vector).
template <int DK, int DV>
__global__ void __launch_bounds__(DK > DV ? DK : DV) compose_decay_simt_kernel(ComposeParams p, unsigned* err) {
    const int LH = p.n_layers * p.n_heads;
    const int chain = blockIdx.x / LH, lh = blockIdx.x % LH;
    const int c = threadIdx.x;
    const bool scol = c < DV;
    const bool scalar = p.family == kRETNET || p.family == kMAMBA2;
    const bool tcol = p.T_out && (scalar ? c == 0 : (p.family == kGLA && c < DK));
    const int64_t obj = (int64_t)chain * LH + lh;
    float col[DK];
#pragma unroll
    for (int i = 0; i < DK; ++i) col[i] = (p.S0 && scol) ? p.S0[(obj * DK + i) * DV + c] : 0.f;
    double tprod = 1.0;
    const int j0 = p.cu_chain[chain], j1 = p.cu_chain[chain + 1];
    for (int j = j0; j < j1; ++j) {
        const int pi = p.seg_idx[j];
        if (pi < 0 || pi >= p.n_pairs) {
            set_error(err, kErrBadIndex);
            break;
        }
        const int64_t pobj = (int64_t)pi * LH + lh;
        const float* Sp = p.S_tab + pobj * DK * DV;
        if (tcol) tprod *= (double)(scalar ? p.T_tab[pobj] : p.T_tab[pobj * DK + c]);
        if (!scol) continue;
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
    if (tcol) p.T_out[scalar ? obj : obj * DK + c] = (float)tprod;
    if (!scol) return;
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
            const size_t smem = sizeof(float) * ((p.T_out ? 3 : 2) * DK * DK + 8);
            auto kern = compose_gdn_simt_kernel<DK>;
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
            kern<<<(unsigned)grid, p.T_out ? 2 * DK : DK, smem, s>>>(p, err);
        } else {
            return cudaErrorInvalidValue;
        }
    } else {
        compose_decay_simt_kernel<DK, DV><<<(unsigned)grid, DK > DV ? DK : DV, 0, s>>>(p, err);
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
