// rope.cu -- state re-rotation of cached pairs for RoPE variants.
//
// The aibase article on HYPIC (paragraph on the linear layers) names a "state
// re-rotation" patch for variants whose keys carry rotary position
// embeddings.  A segment moved by delta positions sees each key as R k, with
// R = R(delta) the rotary rotation; for a family whose per-token transition is
// built from k k^T and scalars (GDN, RetNet, Mamba2, vanilla) every transition
// A becomes R A R^T and every write k v^T becomes R k v^T, so the cached pair
// becomes (R T R^T, R S).  R turns the first rotary_dim features in
// rotate-half pairs: for i < h = rotary_dim / 2, (x_i, x_{i+h}) by the angle
// delta * base^(-2i / rotary_dim).  T's power-of-two exponent is unchanged
// (R is orthogonal).
//
// One CTA per (pair, layer, head); the angles are formed in double (shifts
// reach millions of positions), the rotation itself in float.  Memory-bound:
// one read and one write of the pair.
#include <cuda_runtime.h>
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace hypic {

__global__ void __launch_bounds__(128) rope_kernel(RopeParams p) {
    extern __shared__ float sm[];
    float* cs = sm;        // [64]
    float* sn = cs + 64;   // [64]
    float* Ts = sn + 64;   // [dk][dk + 1] (dense T)
    const int dk = p.dk, dv = p.dv, h = p.rotary_dim / 2, ld = dk + 1;
    const int LH = p.n_layers * p.n_heads;
    const int pair = blockIdx.x / LH;
    const int64_t obj = blockIdx.x;  // (pair, layer, head) in table order
    const int tid = threadIdx.x;
    if (tid < h) {
        const double a = (double)p.delta[pair] * exp(-2.0 * tid / p.rotary_dim * log(p.base));
        cs[tid] = (float)cos(a);
        sn[tid] = (float)sin(a);
    }
    __syncthreads();
    // (loads are issued kB at a time before their stores: a store could alias a later load for
    // the compiler, which would otherwise wait for each load in turn)
    constexpr int kB = 8;
    if (tid < dv) {  // S <- R S: thread j rotates column j
        float* S = p.S + obj * dk * dv;
        for (int i0 = 0; i0 < h; i0 += kB) {
            float x1[kB], x2[kB];
#pragma unroll
            for (int b = 0; b < kB; ++b)
                if (i0 + b < h) {
                    x1[b] = S[(int64_t)(i0 + b) * dv + tid];
                    x2[b] = S[(int64_t)(i0 + b + h) * dv + tid];
                }
#pragma unroll
            for (int b = 0; b < kB; ++b)
                if (i0 + b < h) {
                    const int i = i0 + b;
                    S[(int64_t)i * dv + tid] = x1[b] * cs[i] - x2[b] * sn[i];
                    S[(int64_t)(i + h) * dv + tid] = x2[b] * cs[i] + x1[b] * sn[i];
                }
        }
    }
    if (!p.T) return;
    float* T = p.T + obj * dk * dk;
    for (int e0 = tid; e0 < dk * dk; e0 += kB * blockDim.x) {
        float x[kB];
#pragma unroll
        for (int b = 0; b < kB; ++b) {
            const int e = e0 + b * blockDim.x;
            if (e < dk * dk) x[b] = T[e];
        }
#pragma unroll
        for (int b = 0; b < kB; ++b) {
            const int e = e0 + b * blockDim.x;
            if (e < dk * dk) Ts[(e / dk) * ld + e % dk] = x[b];
        }
    }
    __syncthreads();
    if (tid < dk)  // rows: R T (thread j, column j)
        for (int i = 0; i < h; ++i) {
            const float x1 = Ts[i * ld + tid], x2 = Ts[(i + h) * ld + tid];
            Ts[i * ld + tid] = x1 * cs[i] - x2 * sn[i];
            Ts[(i + h) * ld + tid] = x2 * cs[i] + x1 * sn[i];
        }
    __syncthreads();
    if (tid < dk)  // columns: (R T) R^T (thread i, row i)
        for (int j = 0; j < h; ++j) {
            const float x1 = Ts[tid * ld + j], x2 = Ts[tid * ld + j + h];
            Ts[tid * ld + j] = x1 * cs[j] - x2 * sn[j];
            Ts[tid * ld + j + h] = x2 * cs[j] + x1 * sn[j];
        }
    __syncthreads();
    for (int e = tid; e < dk * dk; e += blockDim.x) T[e] = Ts[(e / dk) * ld + e % dk];
}

cudaError_t launch_rope(const RopeParams& p, cudaStream_t s) {
    const int64_t grid = (int64_t)p.n_pairs * p.n_layers * p.n_heads;
    if (grid == 0) return cudaSuccess;
    const size_t smem = sizeof(float) * (128 + (p.T ? (size_t)p.dk * (p.dk + 1) : 0));
    cudaError_t e = cudaFuncSetAttribute(rope_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    rope_kernel<<<(unsigned)grid, 128, smem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace hypic
