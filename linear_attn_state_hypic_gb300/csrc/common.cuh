// common.cuh -- device helpers shared by the libhypic kernels.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace hypic {

enum : int { kGDN = 0, kRETNET = 1, kGLA = 2, kVANILLA = 3, kKDA = 4, kMAMBA2 = 5 };
enum : int { kF32 = 0, kBF16 = 1 };

// Max of v over the block (every thread takes part; `red` holds one float per
// warp).  Threads with nothing to contribute pass 0.
__device__ __forceinline__ float block_max(float v, float* red) {
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    const int w = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[w] = v;
    __syncthreads();
    float m = 0.f;
    for (int i = 0; i < nw; ++i) m = fmaxf(m, red[i]);
    return m;
}

// Codes written to the device error word (first writer wins).
enum : unsigned { kErrNone = 0, kErrTimeout = 1, kErrBadIndex = 2 };

__device__ __forceinline__ void set_error(unsigned* err, unsigned code) {
    if (err) atomicCAS(err, 0u, code);
}

// Element `i` of a k/v/q array of dtype `dt` (f32 or bf16), widened to f32.
__device__ __forceinline__ float load_in(const void* p, int dt, int64_t i) {
    if (dt == kBF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[i]);
    return reinterpret_cast<const float*>(p)[i];
}

// Row offset of (layer, token, head) in a [n_layers][n_tokens][n_heads] array.
__device__ __forceinline__ int64_t tok_row(int layer, int64_t tok, int head, int64_t n_tokens, int H) {
    return ((int64_t)layer * n_tokens + tok) * H + head;
}

// Stage rows [t0, t0 + n) of one (layer, head) of a [L][N][H][D] array into
// shared memory as f32, dst[t][0..D).  All threads of the block take part.
// A thread issues kBatch loads before it stores any of them: a store could
// alias a later load for the compiler, which would otherwise wait for each
// load in turn.
template <int D>
__device__ __forceinline__ void stage_rows(float* dst, const void* src, int dt, int layer, int64_t t0, int n,
                                           int head, int64_t n_tokens, int H) {
    constexpr int kBatch = 8;
    const int total = n * D, step = blockDim.x;
    for (int e0 = threadIdx.x; e0 < total; e0 += kBatch * step) {
        float x[kBatch];
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            const int e = e0 + b * step;
            x[b] = e < total ? load_in(src, dt, tok_row(layer, t0 + e / D, head, n_tokens, H) * D + e % D) : 0.f;
        }
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            const int e = e0 + b * step;
            if (e < total) dst[e] = x[b];
        }
    }
}

// Stage a per-token gate [L][N][H] for rows [t0, t0 + n).
__device__ __forceinline__ void stage_gate(float* dst, const float* src, int layer, int64_t t0, int n, int head,
                                           int64_t n_tokens, int H, float fill) {
    for (int t = threadIdx.x; t < n; t += blockDim.x)
        dst[t] = src ? src[tok_row(layer, t0 + t, head, n_tokens, H)] : fill;
}

}  // namespace hypic
