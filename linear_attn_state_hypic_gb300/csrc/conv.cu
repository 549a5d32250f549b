// conv.cu -- conv-state warm-up at seam windows.
//
// Variants with a short causal convolution on the linear layers' inputs need
// the K-1 inputs before a seam window from the new prefix, not from the
// cached segment's own past (aibase article on HYPIC, paragraph on the linear
// layers: the "conv-state warm-up" patch).  A depthwise causal convolution of
// width K gives token t of channel c
//     y_t = act(bias_c + sum_{j<K} w[c][j] x_{t-K+1+j}),
// where the inputs before the window are taken from `hist` (zeros when NULL).
// One thread per (layer, token, channel); the window start of a token is
// found by a binary search of cu_seam.  Memory-bound: K reads (cached) and one
// write per output.
#include <cuda_runtime.h>
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace hypic {

__global__ void conv_warmup_kernel(ConvParams p) {
    const int64_t total = (int64_t)p.n_layers * p.n_tokens * p.C;
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < total; e += (int64_t)gridDim.x * blockDim.x) {
        const int c = (int)(e % p.C);
        const int64_t lt = e / p.C;
        const int64_t t = lt % p.n_tokens;
        const int l = (int)(lt / p.n_tokens);
        int lo = 0, hi = p.n_seams;  // window r with cu[r] <= t < cu[r+1]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (p.cu_seam[mid] <= t) lo = mid; else hi = mid;
        }
        const int64_t s0 = p.cu_seam[lo];
        float acc = p.bias ? p.bias[(int64_t)l * p.C + c] : 0.f;
        const float* wc = p.w + ((int64_t)l * p.C + c) * p.K;
        for (int j = 0; j < p.K; ++j) {
            const int64_t src = t - (p.K - 1) + j;
            float xv = 0.f;
            if (src >= s0)
                xv = p.x[((int64_t)l * p.n_tokens + src) * p.C + c];
            else if (p.hist)
                xv = p.hist[(((int64_t)lo * p.n_layers + l) * (p.K - 1) + (p.K - 1) - (s0 - src)) * p.C + c];
            acc = fmaf(wc[j], xv, acc);
        }
        p.y[e] = p.act ? acc / (1.f + expf(-acc)) : acc;
    }
}

cudaError_t launch_conv_warmup(const ConvParams& p, cudaStream_t s) {
    const int64_t total = (int64_t)p.n_layers * p.n_tokens * p.C;
    if (total == 0) return cudaSuccess;
    const int64_t blocks = (total + 255) / 256;
    conv_warmup_kernel<<<(unsigned)(blocks < 4096 ? blocks : 4096), 256, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace hypic
