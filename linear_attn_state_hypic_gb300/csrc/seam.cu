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
// So the CTAs are persistent (one per SM) and take (seam, layer, head) items
// in turn; while one item computes, the next item's state comes into shared
// memory by a bulk copy and its first kPre tokens by asynchronous copies.
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace hypic {

using tc::bulk_load_1d;
using tc::cp_async16;
using tc::cp_async4;
using tc::cp_async_commit;
using tc::cp_async_wait_all;

static constexpr int kPre = 8;  // tokens of an item copied ahead; a longer window stages the rest in turn

// Shared-memory layout of the seam kernel, sized for the input dtype and the
// family (the per-channel gates g of GLA and KDA): the next item's state, two
// buffers of raw token bytes (q, k, g rows of DK, v rows of DV, then a and b),
// the current item's tokens as f32, and the state's barrier.
struct SeamLayout {
    uint32_t row_k, row_v, row_g;  // raw bytes of a q/k, v, g row
    uint32_t raw, off_raw, off_tok, off_bar, bytes;
    __host__ __device__ SeamLayout(int dk, int dv, int in_dtype, int family) {
        const uint32_t es = in_dtype == kBF16 ? 2u : 4u;
        const bool gated = family == kGLA || family == kKDA;
        row_k = dk * es;
        row_v = dv * es;
        row_g = gated ? dk * 4u : 0u;
        raw = ((kPre * (2 * row_k + row_v + row_g) + 2 * kPre * 4u) + 15u) / 16u * 16u;
        off_raw = (uint32_t)dk * dv * 4u;
        off_tok = off_raw + 2 * raw;
        off_bar = off_tok + kPre * (2u * dk + (gated ? dk : 0u) + dv) * 4u + 2u * kPre * 4u;
        off_bar = (off_bar + 15u) / 16u * 16u;
        bytes = off_bar + 16u;
    }
};

// Start the copies of item `item` (state, if any, and its first tokens) into the state buffer and
// raw buffer `raw`.  All threads take part.
template <int DK, int DV>
__device__ __forceinline__ void seam_prefetch(const SeamParams& p, const SeamLayout& Ly, int64_t item, uint8_t* sm,
                                              uint8_t* raw, uint64_t* bar) {
    const int LH = p.n_layers * p.n_heads;
    const int r = (int)(item / LH), lh = (int)(item % LH);
    const int layer = lh / p.n_heads, head = lh % p.n_heads;
    if (p.state_in && threadIdx.x == 0) {
        tc::fence_async_smem();  // (the state buffer's previous contents have been read by every thread)
        tc::mbar_expect_tx(bar, DK * DV * 4);
        bulk_load_1d(sm, p.state_in + item * DK * DV, DK * DV * 4, bar);
    }
    const int64_t tb = p.cu_seam[r], te = p.cu_seam[r + 1];
    const int n = (int)(te - tb < kPre ? te - tb : kPre);
    const int es = p.in_dtype == kBF16 ? 2 : 4;
    const int cq = DK * es / 16, cv = DV * es / 16;  // 16-byte chunks of a q/k row and of a v row
    const bool gated = p.family == kGLA || p.family == kKDA;
    const int cg = DK * 4 / 16;
    const int per = 2 * cq + cv + (gated ? cg : 0);  // chunks of one token
    for (int e = threadIdx.x; e < n * per; e += blockDim.x) {
        const int t = e / per;
        int c = e % per;
        const int64_t row = tok_row(layer, tb + t, head, p.n_tokens, p.n_heads);
        const uint8_t* src;
        uint8_t* dst;
        if (c < cq) {
            src = static_cast<const uint8_t*>(p.q) + row * DK * es + c * 16;
            dst = raw + t * Ly.row_k + c * 16;
        } else if ((c -= cq) < cq) {
            src = static_cast<const uint8_t*>(p.k) + row * DK * es + c * 16;
            dst = raw + kPre * Ly.row_k + t * Ly.row_k + c * 16;
        } else if ((c -= cq) < cv) {
            src = static_cast<const uint8_t*>(p.v) + row * DV * es + c * 16;
            dst = raw + 2 * kPre * Ly.row_k + t * Ly.row_v + c * 16;
        } else {
            c -= cv;
            src = reinterpret_cast<const uint8_t*>(p.g) + row * DK * 4 + c * 16;
            dst = raw + kPre * (2 * Ly.row_k + Ly.row_v) + t * Ly.row_g + c * 16;
        }
        cp_async16(dst, src);
    }
    float* ab = reinterpret_cast<float*>(raw + kPre * (2 * Ly.row_k + Ly.row_v + Ly.row_g));
    const int t = threadIdx.x;
    if (t < n) {
        const int64_t row = tok_row(layer, tb + t, head, p.n_tokens, p.n_heads);
        if (p.alpha) cp_async4(ab + t, p.alpha + row);
        if (p.beta) cp_async4(ab + kPre + t, p.beta + row);
    }
    cp_async_commit();
}

template <int DK, int DV>
__global__ void __launch_bounds__(DV) seam_stream_kernel(SeamParams p, int64_t n_items, uint32_t wait_limit,
                                                         unsigned* err) {
    const int fam = p.family;
    const bool gated = fam == kGLA || fam == kKDA;
    const SeamLayout Ly(DK, DV, p.in_dtype, fam);
    extern __shared__ __align__(128) uint8_t sm[];
    const float* sst = reinterpret_cast<const float*>(sm);   // [DK][DV]: the state of the current item
    float* qs = reinterpret_cast<float*>(sm + Ly.off_tok);  // [kPre][DK]
    float* ks = qs + kPre * DK;                               // [kPre][DK]
    float* vs = ks + kPre * DK;                               // [kPre][DV]
    float* as = vs + kPre * DV;                               // [kPre]
    float* bs = as + kPre;                                    // [kPre]
    float* gs = bs + kPre;                                    // [kPre][DK] (GLA, KDA)
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + Ly.off_bar);
    const int c = threadIdx.x;
    const int LH = p.n_layers * p.n_heads;
    if (c == 0) {
        tc::mbar_init(bar, 1);
        tc::fence_mbar_init();
    }
    __syncthreads();
    int64_t item = blockIdx.x;
    if (item < n_items) seam_prefetch<DK, DV>(p, Ly, item, sm, sm + Ly.off_raw, bar);
    bool ok = true;
    for (uint32_t j = 0; item < n_items; item += gridDim.x, ++j) {
        const int r = (int)(item / LH), lh = (int)(item % LH);
        const int layer = lh / p.n_heads, head = lh % p.n_heads;
        const int64_t tb = p.cu_seam[r], te = p.cu_seam[r + 1];
        const int n0 = (int)(te - tb < kPre ? te - tb : kPre);
        // this item's copies have landed (the bounded wait gives up once: the error word is set and the
        // remaining items are skipped)
        cp_async_wait_all();
        if (p.state_in) {
            uint32_t i = 0;
            while (ok && !tc::mbar_try_wait(bar, j & 1)) {
                if (++i >= wait_limit) {
                    ok = false;
                    set_error(err, kErrTimeout);
                }
            }
        }
        if (!__syncthreads_and(ok)) break;
        // its tokens as f32, and its state column
        {
            const uint8_t* raw = sm + Ly.off_raw + (j & 1) * Ly.raw;
            const bool bf = p.in_dtype == kBF16;
            for (int e = c; e < n0 * DK; e += blockDim.x) {
                const int t = e / DK, i = e % DK;
                const uint8_t* qr = raw + t * Ly.row_k;
                const uint8_t* kr = raw + kPre * Ly.row_k + t * Ly.row_k;
                qs[e] = bf ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(qr)[i])
                           : reinterpret_cast<const float*>(qr)[i];
                ks[e] = bf ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(kr)[i])
                           : reinterpret_cast<const float*>(kr)[i];
                if (gated)
                    gs[e] = reinterpret_cast<const float*>(raw + kPre * (2 * Ly.row_k + Ly.row_v) + t * Ly.row_g)[i];
            }
            for (int e = c; e < n0 * DV; e += blockDim.x) {
                const int t = e / DV, i = e % DV;
                const uint8_t* vr = raw + 2 * kPre * Ly.row_k + t * Ly.row_v;
                vs[e] = bf ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(vr)[i])
                           : reinterpret_cast<const float*>(vr)[i];
            }
            const float* ab = reinterpret_cast<const float*>(raw + kPre * (2 * Ly.row_k + Ly.row_v + Ly.row_g));
            if (c < n0) {
                as[c] = p.alpha ? ab[c] : 1.f;
                bs[c] = p.beta ? ab[kPre + c] : 1.f;
            }
        }
        float col[DK];
#pragma unroll
        for (int i = 0; i < DK; ++i) col[i] = p.state_in ? sst[i * DV + c] : 0.f;
        __syncthreads();  // (the state buffer and this item's raw tokens have been read)
        const int64_t nxt = item + gridDim.x;
        if (nxt < n_items) seam_prefetch<DK, DV>(p, Ly, nxt, sm, sm + Ly.off_raw + ((j + 1) & 1) * Ly.raw, bar);
        const float gm = (fam == kRETNET && p.gamma) ? p.gamma[(int64_t)layer * p.n_heads + head] : 1.f;
        for (int64_t t0 = tb; t0 < te; t0 += kPre) {
            const int n = (int)(te - t0 < kPre ? te - t0 : kPre);
            if (t0 != tb) {  // a window longer than kPre: its later tokens, staged in turn
                __syncthreads();
                stage_rows<DK>(qs, p.q, p.in_dtype, layer, t0, n, head, p.n_tokens, p.n_heads);
                stage_rows<DK>(ks, p.k, p.in_dtype, layer, t0, n, head, p.n_tokens, p.n_heads);
                stage_rows<DV>(vs, p.v, p.in_dtype, layer, t0, n, head, p.n_tokens, p.n_heads);
                if (gated) stage_rows<DK>(gs, p.g, kF32, layer, t0, n, head, p.n_tokens, p.n_heads);
                stage_gate(as, p.alpha, layer, t0, n, head, p.n_tokens, p.n_heads, 1.f);
                stage_gate(bs, p.beta, layer, t0, n, head, p.n_tokens, p.n_heads, 1.f);
                __syncthreads();
            }
            for (int t = 0; t < n; ++t) {
                const float4* kt = reinterpret_cast<const float4*>(ks + t * DK);
                const float4* qt = reinterpret_cast<const float4*>(qs + t * DK);
                const float4* gt = reinterpret_cast<const float4*>(gs + t * DK);
                const float vj = vs[t * DV + c];
                if (fam == kGDN || fam == kKDA) {  // KDA: the per-channel gate first, then a = 1
                    if (fam == kKDA) {
#pragma unroll
                        for (int i = 0; i < DK / 4; ++i) {
                            const float4 g4 = gt[i];
                            col[4 * i] *= g4.x, col[4 * i + 1] *= g4.y, col[4 * i + 2] *= g4.z, col[4 * i + 3] *= g4.w;
                        }
                    }
                    float u0 = 0.f, u1 = 0.f, u2 = 0.f, u3 = 0.f;
#pragma unroll
                    for (int i = 0; i < DK / 4; ++i) {
                        const float4 k4 = kt[i];
                        u0 = fmaf(k4.x, col[4 * i], u0);
                        u1 = fmaf(k4.y, col[4 * i + 1], u1);
                        u2 = fmaf(k4.z, col[4 * i + 2], u2);
                        u3 = fmaf(k4.w, col[4 * i + 3], u3);
                    }
                    const float a = fam == kKDA ? 1.f : as[t], b = bs[t];
                    const float w = b * (vj - a * ((u0 + u1) + (u2 + u3)));
#pragma unroll
                    for (int i = 0; i < DK / 4; ++i) {
                        const float4 k4 = kt[i];
                        col[4 * i] = fmaf(k4.x, w, a * col[4 * i]);
                        col[4 * i + 1] = fmaf(k4.y, w, a * col[4 * i + 1]);
                        col[4 * i + 2] = fmaf(k4.z, w, a * col[4 * i + 2]);
                        col[4 * i + 3] = fmaf(k4.w, w, a * col[4 * i + 3]);
                    }
                } else if (fam == kGLA) {
#pragma unroll
                    for (int i = 0; i < DK / 4; ++i) {
                        const float4 k4 = kt[i], g4 = gt[i];
                        col[4 * i] = fmaf(k4.x, vj, g4.x * col[4 * i]);
                        col[4 * i + 1] = fmaf(k4.y, vj, g4.y * col[4 * i + 1]);
                        col[4 * i + 2] = fmaf(k4.z, vj, g4.z * col[4 * i + 2]);
                        col[4 * i + 3] = fmaf(k4.w, vj, g4.w * col[4 * i + 3]);
                    }
                } else {  // RetNet (gamma), Mamba2 (a_t), vanilla (1)
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
                float o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f;
#pragma unroll
                for (int i = 0; i < DK / 4; ++i) {
                    const float4 q4 = qt[i];
                    o0 = fmaf(q4.x, col[4 * i], o0);
                    o1 = fmaf(q4.y, col[4 * i + 1], o1);
                    o2 = fmaf(q4.z, col[4 * i + 2], o2);
                    o3 = fmaf(q4.w, col[4 * i + 3], o3);
                }
                p.o_out[tok_row(layer, t0 + t, head, p.n_tokens, p.n_heads) * DV + c] = (o0 + o1) + (o2 + o3);
            }
        }
        float* so = p.state_out + item * DK * DV + c;
#pragma unroll
        for (int i = 0; i < DK; ++i) so[i * DV] = col[i];
    }
    cp_async_wait_all();  // (no copy into this CTA's shared memory is left in flight; no bulk copy
                          // follows the last item)
}

template <int DK, int DV>
static cudaError_t launch_seam_dims(const SeamParams& p, unsigned* err, cudaStream_t s) {
    const SeamLayout Ly(DK, DV, p.in_dtype, p.family);
    const int64_t items = (int64_t)p.n_seams * p.n_layers * p.n_heads;
    if (items == 0) return cudaSuccess;
    auto kern = seam_stream_kernel<DK, DV>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Ly.bytes);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    int per_sm = 0;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, DV, Ly.bytes)) != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    const int64_t grid = items < (int64_t)sms * per_sm ? items : (int64_t)sms * per_sm;
    kern<<<(unsigned)grid, DV, Ly.bytes, s>>>(p, items, 1u << 26, err);
    return cudaGetLastError();
}

template <int DK>
static cudaError_t launch_seam_dv(const SeamParams& p, unsigned* err, cudaStream_t s) {
    switch (p.dv) {
        case 16: return launch_seam_dims<DK, 16>(p, err, s);
        case 32: return launch_seam_dims<DK, 32>(p, err, s);
        case 64: return launch_seam_dims<DK, 64>(p, err, s);
        case 128: return launch_seam_dims<DK, 128>(p, err, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_seam(const SeamParams& p, unsigned* err, cudaStream_t s) {
    switch (p.dk) {
        case 16: return launch_seam_dv<16>(p, err, s);
        case 32: return launch_seam_dv<32>(p, err, s);
        case 64: return launch_seam_dv<64>(p, err, s);
        case 128: return launch_seam_dv<128>(p, err, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace hypic
