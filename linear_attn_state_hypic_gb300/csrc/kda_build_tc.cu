// kda_build_tc.cu -- the KDA cached pair (T_C, S(C|0)) at d = 128 with bf16
// keys and values: every 64-token chunk's own pair on the sm_103a tensor
// cores, the chunk pairs of a segment then chained by the tensor-core compose.
//
// What it computes: for a segment C and a head, T_C = A_L ... A_1 with the
// Kimi delta attention transition A_t = (I - b_t k_t k_t^T) Diag(a_t) (a_t the
// per-channel gate) and S(C|0), the state after C from zero with the write
// term b_t k_t v_t^T (aibase article on HYPIC, paragraph on the linear layers:
// the cached pair of a segment, and its composition law
// S(C1.C2) = T(C2) S(C1) + S(C2)).
//
// How.  The body of a segment is cut into chunks of 64 tokens.  A chunk's own
// pair depends on nothing outside the chunk, so all chunks of all segments,
// layers and heads are formed at once (one CTA each), into a table in the
// workspace; the composition law then chains each segment's chunk pairs in
// order (the compose's state mode gives S(C|0) from a zero state, its
// transition mode T_C), which is exact up to rounding.
// Chunk pair.  Inside a chunk let g_t = a_1 ... a_t (per channel, g_0 = 1) and
// g_C its last value.  The rescaled state Diag(g_t)^-1 S_t takes one
// generalised Householder step per token, I - b_t x_t y_t^T with x_t = k_t / g_t
// and y_t = k_t * g_t, so the chunk's product is I - X^T W (WY form) with
//     w_t = b_t (y_t - sum_{s<t} G_ts w_s),  u_t = b_t (v_t - sum_{s<t} G_ts u_s),
//     G_ts = y_t . x_s = sum_c k_t[c] k_s[c] (a_{s+1} ... a_t)[c],
// and, with kbar_t = k_t * (a_{t+1} ... a_L) (= k_t g_C / g_t),
//     T_chunk = Diag(g_C) - Kbar^T W,   S_chunk = Kbar^T U.
// Every factor is a product of gates over a token range, formed as a running
// product (never a ratio of two prefix products, which leaves the fp32 range
// for strong gates), so the chunk pair is in range for any a_t in [0, 1].
// Steps (512 threads, one CTA per chunk, layer and head):
//   stage    keys (fp32), values (bf16), gates, b
//   kbar     reverse running products, written as the bf16 hi + lo operand Kbar^T
//   gram     G_ts for s < t: thread (s, channel group) carries k_s times the gates
//            after s and meets every later key (fp32, CUDA cores)
//   solve    [-W | U] by forward substitution, one column per thread (fp32)
//   MMA      D = Kbar^T [-W | U]: bf16 M = 128, N = 256, K = 64, hi + lo pairs
//            (three products, about 16 significant bits each side), fp32 in tensor memory
//   write    T_chunk = Diag(g_C) + D_left, normalised by a power of two (its exponent
//            kept beside it), and S_chunk = D_right
// The chunk tables cost 128 KB per chunk, layer and head; segments are taken
// in batches whose tables fit the workspace.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stddef.h>
#include <stdint.h>

#include <vector>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace hypic {
namespace {

using namespace tc;

constexpr int kD = 128, kC = 64;
constexpr int kThreads = 512;
constexpr int64_t kPairBytes = 2 * kD * kD * 4;  // T and S of one chunk, layer and head

// Shared memory map (bytes).  The MMA operands are K-major without swizzle:
// core matrices of 8 rows x 8 tokens (16 bytes a row), the 8 of a row group
// adjacent along the tokens (128 bytes apart), row groups 1024 bytes apart.
constexpr uint32_t OFF_KF = 0;               // keys, fp32 [64 t][128 c]
constexpr uint32_t OFF_GA = OFF_KF + 32768;  // gates a, fp32 [64 t][128 c]
constexpr uint32_t OFF_VB = OFF_GA + 32768;  // values, bf16 [64 t][128 c]
constexpr uint32_t OFF_L = OFF_VB + 16384;   // b_t G_ts for s < t, 0 elsewhere: fp32 [64 t][64 s]
constexpr uint32_t OFF_A = OFF_L + 16384;    // Kbar^T hi, lo: bf16 [128 i][64 t], 16 KB each
constexpr uint32_t OFF_B = OFF_A + 32768;    // [-W | U]^T hi, lo: bf16 [256 j][64 t], 32 KB each
constexpr uint32_t OFF_MISC = OFF_B + 65536;

struct KMisc {
    uint64_t mma_done;
    uint32_t tmem_base;
    int pad;
    float gC[kD];     // g_C per channel
    float beta[kC];   // b_t (0 past the body end)
    float red[4];     // max |T| of each T warp
};
constexpr uint32_t kSmemBytes = OFF_MISC + sizeof(KMisc);
static_assert(kSmemBytes <= 232448, "shared memory budget");

constexpr uint32_t kTmemCols = 256;
constexpr uint32_t ID_PAIR = idesc(1, 128, 256, false, false);  // D = Kbar^T [-W | U], both K-major

struct ChunkArgs {
    int n_layers, n_heads, seg0;
    int64_t n_tokens;
    const int32_t* cu;
    const int32_t* skip;
    const int32_t* cu_chunk;   // [batch segments + 1]: first chunk of each segment of the batch
    const int32_t* chunk_seg;  // [batch chunks]: the segment of each chunk
    const __nv_bfloat16* k;
    const __nv_bfloat16* v;
    const float* g;
    const float* beta;
    float* T_tab;       // [chunks][L][H][128][128] mantissa
    int32_t* T_exp_tab;  // [chunks][L][H]
    float* S_tab;       // [chunks][L][H][128][128]
    unsigned* err;
    uint64_t wait_ns;
};

// Byte offset of (row, token) in a K-major operand of 64 tokens.
__device__ __forceinline__ uint32_t core_off(int row, int t) {
    return (uint32_t)((row >> 3) * 1024 + (t >> 3) * 128 + (row & 7) * 16 + (t & 7) * 2);
}

// x = hi + lo as a pair of bf16 (hi rounded to nearest, lo the rounded rest).
__device__ __forceinline__ void split2(float x0, float x1, uint32_t& h, uint32_t& l) {
    const __nv_bfloat162 hh = __floats2bfloat162_rn(x0, x1);
    const float2 hf = __bfloat1622float2(hh);
    const __nv_bfloat162 ll = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
    h = *reinterpret_cast<const uint32_t*>(&hh);
    l = *reinterpret_cast<const uint32_t*>(&ll);
}

// Eight consecutive tokens of one operand row, as hi and lo 16-byte pieces.
__device__ __forceinline__ void store_row8(uint8_t* hi, uint8_t* lo, uint32_t off, const float (&x)[8]) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) split2(x[2 * e], x[2 * e + 1], h[e], l[e]);
    *reinterpret_cast<uint4*>(hi + off) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4*>(lo + off) = make_uint4(l[0], l[1], l[2], l[3]);
}

// x * 2^e for any int e with the result in range (two exact power-of-two factors).
__device__ __forceinline__ float scale_pow2(float x, int e) {
    const int e1 = e / 2, e2 = e - e1;
    return x * __int_as_float((e1 + 127) << 23) * __int_as_float((e2 + 127) << 23);
}

__device__ __noinline__ bool wait_done(uint64_t* bar, uint64_t wait_ns, unsigned* err) {
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
#pragma unroll 1
        for (int j = 0; j < 16; ++j)
            if (mbar_try_wait(bar, 0)) return true;
        if (globaltimer_ns() - t0 > wait_ns) break;
    }
    set_error(err, kErrTimeout);
    return false;
}

__global__ void __launch_bounds__(kThreads, 1) kda_chunk_pair_kernel(const ChunkArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    KMisc* ms = reinterpret_cast<KMisc*>(smem + OFF_MISC);
    float* KF = reinterpret_cast<float*>(smem + OFF_KF);
    float* GA = reinterpret_cast<float*>(smem + OFF_GA);
    const __nv_bfloat16* VB = reinterpret_cast<const __nv_bfloat16*>(smem + OFF_VB);
    float* L = reinterpret_cast<float*>(smem + OFF_L);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int LH = a.n_layers * a.n_heads;
    const int p = blockIdx.x / LH, lh = blockIdx.x % LH;
    const int layer = lh / a.n_heads, head = lh % a.n_heads;
    const int seg = a.chunk_seg[p];
    const int64_t b0 = (int64_t)a.cu[seg] + (a.skip ? a.skip[seg] : 0), b1 = a.cu[seg + 1];
    const int64_t t0 = b0 + (int64_t)(p - a.cu_chunk[seg - a.seg0]) * kC;
    const int n = (int)(b1 - t0 < kC ? b1 - t0 : kC);
    if (n <= 0) {  // the batch plan makes this unreachable
        if (tid == 0) set_error(a.err, kErrBadIndex);
        return;
    }
    if (tid == 0) {
        mbar_init(&ms->mma_done, 1);
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(&ms->tmem_base, kTmemCols);

    // ---- stage: every load of a thread issued before its stores
    {
        const int64_t rs = (int64_t)a.n_heads * kD;  // elements between consecutive tokens
        const int64_t row0 = tok_row(layer, t0, head, a.n_tokens, a.n_heads) * kD;
        uint4 xk[2], xv[2];
        float4 xg[4];
        float bt = 0.f;
#pragma unroll
        for (int m = 0; m < 2; ++m) {
            const int e = tid + kThreads * m, t = e >> 4, q = e & 15;
            const bool ok = t < n;
            xk[m] = ok ? *reinterpret_cast<const uint4*>(a.k + row0 + t * rs + 8 * q) : make_uint4(0u, 0u, 0u, 0u);
            xv[m] = ok ? *reinterpret_cast<const uint4*>(a.v + row0 + t * rs + 8 * q) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const int e = tid + kThreads * m, t = e >> 5, q = e & 31;
            xg[m] = t < n ? *reinterpret_cast<const float4*>(a.g + row0 + t * rs + 4 * q)
                          : make_float4(1.f, 1.f, 1.f, 1.f);
        }
        if (tid < kC && tid < n) bt = a.beta[tok_row(layer, t0 + tid, head, a.n_tokens, a.n_heads)];
#pragma unroll
        for (int m = 0; m < 2; ++m) {
            const int e = tid + kThreads * m, t = e >> 4, q = e & 15;
            const uint32_t w[4] = {xk[m].x, xk[m].y, xk[m].z, xk[m].w};
            float4* dk = reinterpret_cast<float4*>(KF + t * kD + 8 * q);
            dk[0] = make_float4(__uint_as_float(w[0] << 16), __uint_as_float(w[0] & 0xffff0000u),
                                __uint_as_float(w[1] << 16), __uint_as_float(w[1] & 0xffff0000u));
            dk[1] = make_float4(__uint_as_float(w[2] << 16), __uint_as_float(w[2] & 0xffff0000u),
                                __uint_as_float(w[3] << 16), __uint_as_float(w[3] & 0xffff0000u));
            *reinterpret_cast<uint4*>(smem + OFF_VB + (t * kD + 8 * q) * 2) = xv[m];
        }
#pragma unroll
        for (int m = 0; m < 4; ++m) reinterpret_cast<float4*>(GA)[tid + kThreads * m] = xg[m];
        if (tid < kC) ms->beta[tid] = bt;
#pragma unroll
        for (int m = 0; m < 2; ++m) reinterpret_cast<float4*>(L)[tid + kThreads * m] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ms->tmem_base;

    // ---- kbar: thread c < 128 runs over channel c from the last token back
    if (tid < kD) {
        const int c = tid;
        uint8_t* hi = smem + OFF_A;
        uint8_t* lo = hi + 16384;
        float suf = 1.f;  // gates after token t
#pragma unroll 1
        for (int q = 7; q >= 0; --q) {
            float x[8];
#pragma unroll
            for (int e = 7; e >= 0; --e) {
                const int t = 8 * q + e;
                x[e] = KF[t * kD + c] * suf;
                suf *= GA[t * kD + c];
            }
            store_row8(hi, lo, core_off(c, 8 * q), x);
        }
        ms->gC[c] = suf;
        fence_async_smem();
    }

    // ---- gram: thread (s, group) holds k_s over the channels 4 group + 32 m + e (m, e < 4), times
    // the gates after s, and forms its part of G_ts for every later token t; the eight groups of a
    // column are adjacent lanes and meet by shuffles.  A warp holds columns 4 warp .. 4 warp + 3, so
    // its loop starts at t = 4 warp + 1.
    {
        const int s = tid >> 3, grp = tid & 7;
        float z[16];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const float4 x = *reinterpret_cast<const float4*>(KF + s * kD + 4 * grp + 32 * m);
            z[4 * m] = x.x, z[4 * m + 1] = x.y, z[4 * m + 2] = x.z, z[4 * m + 3] = x.w;
        }
#pragma unroll 1
        for (int t = 4 * warp + 1; t < n; ++t) {
            float4 ga[4], kt[4];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                ga[m] = *reinterpret_cast<const float4*>(GA + t * kD + 4 * grp + 32 * m);
                kt[m] = *reinterpret_cast<const float4*>(KF + t * kD + 4 * grp + 32 * m);
            }
            const bool act = t > s;
            if (act) {
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    z[4 * m] *= ga[m].x, z[4 * m + 1] *= ga[m].y, z[4 * m + 2] *= ga[m].z, z[4 * m + 3] *= ga[m].w;
                }
            }
            float p0 = 0.f, p1 = 0.f;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                p0 = fmaf(kt[m].x, z[4 * m], p0);
                p1 = fmaf(kt[m].y, z[4 * m + 1], p1);
                p0 = fmaf(kt[m].z, z[4 * m + 2], p0);
                p1 = fmaf(kt[m].w, z[4 * m + 3], p1);
            }
            float pr = p0 + p1;
            pr += __shfl_xor_sync(0xffffffffu, pr, 1);
            pr += __shfl_xor_sync(0xffffffffu, pr, 2);
            pr += __shfl_xor_sync(0xffffffffu, pr, 4);
            if (act && grp == 0) L[t * kC + s] = ms->beta[t] * pr;
        }
    }
    __syncthreads();

    // ---- solve: thread j < 256 forms column j of [-W | U] over the chunk's tokens.
    if (tid < 2 * kD) {
        const int j = tid;
        const bool isw = j < kD;
        const int c = isw ? j : j - kD;
        float w[kC];
        float gp = 1.f;  // g_t of channel c
#pragma unroll
        for (int t = 0; t < kC; ++t) {
            float x;
            if (isw) {
                gp *= GA[t * kD + c];
                x = -ms->beta[t] * KF[t * kD + c] * gp;
            } else {
                x = ms->beta[t] * __bfloat162float(VB[t * kD + c]);
            }
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int m = 0; 4 * m < t; ++m) {
                const float4 l4 = *reinterpret_cast<const float4*>(L + t * kC + 4 * m);
                acc[m & 3] = fmaf(l4.x, w[4 * m], acc[m & 3]);
                if (4 * m + 1 < t) acc[m & 3] = fmaf(l4.y, w[4 * m + 1], acc[m & 3]);
                if (4 * m + 2 < t) acc[m & 3] = fmaf(l4.z, w[4 * m + 2], acc[m & 3]);
                if (4 * m + 3 < t) acc[m & 3] = fmaf(l4.w, w[4 * m + 3], acc[m & 3]);
            }
            w[t] = x - ((acc[0] + acc[1]) + (acc[2] + acc[3]));
        }
        uint8_t* hi = smem + OFF_B;
        uint8_t* lo = hi + 32768;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = w[8 * q + e];
            store_row8(hi, lo, core_off(j, 8 * q), x);
        }
        fence_async_smem();
    }
    __syncthreads();

    // ---- MMA: D = Kbar^T [-W | U] = hi hi + hi lo + lo hi, four steps of 16 tokens
    if (tid == 0) {
        tc_fence_after();
        const uint32_t sb = smem_u32(smem);
        const uint32_t ah = sb + OFF_A, al = ah + 16384, bh = sb + OFF_B, bl = bh + 32768;
#pragma unroll 1
        for (int kk = 0; kk < 4; ++kk) {
            const uint64_t dah = sdesc_plain(ah + 256 * kk, 128, 1024), dal = sdesc_plain(al + 256 * kk, 128, 1024);
            const uint64_t dbh = sdesc_plain(bh + 256 * kk, 128, 1024), dbl = sdesc_plain(bl + 256 * kk, 128, 1024);
            mma_bf16_ss(tmem, dah, dbh, ID_PAIR, kk > 0);
            mma_bf16_ss(tmem, dah, dbl, ID_PAIR, true);
            mma_bf16_ss(tmem, dal, dbh, ID_PAIR, true);
        }
        mma_commit(&ms->mma_done);
    }
    __syncwarp();
    const bool ok = warp < 8 ? wait_done(&ms->mma_done, a.wait_ns, a.err) : true;
    tc_fence_after();

    // ---- write: warps 0-3 T_chunk (row i = lane of the accumulator), warps 4-7 S_chunk
    const int64_t obj = (int64_t)p * LH + lh;
    if (warp < 8) {
        const int i = 32 * (warp & 3) + lane;
        const uint32_t tl = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
        if (warp < 4) {
            const float gci = ms->gC[i];
            float mx = 0.f;
            if (ok) {
#pragma unroll 1
                for (int cb = 0; cb < 4; ++cb) {
                    uint32_t x[32];
                    tmem_ld32(tl + 32 * cb, x);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const float y = __uint_as_float(x[e]) + (32 * cb + e == i ? gci : 0.f);
                        mx = fmaxf(mx, fabsf(y));
                    }
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            if (lane == 0) ms->red[warp] = mx;
            asm volatile("bar.sync 1, 128;" ::: "memory");
            const float M = fmaxf(fmaxf(ms->red[0], ms->red[1]), fmaxf(ms->red[2], ms->red[3]));
            const int ex = (M > 0.f && isfinite(M)) ? ilogbf(M) : 0;
            if (ok) {
                float* T = a.T_tab + obj * kD * kD + (int64_t)i * kD;
#pragma unroll 1
                for (int cb = 0; cb < 4; ++cb) {
                    uint32_t x[32];
                    tmem_ld32(tl + 32 * cb, x);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; e += 4) {
                        float y[4];
#pragma unroll
                        for (int f = 0; f < 4; ++f)
                            y[f] = scale_pow2(__uint_as_float(x[e + f]) + (32 * cb + e + f == i ? gci : 0.f), -ex);
                        *reinterpret_cast<float4*>(T + 32 * cb + e) = make_float4(y[0], y[1], y[2], y[3]);
                    }
                }
                if (i == 0) a.T_exp_tab[obj] = ex;
            }
        } else if (ok) {
            float* S = a.S_tab + obj * kD * kD + (int64_t)i * kD;
#pragma unroll 1
            for (int cb = 0; cb < 4; ++cb) {
                uint32_t x[32];
                tmem_ld32(tl + kD + 32 * cb, x);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; e += 4)
                    *reinterpret_cast<float4*>(S + 32 * cb + e) = make_float4(
                        __uint_as_float(x[e]), __uint_as_float(x[e + 1]), __uint_as_float(x[e + 2]),
                        __uint_as_float(x[e + 3]));
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// The batch's chunk index: cu_chunk[i] = first chunk of segment seg0 + i (i <= nseg),
// chunk_seg[c] = its segment, iota[c] = c.  One block of 1024 threads.
__global__ void __launch_bounds__(1024) kda_batch_plan_kernel(const int32_t* cu, const int32_t* skip, int seg0,
                                                              int nseg, int32_t* cu_chunk, int32_t* chunk_seg,
                                                              int32_t* iota) {
    __shared__ int32_t wsum[32];
    __shared__ int32_t carry;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    if (tid == 0) carry = 0;
    __syncthreads();
    for (int base = 0; base <= nseg; base += 1024) {
        const int i = base + tid;
        int nc = 0;
        if (i < nseg) {
            const int s = seg0 + i;
            const int body = cu[s + 1] - cu[s] - (skip ? skip[s] : 0);
            nc = body > 0 ? (body + kC - 1) / kC : 0;
        }
        int x = nc;  // inclusive scan in the warp
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) wsum[w] = x;
        __syncthreads();
        if (w == 0) {
            int y = wsum[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int z = __shfl_up_sync(0xffffffffu, y, o);
                if (lane >= o) y += z;
            }
            wsum[lane] = y;  // inclusive over warps
        }
        __syncthreads();
        const int excl = carry + (w > 0 ? wsum[w - 1] : 0) + x - nc;
        if (i <= nseg) cu_chunk[i] = excl;
        __syncthreads();
        if (tid == 0) carry += wsum[31];
        __syncthreads();
    }
    for (int i = tid; i < nseg; i += 1024)
        for (int c = cu_chunk[i]; c < cu_chunk[i + 1]; ++c) {
            chunk_seg[c] = seg0 + i;
            iota[c] = c;
        }
}

size_t al256(size_t b) { return (b + 255) & ~(size_t)255; }

// Chunks of each segment's body and the largest of them, from the host copies.
void chunk_counts(const BuildParams& p, std::vector<int64_t>& nc, int64_t& total, int64_t& most) {
    nc.assign(p.n_seg, 0);
    total = most = 0;
    for (int s = 0; s < p.n_seg; ++s) {
        const int64_t body = (int64_t)p.cu_host[s + 1] - p.cu_host[s] - (p.skip_host ? p.skip_host[s] : 0);
        nc[s] = body > 0 ? (body + kC - 1) / kC : 0;
        total += nc[s];
        most = nc[s] > most ? nc[s] : most;
    }
}

// Workspace of the tensor-core path for batches of up to `cap` chunks:
// [build plan][cu_chunk][chunk_seg][iota][T_exp_tab][T_tab][S_tab].
struct KdaLayout {
    size_t cu_chunk, chunk_seg, iota, t_exp, t_tab, s_tab, end;
};
KdaLayout kda_layout(int n_seg, int64_t cap, int LH) {
    KdaLayout l;
    l.cu_chunk = build_workspace_bytes(n_seg);
    l.chunk_seg = l.cu_chunk + al256(((size_t)n_seg + 1) * 4);
    l.iota = l.chunk_seg + al256((size_t)cap * 4);
    l.t_exp = l.iota + al256((size_t)cap * 4);
    l.t_tab = l.t_exp + al256((size_t)cap * LH * 4);
    l.s_tab = l.t_tab + (size_t)cap * LH * kD * kD * 4;
    l.end = l.s_tab + (size_t)cap * LH * kD * kD * 4;
    return l;
}

constexpr size_t kTableCap = (size_t)4 << 30;  // bytes of chunk tables the reported workspace allows

// Chunks a batch may hold in `bytes` of workspace (0 when not even one).
int64_t cap_for(int n_seg, int LH, size_t bytes) {
    const size_t fixed = kda_layout(n_seg, 0, LH).end;
    if (bytes <= fixed) return 0;
    const size_t per = (size_t)LH * (kPairBytes + 4) + 8;
    int64_t cap = (int64_t)((bytes - fixed) / per);
    while (cap > 0 && kda_layout(n_seg, cap, LH).end > bytes) --cap;  // padding
    return cap;
}

int sm_count_kda() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

}  // namespace

bool kda_build_tc_supported(const BuildParams& p) {
    if (!(p.family == kKDA && p.dk == kD && p.dv == kD && p.in_dtype == kBF16 && p.n_tokens > 0 && p.cu_host &&
          p.g && p.beta && (reinterpret_cast<uintptr_t>(p.g) & 15u) == 0))
        return false;
    std::vector<int64_t> nc;
    int64_t total, most;
    chunk_counts(p, nc, total, most);
    const int64_t LH = (int64_t)p.n_layers * p.n_heads;
    // one segment's chunk pairs must fit a compose table (32-bit TMA row index)
    return total > 0 && most * LH * kD < INT32_MAX;
}

size_t kda_build_tc_workspace_bytes(const BuildParams& p) {
    std::vector<int64_t> nc;
    int64_t total, most;
    chunk_counts(p, nc, total, most);
    const int LH = p.n_layers * p.n_heads;
    const int64_t by_cap = (int64_t)(kTableCap / ((size_t)LH * kPairBytes));
    int64_t cap = total < by_cap ? total : by_cap;
    if (cap < most) cap = most;
    return kda_layout(p.n_seg, cap, LH).end;
}

cudaError_t launch_kda_build_tc(const BuildParams& p, void* workspace, size_t workspace_bytes, unsigned* err,
                                cudaStream_t s) {
    std::vector<int64_t> nc;
    int64_t total, most;
    chunk_counts(p, nc, total, most);
    const int L = p.n_layers, H = p.n_heads, LH = L * H;
    const int64_t cap = cap_for(p.n_seg, LH, workspace_bytes);
    if (cap < most || total == 0) return cudaErrorInvalidValue;
    const KdaLayout ly = kda_layout(p.n_seg, cap, LH);
    char* ws = static_cast<char*>(workspace);
    int32_t* cu_chunk = reinterpret_cast<int32_t*>(ws + ly.cu_chunk);
    int32_t* chunk_seg = reinterpret_cast<int32_t*>(ws + ly.chunk_seg);
    int32_t* iota = reinterpret_cast<int32_t*>(ws + ly.iota);
    int32_t* t_exp = reinterpret_cast<int32_t*>(ws + ly.t_exp);
    float* t_tab = reinterpret_cast<float*>(ws + ly.t_tab);
    float* s_tab = reinterpret_cast<float*>(ws + ly.s_tab);
    if (sm_count_kda() <= 0) return cudaErrorInvalidDevice;
    cudaError_t e = cudaFuncSetAttribute(kda_chunk_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    const int64_t plane = (int64_t)kD * kD;
    for (int s0 = 0; s0 < p.n_seg;) {
        int s1 = s0;
        int64_t np = 0;
        while (s1 < p.n_seg && np + nc[s1] <= cap) np += nc[s1++];
        const int nb = s1 - s0;
        kda_batch_plan_kernel<<<1, 1024, 0, s>>>(p.cu, p.skip, s0, nb, cu_chunk, chunk_seg, iota);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        if (np > 0) {
            ChunkArgs a;
            a.n_layers = L;
            a.n_heads = H;
            a.seg0 = s0;
            a.n_tokens = p.n_tokens;
            a.cu = p.cu;
            a.skip = p.skip;
            a.cu_chunk = cu_chunk;
            a.chunk_seg = chunk_seg;
            a.k = static_cast<const __nv_bfloat16*>(p.k);
            a.v = static_cast<const __nv_bfloat16*>(p.v);
            a.g = p.g;
            a.beta = p.beta;
            a.T_tab = t_tab;
            a.T_exp_tab = t_exp;
            a.S_tab = s_tab;
            a.err = err;
            a.wait_ns = 2000000000ull;
            kda_chunk_pair_kernel<<<(unsigned)(np * LH), kThreads, kSmemBytes, s>>>(a);
            if ((e = cudaGetLastError()) != cudaSuccess) return e;
        }
        ComposeParams c;
        c.family = kKDA;
        c.n_layers = L;
        c.n_heads = H;
        c.dk = c.dv = kD;
        c.n_pairs = (int)np;
        c.n_chains = nb;
        c.T_tab = t_tab;
        c.T_exp_tab = t_exp;
        c.S_tab = s_tab;
        c.cu_chain = cu_chunk;
        c.seg_idx = iota;
        c.S0 = nullptr;
        c.S_out = p.S_out + (int64_t)s0 * LH * plane;
        c.T_out = p.T_out + (int64_t)s0 * LH * plane;
        c.T_exp_out = p.T_exp + (int64_t)s0 * LH;
        e = np > 0 && compose_tc_supported(c) ? launch_compose_tc(c, err, s) : launch_compose_simt(c, err, s);
        if (e != cudaSuccess) return e;
        s0 = s1;
    }
    return cudaSuccess;
}

}  // namespace hypic
