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
// layers and heads are formed independently into a table in the workspace;
// the composition law then chains each segment's chunk pairs in order (the
// compose's state mode gives S(C|0) from a zero state, its transition mode
// T_C), which is exact up to rounding.
// Chunk pair.  Inside a chunk let g_t = a_1 ... a_t (per channel) and g_C its
// last value.  The rescaled state Diag(g_t)^-1 S_t takes one generalised
// Householder step per token, I - b_t x_t y_t^T with x_t = k_t / g_t and
// y_t = k_t * g_t, so the chunk's product is I - X^T W (WY form) with
//     w_t = b_t (y_t - sum_{s<t} G_ts w_s),  u_t = b_t (v_t - sum_{s<t} G_ts u_s),
//     G_ts = y_t . x_s = sum_c k_t[c] k_s[c] (a_{s+1} ... a_t)[c],
// and, with kbar_t = k_t * (a_{t+1} ... a_L) (= k_t g_C / g_t),
//     T_chunk = Diag(g_C) - Kbar^T W,   S_chunk = Kbar^T U.
// Gate products over token ranges come from 16-token block products joined by
// the blocks' totals (never a ratio), so g_t, kbar_t and y_t are in range for
// any a_t in [0, 1].  The gram is the bf16 MMA Y X^T in hi + lo pairs when
// every channel's g_C is at least 2^-100 (x_t = k_t / g_t then stays below
// 2^100 |k_t|); otherwise the chunk forms it on CUDA cores from running
// products of the gates (k_s times the gates after s, met by every later key),
// exact for any gate.
// Steps of a chunk (512 threads; persistent CTAs, the next chunk's keys,
// values, gates and b loaded by cp.async on warps 8-15 while warps 0-7 finish
// Tinv):
//   scan     16-token block products per channel -> g_C, g_t, Kbar^T (bf16 hi + lo operand)
//   gram     Y, X operands -> [Yhi; Ylo] [Xhi; Xlo]^T (M = N = 128, K = 128: the four
//            hi/lo products of G = Y X^T in one accumulator) -> b_t G_ts
//   solve    Tinv = (I + L)^-1, L_ts = b_t G_ts (32 x 32 diagonal blocks by forward
//            substitution, the block below from them); [-W | U] = Tinv X' with rows
//            x_t = [-b_t k_t g_t | b_t v_t], so the pair is Kbar^T Tinv X': first
//            P = Kbar^T Tinv (M = 128, N = 64, K = 64 MMAs in hi + lo pairs)
//   MMA      D = P X': M = 128, N = 256, K = 64 in hi + lo pairs (three products), fp32 in
//            tensor memory
//   write    T_chunk = Diag(g_C) + D_left, normalised by a power of two (its exponent
//            kept beside it), and S_chunk = D_right, one tensor-memory pass on 16 warps into
//            128-byte-swizzled boxes over the spent operands, written out by TMA tile stores
//            (each half of S as soon as its four warps have staged it)
// The chunk tables cost 128 KB per chunk, layer and head; segments are taken
// in batches whose tables fit the workspace (up to 4 GiB of them), and a
// segment longer than a batch in parts: each part's chain starts with the pair
// of the parts before it, copied into the table's first slot.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <stddef.h>
#include <stdint.h>

#include <mutex>
#include <vector>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace hypic {
namespace {

using namespace tc;

constexpr int kD = 128, kC = 64;
constexpr int kThreads = 512;
constexpr int kSStoreB = 128;  // the thread that stores the second half of S_chunk (thread 0 the first, and T)
constexpr int64_t kPairBytes = 2 * kD * kD * 4;  // T and S of one chunk, layer and head

// Shared memory map (bytes).  The MMA operands are K-major without swizzle:
// core matrices of 8 rows x 16 bytes, adjacent along K 128 bytes apart, row
// groups 1024 (K = 64 tokens) or 2048 (K = 128 channels) bytes apart.
// L's rows are kLs floats apart: a warp's lanes, one row each, then write 16-byte pieces of the same
// columns without bank conflicts (4 banks further per row)
constexpr int kLs = 68;
constexpr uint32_t OFF_KB = 0;               // keys, bf16 [64 t][128 c]; 16-byte chunk q of row t at q ^ (t & 15)
constexpr uint32_t OFF_VB = OFF_KB + 16384;  // values, bf16 [64 t][128 c]
constexpr uint32_t OFF_GA = OFF_VB + 16384;  // gates, fp32 [64 t][128 c]; chunk q of row t at q ^ (t & 31);
                                             // then g_t when the gram runs on the tensor cores
constexpr uint32_t OFF_L = OFF_GA + 32768;   // b_t G_ts for s < t, 0 elsewhere: fp32 [64 t][64 s], rows kLs apart
constexpr uint32_t OFF_B = OFF_L + 17408;    // X'^T hi, lo: bf16 [256 j][64 t], 32 KB each; before them
                                             // the gram operands Y hi, lo, X hi, lo: bf16 [64 t][128 c]
constexpr uint32_t OFF_A = OFF_B + 65536;    // Kbar^T, then P = Kbar^T Tinv: hi, lo bf16 [128 i][64 t], 16 KB each
constexpr uint32_t OFF_TI = OFF_A + 32768;    // Tinv = (I + L)^-1: fp32 [64 t][64 s]
constexpr uint32_t OFF_TIO = OFF_TI + 16384;  // Tinv^T hi, lo: bf16 [64 t][64 s] operand, 8 KB each
constexpr uint32_t OFF_R = OFF_TIO + 16384;   // solve scratch: fp32 [32][32]
constexpr uint32_t OFF_MISC = OFF_R + 4096;
constexpr uint32_t OFF_STAGE_S = OFF_B;       // S_chunk as 4 boxes of 128 rows x 32 (128-byte swizzle) over
                                              // X'^T; each half is stored as soon as it is staged, so the
                                              // next chunk's gram operands find the region read
constexpr uint32_t OFF_STAGE_T = OFF_A;       // T_chunk's 4 boxes over P, Tinv and its operand (64 KB): the
                                              // next chunk waits for their read before it forms Kbar^T there

struct KMisc {
    uint64_t gram_done, solve_done, pair_done;
    uint32_t tmem_base;
    int pad;
    float beta[kC];      // b_t of the staged chunk (0 past the body end)
    float gC[kD];        // g_C per channel
    float btot[4][kD];   // gate product of each 16-token block, per channel
    float red[16];       // max |T| of each T warp
};
constexpr uint32_t kSmemBytes = OFF_MISC + sizeof(KMisc);
static_assert(kSmemBytes <= 232448, "shared memory budget");

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t TM_PAIR = 0, TM_GRAM = 256, TM_SOLVE = 384;
constexpr uint32_t ID_PAIR = idesc(1, 128, 256, false, false);  // D = P X' = Kbar^T [-W | U], both K-major
constexpr uint32_t ID_GRAM = idesc(1, 128, 128, false, false);  // [Yhi; Ylo] [Xhi; Xlo]^T, both K-major
constexpr uint32_t ID_SOLVE = idesc(1, 128, 64, false, false);  // P = Kbar^T Tinv
constexpr float kSafeGC = 0x1p-100f;

struct ChunkArgs {
    int n_layers, n_heads, n_items;
    int64_t n_tokens;
    const int64_t* chunk_t0;  // [batch chunks]: first token of each chunk
    const int32_t* chunk_n;   // [batch chunks]: its tokens (1..64)
    const __nv_bfloat16* k;
    const __nv_bfloat16* v;
    const float* g;
    const float* beta;
    float* T_tab;        // [chunks][L][H][128][128] mantissa
    int32_t* T_exp_tab;  // [chunks][L][H]
    float* S_tab;        // [chunks][L][H][128][128]
    unsigned* err;
    uint64_t wait_ns;
};

struct Item {
    int64_t t0, obj;
    int n, layer, head;
};

__device__ __forceinline__ Item decode(const ChunkArgs& a, int item) {
    const int LH = a.n_layers * a.n_heads;
    const int p = item / LH, lh = item % LH;
    Item it;
    it.t0 = a.chunk_t0[p];
    it.n = a.chunk_n[p];
    it.layer = lh / a.n_heads;
    it.head = lh % a.n_heads;
    it.obj = (int64_t)p * LH + lh;
    return it;
}

// Byte offsets: key (t, c) in the staged tile, gate (t, c), and (row, token)
// in a K-major operand of 64 tokens.
__device__ __forceinline__ uint32_t kb_off(int t, int c) {
    return (uint32_t)(t * 256 + ((((c >> 3) ^ (t & 15))) << 4) + (c & 7) * 2);
}
__device__ __forceinline__ uint32_t ga_off(int t, int c) {
    return (uint32_t)(t * 512 + ((((c >> 2) ^ (t & 31))) << 4) + (c & 3) * 4);
}
__device__ __forceinline__ uint32_t core_off(int row, int t) {
    return (uint32_t)((row >> 3) * 1024 + (t >> 3) * 128 + (row & 7) * 16 + (t & 7) * 2);
}
__device__ __forceinline__ float bf_at(const uint8_t* p) {
    return __uint_as_float((uint32_t)(*reinterpret_cast<const uint16_t*>(p)) << 16);
}

// x = hi + lo as a pair of bf16 (hi rounded to nearest, lo the rounded rest).
__device__ __forceinline__ void split2(float x0, float x1, uint32_t& h, uint32_t& l) {
    const __nv_bfloat162 hh = __floats2bfloat162_rn(x0, x1);
    const float2 hf = __bfloat1622float2(hh);
    const __nv_bfloat162 ll = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
    h = *reinterpret_cast<const uint32_t*>(&hh);
    l = *reinterpret_cast<const uint32_t*>(&ll);
}

// Eight consecutive K elements of one operand row, as hi and lo 16-byte pieces.
__device__ __forceinline__ void store_row8(uint8_t* hi, uint8_t* lo, uint32_t off, const float (&x)[8]) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) split2(x[2 * e], x[2 * e + 1], h[e], l[e]);
    *reinterpret_cast<uint4*>(hi + off) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4*>(lo + off) = make_uint4(l[0], l[1], l[2], l[3]);
}

// 1 / x to about one ulp (x normal).
__device__ __forceinline__ float rcp_approx(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

__device__ __noinline__ bool wait_done(uint64_t* bar, uint32_t parity, uint64_t wait_ns, unsigned* err) {
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
#pragma unroll 1
        for (int j = 0; j < 16; ++j)
            if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > wait_ns) break;
    }
    set_error(err, kErrTimeout);
    return false;
}

// The chunk's keys, values and gates (rows past the body end zero-filled) and
// b, by cp.async of every thread.
template <int kNthr>
__device__ __forceinline__ void prefetch(uint8_t* smem, KMisc* ms, const ChunkArgs& a, const Item& it, int tid) {
    const int64_t rs = (int64_t)a.n_heads * kD;
    const int64_t row0 = tok_row(it.layer, it.t0, it.head, a.n_tokens, a.n_heads) * kD;
#pragma unroll
    for (int m = 0; m < 1024 / kNthr; ++m) {
        const int e = tid + kNthr * m, t = e >> 4, q = e & 15;
        const bool ok = t < it.n;
        const int64_t off = ok ? row0 + t * rs + 8 * q : row0;
        cp_async16_zfill(smem + OFF_KB + t * 256 + ((q ^ (t & 15)) << 4), a.k + off, ok);
        cp_async16_zfill(smem + OFF_VB + t * 256 + q * 16, a.v + off, ok);
    }
#pragma unroll
    for (int m = 0; m < 2048 / kNthr; ++m) {
        const int e = tid + kNthr * m, t = e >> 5, q = e & 31;
        const bool ok = t < it.n;
        cp_async16_zfill(smem + OFF_GA + t * 512 + ((q ^ (t & 31)) << 4), a.g + (ok ? row0 + t * rs + 4 * q : row0), ok);
    }
    if (tid < kC) {
        const bool ok = tid < it.n;
        const int64_t r = tok_row(it.layer, it.t0 + (ok ? tid : 0), it.head, a.n_tokens, a.n_heads);
        cp_async4_zfill(&ms->beta[tid], a.beta + r, ok);
    }
    cp_async_commit();
}

__global__ void __launch_bounds__(kThreads, 1)
    kda_chunk_pair_kernel(const __grid_constant__ CUtensorMap tmT, const __grid_constant__ CUtensorMap tmS,
                          const ChunkArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    KMisc* ms = reinterpret_cast<KMisc*>(smem + OFF_MISC);
    float* L = reinterpret_cast<float*>(smem + OFF_L);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if ((smem_u32(smem) & 1023u) != 0) {  // the swizzled staging boxes need 1024-byte alignment
        if (tid == 0) set_error(a.err, kErrBadIndex);
        return;
    }
    if (tid == 0) {
        mbar_init(&ms->gram_done, 1);
        mbar_init(&ms->solve_done, 1);
        mbar_init(&ms->pair_done, 1);
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(&ms->tmem_base, kTmemCols);
    Item nxt = {};  // the next item, decoded when its loads are issued
    if ((int)blockIdx.x < a.n_items) {
        nxt = decode(a, blockIdx.x);
        prefetch<kThreads>(smem, ms, a, nxt, tid);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ms->tmem_base;
    uint32_t n_gram = 0, n_pair = 0;

#pragma unroll 1
    for (int item = blockIdx.x; item < a.n_items; item += gridDim.x) {
        const Item it = nxt;
        const bool more = item + (int)gridDim.x < a.n_items;
        if (more) nxt = decode(a, item + gridDim.x);  // loads issued here, used at the prefetch
        // After the first chunk only warps 8-15 have loads in flight (they issue the prefetch); in
        // threads 0 and kSStoreB (warps 0 and 4) the wait would also cover the pair's bulk stores.
        if (item == (int)blockIdx.x || warp >= 8) cp_async_wait_all();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();

        // ---- scan: thread (channel c, block b) over tokens 16 b .. 16 b + 15
        bool safe;
        {
            const int c = tid & (kD - 1), blk = tid >> 7;
            // token t = 16 blk + e of channel c: gate chunk (c / 4) ^ (t & 31), the thread's parts hoisted
            uint8_t* gr = smem + OFF_GA + 16 * blk * 512 + (c & 3) * 4;
            const int gq = (c >> 2) ^ ((16 * blk) & 31);
            float al[16], pi[16], sg[16];
#pragma unroll
            for (int e = 0; e < 16; ++e)
                al[e] = 16 * blk + e < it.n ? *reinterpret_cast<const float*>(gr + e * 512 + ((gq ^ e) << 4)) : 1.f;
            pi[0] = al[0];
#pragma unroll
            for (int e = 1; e < 16; ++e) pi[e] = pi[e - 1] * al[e];
            sg[15] = 1.f;
#pragma unroll
            for (int e = 14; e >= 0; --e) sg[e] = sg[e + 1] * al[e + 1];
            ms->btot[blk][c] = pi[15];
            __syncthreads();
            float E = 1.f, F = 1.f;  // gate products of the blocks before and after this one
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const float P = ms->btot[b][c];
                if (b < blk) E *= P;
                if (b > blk) F *= P;
            }
            const float gC = ((ms->btot[0][c] * ms->btot[1][c]) * ms->btot[2][c]) * ms->btot[3][c];
            if (blk == 0) ms->gC[c] = gC;
            safe = __syncthreads_and(gC >= kSafeGC) != 0;
            if (safe) {
#pragma unroll
                for (int e = 0; e < 16; ++e) *reinterpret_cast<float*>(gr + e * 512 + ((gq ^ e) << 4)) = E * pi[e];
            } else {
                // Kbar^T from the gates themselves (k_t g_C / g_t is not in range here), once the previous
                // chunk's T stores have read the A region; the other path forms it beside the gram MMAs
                if (tid == 0 || tid == kSStoreB) cp_bulk_wait_read();
                __syncthreads();
                uint8_t* ahi = smem + OFF_A;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float x[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int tt = 8 * h + e;
                        x[e] = bf_at(smem + OFF_KB + kb_off(16 * blk + tt, c)) * (sg[tt] * F);
                    }
                    store_row8(ahi, ahi + 16384, core_off(c, 16 * blk + 8 * h), x);
                }
                fence_async_smem();
            }
        }

        if (safe) {
            // ---- gram operands: task (channel octet q8, token t); Y = k g, X = k / g, over the boxes
            // that the previous chunk's S stores have read by now (the other path waited above)
            if (tid == 0) cp_bulk_wait_read_n<1>();
            if (tid == kSStoreB) cp_bulk_wait_read();
            __syncthreads();  // every g_t written
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                const int task = tid + kThreads * m, q8 = task >> 6, t = task & 63;
                const uint4 kx = *reinterpret_cast<const uint4*>(smem + OFF_KB + t * 256 + ((q8 ^ (t & 15)) << 4));
                const float4 g0 = *reinterpret_cast<const float4*>(smem + OFF_GA + t * 512 + (((2 * q8) ^ (t & 31)) << 4));
                const float4 g1 =
                    *reinterpret_cast<const float4*>(smem + OFF_GA + t * 512 + (((2 * q8 + 1) ^ (t & 31)) << 4));
                const uint32_t kw[4] = {kx.x, kx.y, kx.z, kx.w};
                const float gv[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
                float y[8], x[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float kv = __uint_as_float((e & 1) ? (kw[e >> 1] & 0xffff0000u) : (kw[e >> 1] << 16));
                    y[e] = kv * gv[e];
                    x[e] = kv * rcp_approx(gv[e]);
                }
                const uint32_t off = (uint32_t)((t >> 3) * 2048 + q8 * 128 + (t & 7) * 16);
                store_row8(smem + OFF_B, smem + OFF_B + 16384, off, y);
                store_row8(smem + OFF_B + 32768, smem + OFF_B + 49152, off, x);
            }
            fence_async_smem();
            __syncthreads();
            if (tid == kThreads - 32) {  // lane 0 of warp 15 issues; warps 0-14 go on to Kbar^T
                tc_fence_after();
                const uint32_t sb = smem_u32(smem);
                const uint32_t yh = sb + OFF_B, xh = yh + 32768;
                // Y lo follows Y hi and X lo follows X hi at the 8-row group stride, so [Yhi; Ylo] and
                // [Xhi; Xlo] are M = 128 and N = 128 operands: one MMA a K step gives all four products
#pragma unroll 1
                for (int kk = 0; kk < 8; ++kk)
                    mma_bf16_ss(tmem + TM_GRAM, sdesc_plain(yh + 256 * kk, 128, 2048), sdesc_plain(xh + 256 * kk, 128, 2048),
                                ID_GRAM, kk > 0);
                mma_commit(&ms->gram_done);
            }
            // Kbar^T (k_t g_C / g_t) on warps 0-14 while the gram's MMAs run, once the previous chunk's
            // T stores have read the A region: task (row i, tokens 8 o ..)
            if (warp < 15) {
                if (tid == 0) cp_bulk_wait_read();
                asm volatile("bar.sync 3, 480;" ::: "memory");
            }
            for (int task = tid; warp < 15 && task < 1024; task += kThreads - 32) {
                const int i = task & (kD - 1), o = task >> 7;
                const float gci = ms->gC[i];
                // token t = 8 o + e: swizzled chunks (i / 8) ^ (t & 15) and (i / 4) ^ (t & 31), the task's
                // parts hoisted
                const uint8_t* kr = smem + OFF_KB + 8 * o * 256 + (i & 7) * 2;
                const uint8_t* gr = smem + OFF_GA + 8 * o * 512 + (i & 3) * 4;
                const int kq = (i >> 3) ^ ((8 * o) & 15), gq = (i >> 2) ^ ((8 * o) & 31);
                float x[8];
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    x[e] = bf_at(kr + e * 256 + ((kq ^ e) << 4)) *
                           (gci * rcp_approx(*reinterpret_cast<const float*>(gr + e * 512 + ((gq ^ e) << 4))));
                store_row8(smem + OFF_A, smem + OFF_A + 16384, core_off(i, 8 * o), x);
            }
            fence_async_smem();
            __syncwarp();
            const bool ok = __syncthreads_and(wait_done(&ms->gram_done, n_gram & 1, a.wait_ns, a.err)) != 0;
            ++n_gram;
            if (!ok) break;
            tc_fence_after();
            // b_t G_ts for s < t, G = Yhi Xhi + Yhi Xlo + Ylo Xhi + Ylo Xlo: accumulator rows 64 + t hold
            // the Y lo products and columns 64 + s the X lo ones. Warp (quarter q, columns 16 cb ..):
            // quarters 2 and 3 leave their sums in L, then quarters 0 and 1 add theirs, scale and mask.
            {
                const int q = warp & 3, cb = warp >> 2, t = 32 * (q & 1) + lane;
                uint32_t g0[16], g1[16];
                tmem_ld16(tmem + ((32u * q) << 16) + TM_GRAM + 16 * cb, g0);
                tmem_ld16(tmem + ((32u * q) << 16) + TM_GRAM + 64 + 16 * cb, g1);
                tmem_wait_ld();
                float4* Lr = reinterpret_cast<float4*>(L + t * kLs + 16 * cb);
                if (q >= 2) {
#pragma unroll
                    for (int e = 0; e < 16; e += 4)
                        Lr[e / 4] = make_float4(__uint_as_float(g0[e]) + __uint_as_float(g1[e]),
                                                __uint_as_float(g0[e + 1]) + __uint_as_float(g1[e + 1]),
                                                __uint_as_float(g0[e + 2]) + __uint_as_float(g1[e + 2]),
                                                __uint_as_float(g0[e + 3]) + __uint_as_float(g1[e + 3]));
                }
                __syncthreads();
                if (q < 2) {
                    const float coef = ms->beta[t];
#pragma unroll
                    for (int e = 0; e < 16; e += 4) {
                        const int s = 16 * cb + e;
                        const float4 lo = Lr[e / 4];
                        float4 o;
                        o.x = s < t ? coef * ((__uint_as_float(g0[e]) + __uint_as_float(g1[e])) + lo.x) : 0.f;
                        o.y = s + 1 < t ? coef * ((__uint_as_float(g0[e + 1]) + __uint_as_float(g1[e + 1])) + lo.y) : 0.f;
                        o.z = s + 2 < t ? coef * ((__uint_as_float(g0[e + 2]) + __uint_as_float(g1[e + 2])) + lo.z) : 0.f;
                        o.w = s + 3 < t ? coef * ((__uint_as_float(g0[e + 3]) + __uint_as_float(g1[e + 3])) + lo.w) : 0.f;
                        Lr[e / 4] = o;
                    }
                }
            }
        } else {
            // ---- gram on CUDA cores, exact for any gate: thread (s, group) holds k_s over the
            // channels 4 group + 32 m + e, times the gates after s, and meets every later key
#pragma unroll
            for (int m = 0; m < 3; ++m)
                if (tid + kThreads * m < 64 * kLs / 4)
                    reinterpret_cast<float4*>(L)[tid + kThreads * m] = make_float4(0.f, 0.f, 0.f, 0.f);
            __syncthreads();
            const int s = tid >> 3, grp = tid & 7;
            float z[16];
#pragma unroll
            for (int m = 0; m < 4; ++m)
#pragma unroll
                for (int e = 0; e < 4; ++e) z[4 * m + e] = bf_at(smem + OFF_KB + kb_off(s, 4 * grp + 32 * m + e));
#pragma unroll 1
            for (int t = 4 * warp + 1; t < it.n; ++t) {
                float4 ga[4];
                uint2 kt[4];
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const int c0 = 4 * grp + 32 * m;
                    ga[m] = *reinterpret_cast<const float4*>(smem + OFF_GA + ga_off(t, c0));
                    kt[m] = *reinterpret_cast<const uint2*>(smem + OFF_KB + kb_off(t, c0));
                }
                if (t > s) {
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        z[4 * m] *= ga[m].x, z[4 * m + 1] *= ga[m].y, z[4 * m + 2] *= ga[m].z, z[4 * m + 3] *= ga[m].w;
                    }
                }
                float p0 = 0.f, p1 = 0.f;
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    p0 = fmaf(__uint_as_float(kt[m].x << 16), z[4 * m], p0);
                    p1 = fmaf(__uint_as_float(kt[m].x & 0xffff0000u), z[4 * m + 1], p1);
                    p0 = fmaf(__uint_as_float(kt[m].y << 16), z[4 * m + 2], p0);
                    p1 = fmaf(__uint_as_float(kt[m].y & 0xffff0000u), z[4 * m + 3], p1);
                }
                float pr = p0 + p1;
                pr += __shfl_xor_sync(0xffffffffu, pr, 1);
                pr += __shfl_xor_sync(0xffffffffu, pr, 2);
                pr += __shfl_xor_sync(0xffffffffu, pr, 4);
                if (t > s && grp == 0) L[t * kLs + s] = ms->beta[t] * pr;
            }
        }
        if (tid == 0) cp_bulk_wait_read();  // the previous chunk's T stores have read the A region
        __syncthreads();

        // ---- solve: (I + L) [-W | U] = X' with rows x_t = [-b_t k_t g_t | b_t v_t]: Tinv = (I + L)^-1
        // formed on CUDA cores, then Kbar^T [-W | U] = (Kbar^T Tinv) X' on the tensor cores.
        if (!safe) {  // the gates were kept for the CUDA-core gram: now g_t as on the other path
            const int c = tid & (kD - 1), blk = tid >> 7;
            float E = 1.f, gp[16];
#pragma unroll
            for (int b = 0; b < 4; ++b)
                if (b < blk) E *= ms->btot[b][c];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const int t = 16 * blk + e;
                gp[e] = t < it.n ? *reinterpret_cast<const float*>(smem + OFF_GA + ga_off(t, c)) : 1.f;
            }
            float pr = E;
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                pr *= gp[e];
                *reinterpret_cast<float*>(smem + OFF_GA + ga_off(16 * blk + e, c)) = pr;
            }
            __syncthreads();
        }
        {
            // warps 0-1: the 32 x 32 diagonal blocks of Tinv, (I + L_II)^-1 by forward substitution
            // (thread: block I, column r); the other warps: X'^T rows j (K-major over the chunk's
            // tokens), task (octet o, row j) of eight tokens, and zeros in the block above the diagonal
            float* TI = reinterpret_cast<float*>(smem + OFF_TI);
            if (tid < 64) {
                const int I = tid >> 5, r = tid & 31;
                float y[32];
                // every load before any store (a store could alias a later load for the compiler); the
                // inner loop has a fixed trip count, so that it unrolls in full and y stays in registers
#pragma unroll
                for (int t = 0; t < 32; ++t) {
                    const float4* Lr = reinterpret_cast<const float4*>(L + (32 * I + t) * kLs + 32 * I);
                    float acc = t == r ? 1.f : 0.f;
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        if (4 * q >= t) continue;
                        const float4 l4 = Lr[q];
                        acc = fmaf(-l4.x, y[4 * q], acc);
                        if (4 * q + 1 < t) acc = fmaf(-l4.y, y[4 * q + 1], acc);
                        if (4 * q + 2 < t) acc = fmaf(-l4.z, y[4 * q + 2], acc);
                        if (4 * q + 3 < t) acc = fmaf(-l4.w, y[4 * q + 3], acc);
                    }
                    y[t] = acc;
                }
#pragma unroll
                for (int t = 0; t < 32; ++t) TI[(32 * I + t) * kC + 32 * I + r] = y[t];
            } else {
                for (int task = tid - 64; task < 2048; task += kThreads - 64) {
                    const int j = task & 255, o = task >> 8;
                    const bool isw = j < kD;
                    const int c = isw ? j : j - kD;
                    const float4 b0 = *reinterpret_cast<const float4*>(&ms->beta[8 * o]);
                    const float4 b1 = *reinterpret_cast<const float4*>(&ms->beta[8 * o + 4]);
                    const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
                    float x[8];
                    if (isw) {
                        // token t = 8 o + e: the swizzled chunk of channel c is (c / 8) ^ (t & 15) in the
                        // keys, (c / 4) ^ (t & 31) in the gates; the parts fixed by the task hoisted
                        const uint8_t* kr = smem + OFF_KB + 8 * o * 256 + (c & 7) * 2;
                        const uint8_t* gr = smem + OFF_GA + 8 * o * 512 + (c & 3) * 4;
                        const int kq = (c >> 3) ^ ((8 * o) & 15), gq = (c >> 2) ^ ((8 * o) & 31);
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            x[e] = -bv[e] * bf_at(kr + e * 256 + ((kq ^ e) << 4)) *
                                   *reinterpret_cast<const float*>(gr + e * 512 + ((gq ^ e) << 4));
                    } else {
                        const uint8_t* vr = smem + OFF_VB + (8 * o * kD + c) * 2;
#pragma unroll
                        for (int e = 0; e < 8; ++e) x[e] = bv[e] * bf_at(vr + e * kD * 2);
                    }
                    store_row8(smem + OFF_B, smem + OFF_B + 32768, core_off(j, 8 * o), x);
                }
                fence_async_smem();
                // the block above the diagonal: rows 0-31, columns 32-63 (eight float4 a row)
                for (int e = tid - 64; e < 32 * 8; e += kThreads - 64)
                    *reinterpret_cast<float4*>(TI + (e >> 3) * kC + 32 + 4 * (e & 7)) = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        __syncthreads();
        // ---- the staged tiles are read: warps 8-15 load the next chunk while warps 0-7 finish Tinv
        if (warp >= 8) {
            if (more) prefetch<kThreads / 2>(smem, ms, a, nxt, tid - kThreads / 2);
        } else {
            // the block below the diagonal: Tinv_10 = -Tinv_11 (L_10 Tinv_00), 32 x 32 each; thread:
            // column col, rows 4 g4 .. 4 g4 + 3
            float* TI = reinterpret_cast<float*>(smem + OFF_TI);
            float* R = reinterpret_cast<float*>(smem + OFF_R);
            const int col = tid & 31, g4 = tid >> 5;
            {
                const float* L0 = L + (32 + 4 * g4) * kLs;
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int s4 = 0; s4 < 8; ++s4) {
                    float tv[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) tv[e] = TI[(4 * s4 + e) * kC + col];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float4 l = *reinterpret_cast<const float4*>(L0 + k * kLs + 4 * s4);
                        acc[k] = fmaf(l.x, tv[0], fmaf(l.y, tv[1], fmaf(l.z, tv[2], fmaf(l.w, tv[3], acc[k]))));
                    }
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) R[(4 * g4 + k) * 32 + col] = acc[k];
            }
            asm volatile("bar.sync 2, 256;" ::: "memory");
            {
                const float* D0 = TI + (32 + 4 * g4) * kC + 32;  // rows of Tinv_11 (zero above the diagonal)
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int u4 = 0; u4 < 8; ++u4) {
                    if (u4 > g4) break;
                    float rv[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) rv[e] = R[(4 * u4 + e) * 32 + col];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float4 d = *reinterpret_cast<const float4*>(D0 + k * kC + 4 * u4);
                        acc[k] = fmaf(d.x, rv[0], fmaf(d.y, rv[1], fmaf(d.z, rv[2], fmaf(d.w, rv[3], acc[k]))));
                    }
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) TI[(32 + 4 * g4 + k) * kC + col] = -acc[k];
            }
            asm volatile("bar.sync 2, 256;" ::: "memory");
            // Tinv^T as the bf16 hi + lo operand (rows t, K-major over s: Tinv[s][t]): task (row t, octet o)
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                const int task = tid + 256 * m, t = task & 63, o = task >> 6;
                float x[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] = TI[(8 * o + e) * kC + t];
                store_row8(smem + OFF_TIO, smem + OFF_TIO + 8192, core_off(t, 8 * o), x);
            }
            fence_async_smem();
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        // P = Kbar^T Tinv (M = 128, N = 64, K = 64 in hi + lo pairs), then P as the A operand in place
        // of Kbar^T: the pair is D = P X'.
        if (tid == 0) {
            const uint32_t sb = smem_u32(smem);
            const uint32_t ah = sb + OFF_A, al = ah + 16384, th = sb + OFF_TIO, tlo = th + 8192;
#pragma unroll 1
            for (int kk = 0; kk < 4; ++kk) {
                const uint64_t dah = sdesc_plain(ah + 256 * kk, 128, 1024), dal = sdesc_plain(al + 256 * kk, 128, 1024);
                const uint64_t dth = sdesc_plain(th + 256 * kk, 128, 1024), dtl = sdesc_plain(tlo + 256 * kk, 128, 1024);
                mma_bf16_ss(tmem + TM_SOLVE, dah, dth, ID_SOLVE, kk > 0);
                mma_bf16_ss(tmem + TM_SOLVE, dah, dtl, ID_SOLVE, true);
                mma_bf16_ss(tmem + TM_SOLVE, dal, dth, ID_SOLVE, true);
            }
            mma_commit(&ms->solve_done);
        }
        __syncwarp();
        {
            const bool ok = __syncthreads_and(wait_done(&ms->solve_done, n_pair & 1, a.wait_ns, a.err)) != 0;
            if (!ok) break;
        }
        tc_fence_after();
        {
            // warp (quarter q, token quarter cq): rows i = 32 q + lane, tokens 16 cq .. 16 cq + 15
            const int q = warp & 3, cq = warp >> 2, i = 32 * q + lane;
            uint32_t xv[16];
            tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + TM_SOLVE + 16 * cq, xv);
            tmem_wait_ld();
#pragma unroll
            for (int o = 0; o < 2; ++o) {
                float x[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] = __uint_as_float(xv[8 * o + e]);
                store_row8(smem + OFF_A, smem + OFF_A + 16384, core_off(i, 16 * cq + 8 * o), x);
            }
            fence_async_smem();
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();

        // ---- MMA: D = P X' = Kbar^T [-W | U], hi hi + hi lo + lo hi, four steps of 16 tokens
        if (tid == 0) {
            const uint32_t sb = smem_u32(smem);
            const uint32_t ah = sb + OFF_A, al = ah + 16384, bh = sb + OFF_B, bl = bh + 32768;
#pragma unroll 1
            for (int kk = 0; kk < 4; ++kk) {
                const uint64_t dah = sdesc_plain(ah + 256 * kk, 128, 1024), dal = sdesc_plain(al + 256 * kk, 128, 1024);
                const uint64_t dbh = sdesc_plain(bh + 256 * kk, 128, 1024), dbl = sdesc_plain(bl + 256 * kk, 128, 1024);
                mma_bf16_ss(tmem + TM_PAIR, dah, dbh, ID_PAIR, kk > 0);
                mma_bf16_ss(tmem + TM_PAIR, dah, dbl, ID_PAIR, true);
                mma_bf16_ss(tmem + TM_PAIR, dal, dbh, ID_PAIR, true);
            }
            mma_commit(&ms->pair_done);
        }
        __syncwarp();
        const bool ok = __syncthreads_and(wait_done(&ms->pair_done, n_pair & 1, a.wait_ns, a.err)) != 0;
        ++n_pair;
        if (!ok) break;
        tc_fence_after();

        // ---- write: warp (quarter q, part r): r = 0, 1 columns 64 r .. of S_chunk, r = 2, 3 columns
        // 64 (r - 2) .. of T_chunk, staged as 32-column boxes (128-byte swizzle) in the operand area,
        // then stored by TMA: each S part as soon as its four warps have staged it (the next chunk's
        // gram operands go over the S boxes), T after the whole CTA
        {
            const int q = warp & 3, r = warp >> 2, i = 32 * q + lane;
            const bool isT = r >= 2;
            const uint32_t tl = tmem + ((uint32_t)(32 * q) << 16) + TM_PAIR + (isT ? 64 * (r - 2) : 128 + 64 * r);
            uint32_t x0[32], x1[32];
            tmem_ld32(tl, x0);
            tmem_ld32(tl + 32, x1);
            tmem_wait_ld();
            int ex = 0;
            float s1 = 1.f, s2 = 1.f;
            bool two = false;
            if (isT) {
                // Diag(g_C): element (i, i) lies in this warp's 64 columns when r - 2 = q / 2, at column
                // 32 (q & 1) + lane of them (x1 for odd q, x0 for even q)
                if (r - 2 == (q >> 1)) {
                    const float gci = ms->gC[i];
                    if (q & 1) {
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            if (e == lane) x1[e] = __float_as_uint(__uint_as_float(x1[e]) + gci);
                    } else {
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            if (e == lane) x0[e] = __float_as_uint(__uint_as_float(x0[e]) + gci);
                    }
                }
                float mx = 0.f;
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    mx = fmaxf(mx, fmaxf(fabsf(__uint_as_float(x0[e])), fabsf(__uint_as_float(x1[e]))));
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                if (lane == 0) ms->red[warp] = mx;
                asm volatile("bar.sync 1, 256;" ::: "memory");
                float M = 0.f;
#pragma unroll
                for (int wv = 8; wv < 16; ++wv) M = fmaxf(M, ms->red[wv]);
                ex = (M > 0.f && isfinite(M)) ? ilogbf(M) : 0;
                if (i == 0 && r == 2) a.T_exp_tab[it.obj] = ex;
                // 2^-ex as one normal factor where it is one, else as two
                two = ex < -126 || ex > 126;
                const int e1 = two ? -ex / 2 : -ex, e2 = -ex - e1;
                s1 = __int_as_float((e1 + 127) << 23);
                s2 = __int_as_float((e2 + 127) << 23);
            }
            // box b of this warp's 64 columns: row i at i * 128, 16-byte chunk j at j ^ (i & 7)
            uint8_t* box = smem + (isT ? OFF_STAGE_T + (uint32_t)(r - 2) * 32768 : OFF_STAGE_S + (uint32_t)r * 32768);
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                const uint32_t* xs = b ? x1 : x0;
                uint8_t* row = box + b * 16384 + i * 128;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    float4 v = make_float4(__uint_as_float(xs[4 * j]), __uint_as_float(xs[4 * j + 1]),
                                           __uint_as_float(xs[4 * j + 2]), __uint_as_float(xs[4 * j + 3]));
                    if (isT) {
                        v = make_float4(v.x * s1, v.y * s1, v.z * s1, v.w * s1);
                        if (two) v = make_float4(v.x * s2, v.y * s2, v.z * s2, v.w * s2);
                    }
                    *reinterpret_cast<float4*>(row + ((j ^ (i & 7)) << 4)) = v;
                }
            }
            fence_async_smem();
            if (!isT) {
                // the four warps of S part r, then its two boxes by thread 0 (r = 0) or kSStoreB (r = 1)
                if (r == 0)
                    asm volatile("bar.sync 4, 128;" ::: "memory");
                else
                    asm volatile("bar.sync 5, 128;" ::: "memory");
                if (q == 0 && lane == 0) {
                    const int y = (int)(it.obj * kD);
                    tma_store_2d(&tmS, smem + OFF_STAGE_S + r * 32768, 64 * r, y);
                    tma_store_2d(&tmS, smem + OFF_STAGE_S + r * 32768 + 16384, 64 * r + 32, y);
                    cp_bulk_commit();
                }
            }
        }
        __syncthreads();
        if (tid == 0) {
            const int y = (int)(it.obj * kD);
#pragma unroll
            for (int b = 0; b < 4; ++b) tma_store_2d(&tmT, smem + OFF_STAGE_T + b * 16384, 32 * b, y);
            cp_bulk_commit();
        }
    }
    if (tid == 0 || tid == kSStoreB) cp_bulk_wait_all();
    cp_async_wait_all();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// The batch's chunk index: cu_chunk[i] = first chunk of segment seg0 + i (i <= nseg),
// chunk_t0[c], chunk_n[c] = the first token and the tokens of chunk c, iota[c] = c.
// One block of 1024 threads.
__global__ void __launch_bounds__(1024) kda_batch_plan_kernel(const int32_t* cu, const int32_t* skip, int seg0,
                                                              int nseg, int32_t* cu_chunk, int64_t* chunk_t0,
                                                              int32_t* chunk_n, int32_t* iota) {
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
            const int s = seg0 + i;
            const int64_t b0 = (int64_t)cu[s] + (skip ? skip[s] : 0) + (int64_t)(c - cu_chunk[i]) * kC;
            const int64_t rest = cu[s + 1] - b0;
            chunk_t0[c] = b0;
            chunk_n[c] = (int32_t)(rest < kC ? rest : kC);
            iota[c] = c;
        }
}

// One part of a segment too long for a batch: chunks c0 .. c0 + m - 1 of segment `seg` into
// table slots off .. off + m - 1 (slot 0 holds the pair of the chunks before them when off = 1),
// cu_chunk = {0, off + m}, iota over the off + m slots.  One block.
__global__ void kda_part_plan_kernel(const int32_t* cu, const int32_t* skip, int seg, int64_t c0, int m, int off,
                                     int32_t* cu_chunk, int64_t* chunk_t0, int32_t* chunk_n, int32_t* iota) {
    const int64_t b0 = (int64_t)cu[seg] + (skip ? skip[seg] : 0), b1 = cu[seg + 1];
    for (int i = threadIdx.x; i < m; i += blockDim.x) {
        const int64_t t0 = b0 + (c0 + i) * kC, rest = b1 - t0;
        chunk_t0[off + i] = t0;
        chunk_n[off + i] = (int32_t)(rest < kC ? rest : kC);
    }
    for (int j = threadIdx.x; j < off + m; j += blockDim.x) iota[j] = j;
    if (threadIdx.x == 0) {
        cu_chunk[0] = 0;
        cu_chunk[1] = off + m;
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
// [build plan][cu_chunk][chunk_t0][chunk_n][iota][T_exp_tab][T_tab][S_tab].
struct KdaLayout {
    size_t cu_chunk, chunk_t0, chunk_n, iota, t_exp, t_tab, s_tab, end;
};
KdaLayout kda_layout(int n_seg, int64_t cap, int LH) {
    KdaLayout l;
    l.cu_chunk = build_workspace_bytes(n_seg);
    l.chunk_t0 = l.cu_chunk + al256(((size_t)n_seg + 1) * 4);
    l.chunk_n = l.chunk_t0 + al256((size_t)cap * 8);
    l.iota = l.chunk_n + al256((size_t)cap * 4);
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
    const size_t per = (size_t)LH * (kPairBytes + 4) + 16;
    int64_t cap = (int64_t)((bytes - fixed) / per);
    while (cap > 0 && kda_layout(n_seg, cap, LH).end > bytes) --cap;  // padding
    return cap;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn_kda() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// A pair table [rows][128] fp32 as a 2-D tensor: boxes of 32 columns x 128 rows, 128-byte swizzle.
bool table_map(CUtensorMap* m, float* base, uint64_t rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn_kda();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)kD * 4};
    cuuint32_t box[2] = {32, (cuuint32_t)kD}, es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count_kda() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

}  // namespace

// Chunks a batch of the reported workspace holds: all of them, up to 4 GiB of tables, and at
// least 2 (a part of a long segment needs the pair before it plus one chunk).
int64_t reported_cap(const BuildParams& p, int64_t total) {
    const int64_t LH = (int64_t)p.n_layers * p.n_heads;
    const int64_t by_cap = (int64_t)(kTableCap / ((size_t)LH * kPairBytes));
    int64_t cap = total < by_cap ? total : by_cap;
    return cap < 2 ? 2 : cap;
}

bool kda_build_tc_supported(const BuildParams& p) {
    if (!(p.family == kKDA && p.dk == kD && p.dv == kD && p.in_dtype == kBF16 && p.n_tokens > 0 && p.cu_host &&
          p.g && p.beta && (reinterpret_cast<uintptr_t>(p.g) & 15u) == 0))
        return false;
    std::vector<int64_t> nc;
    int64_t total, most;
    chunk_counts(p, nc, total, most);
    const int64_t LH = (int64_t)p.n_layers * p.n_heads;
    // a batch's chunk tables as one compose table (32-bit TMA row index)
    return total > 0 && reported_cap(p, total) * LH * kD < INT32_MAX;
}

size_t kda_build_tc_workspace_bytes(const BuildParams& p) {
    std::vector<int64_t> nc;
    int64_t total, most;
    chunk_counts(p, nc, total, most);
    return kda_layout(p.n_seg, reported_cap(p, total), p.n_layers * p.n_heads).end;
}

cudaError_t launch_kda_build_tc(const BuildParams& p, void* workspace, size_t workspace_bytes, unsigned* err,
                                cudaStream_t s) {
    std::vector<int64_t> nc;
    int64_t total, most;
    chunk_counts(p, nc, total, most);
    const int L = p.n_layers, H = p.n_heads, LH = L * H;
    const int64_t cap = cap_for(p.n_seg, LH, workspace_bytes);
    if (cap < 2 || total == 0) return cudaErrorInvalidValue;
    const KdaLayout ly = kda_layout(p.n_seg, cap, LH);
    char* ws = static_cast<char*>(workspace);
    int32_t* cu_chunk = reinterpret_cast<int32_t*>(ws + ly.cu_chunk);
    int64_t* chunk_t0 = reinterpret_cast<int64_t*>(ws + ly.chunk_t0);
    int32_t* chunk_n = reinterpret_cast<int32_t*>(ws + ly.chunk_n);
    int32_t* iota = reinterpret_cast<int32_t*>(ws + ly.iota);
    int32_t* t_exp = reinterpret_cast<int32_t*>(ws + ly.t_exp);
    float* t_tab = reinterpret_cast<float*>(ws + ly.t_tab);
    float* s_tab = reinterpret_cast<float*>(ws + ly.s_tab);
    const int sms = sm_count_kda();
    if (sms <= 0) return cudaErrorInvalidDevice;
    cudaError_t e = cudaFuncSetAttribute(kda_chunk_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    const int64_t plane = (int64_t)kD * kD;

    // The pairs of np chunks (already planned) into table slots off .. off + np - 1.
    auto chunk_pairs = [&](int64_t np, int64_t off) -> cudaError_t {
        ChunkArgs a;
        a.n_layers = L;
        a.n_heads = H;
        a.n_tokens = p.n_tokens;
        a.chunk_t0 = chunk_t0 + off;
        a.chunk_n = chunk_n + off;
        a.k = static_cast<const __nv_bfloat16*>(p.k);
        a.v = static_cast<const __nv_bfloat16*>(p.v);
        a.g = p.g;
        a.beta = p.beta;
        a.T_tab = t_tab + off * LH * plane;
        a.T_exp_tab = t_exp + off * LH;
        a.S_tab = s_tab + off * LH * plane;
        a.err = err;
        a.wait_ns = 2000000000ull;
        a.n_items = (int)(np * LH);
        const int grid = a.n_items < sms ? a.n_items : sms;
        CUtensorMap tmT, tmS;
        if (!table_map(&tmT, a.T_tab, (uint64_t)np * LH * kD) || !table_map(&tmS, a.S_tab, (uint64_t)np * LH * kD))
            return cudaErrorInvalidValue;
        kda_chunk_pair_kernel<<<grid, kThreads, kSmemBytes, s>>>(tmT, tmS, a);
        return cudaGetLastError();
    };
    // Chains cu_chunk[0..nb] over the np table slots into the outputs of segments s0 .. s0 + nb - 1.
    auto compose = [&](int s0, int nb, int64_t np) -> cudaError_t {
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
        return np > 0 && compose_tc_supported(c) ? launch_compose_tc(c, err, s) : launch_compose_simt(c, err, s);
    };

    for (int s0 = 0; s0 < p.n_seg;) {
        if (nc[s0] > cap) {
            // A segment longer than a batch, in parts: the first part's chunks from slot 0, each later
            // part's after slot 0, which holds the segment's pair so far (the composition law makes
            // that pair followed by the part's chunks the pair of everything up to the part's end).
            for (int64_t c0 = 0; c0 < nc[s0];) {
                const int off = c0 > 0 ? 1 : 0;
                const int64_t m = (nc[s0] - c0 < cap - off) ? nc[s0] - c0 : cap - off;
                if (off) {
                    const size_t tb = (size_t)LH * plane * sizeof(float);
                    if ((e = cudaMemcpyAsync(t_tab, p.T_out + (int64_t)s0 * LH * plane, tb, cudaMemcpyDeviceToDevice,
                                             s)) != cudaSuccess ||
                        (e = cudaMemcpyAsync(t_exp, p.T_exp + (int64_t)s0 * LH, (size_t)LH * sizeof(int32_t),
                                             cudaMemcpyDeviceToDevice, s)) != cudaSuccess ||
                        (e = cudaMemcpyAsync(s_tab, p.S_out + (int64_t)s0 * LH * plane, tb, cudaMemcpyDeviceToDevice,
                                             s)) != cudaSuccess)
                        return e;
                }
                kda_part_plan_kernel<<<1, 256, 0, s>>>(p.cu, p.skip, s0, c0, (int)m, off, cu_chunk, chunk_t0, chunk_n,
                                                       iota);
                if ((e = cudaGetLastError()) != cudaSuccess) return e;
                if ((e = chunk_pairs(m, off)) != cudaSuccess) return e;
                if ((e = compose(s0, 1, m + off)) != cudaSuccess) return e;
                c0 += m;
            }
            ++s0;
            continue;
        }
        int s1 = s0;
        int64_t np = 0;
        while (s1 < p.n_seg && nc[s1] <= cap && np + nc[s1] <= cap) np += nc[s1++];
        const int nb = s1 - s0;
        kda_batch_plan_kernel<<<1, 1024, 0, s>>>(p.cu, p.skip, s0, nb, cu_chunk, chunk_t0, chunk_n, iota);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        if (np > 0 && (e = chunk_pairs(np, 0)) != cudaSuccess) return e;
        if ((e = compose(s0, nb, np)) != cudaSuccess) return e;
        s0 = s1;
    }
    return cudaSuccess;
}

}  // namespace hypic
