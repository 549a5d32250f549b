// decay_build_tc.cu -- the cached pair of the decay families (RetNet, Mamba2,
// GLA, vanilla linear attention) on the sm_103a tensor cores (d = 128, bf16
// keys and values).
//
// What it computes (aibase article on HYPIC, paragraph on the linear layers:
// the families whose transition is a decay): the transition of every token is
// a scalar (RetNet gamma, Mamba2 a_t) or diagonal (GLA Diag(g_t)) decay, or
// none (vanilla), and the write term k_t v_t^T, so that
//     S(C|0) = sum_t Diag(w_t) k_t v_t^T,  w_t = the product of the decays of
//     the tokens after t in the segment (per key feature for GLA),
//     T_C = the product of all of them (RetNet gamma^L, Mamba2 prod a_t, GLA
//     prod g_t per feature, vanilla I, not stored).
// How: the closed form as a contraction.  Chunks of 64 tokens are taken from
// the segment's end backwards, so that the weight of a token is its in-chunk
// suffix decay times the running decay of the chunks already taken (a scan of
// log2 decays for the scalar families, suffix products of the gates per
// feature for GLA); no accumulator is ever rescaled.  The
// weighted keys K~ = Diag(w) K are formed in shared memory as a pair of bf16
// values (hi + lo, about 16 significant bits) and S^T += V^T K~ runs as bf16
// MMAs (M = N = 128, K = 64 per chunk) into a tensor-memory accumulator; the
// keys of vanilla attention need no weights and go straight from the TMA tile.
// The contraction is 32k flop per token and head against 512 bytes of inputs
// (1 KB with GLA's per-feature gates): the kernel is bound by HBM, not by the
// tensor pipe.
//
// Roles (320 threads): warp 0 takes items from the queue and loads keys,
// values (and GLA gates) by TMA into a ring; warps 1-8 form the weights and
// K~ and write the result (eight warps, so that the latency of one chunk's
// shared-memory traffic is hidden); warp 9 issues the MMAs (one thread), so
// that the workers never wait on MMA issue.  One CTA per SM,
// persistent over (segment, layer, head) items in longest-body-first order;
// every wait is bounded and a wait that runs out sets the device error word.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <float.h>
#include <math.h>
#include <stddef.h>
#include <stdint.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace hypic {
namespace {

using namespace tc;

constexpr int kD = 128, kC = 64;
constexpr int kThreads = 320;
constexpr int kWorkers = 256;   // warps 1-8
constexpr int kWarpMma = 9;
constexpr uint32_t kTile = 16384;   // 64 tokens x 128 bf16: two 64-column TMA boxes, 128-byte swizzle
constexpr uint32_t kGTile = 32768;  // 64 tokens x 128 fp32 gates: four 32-column boxes, unswizzled
constexpr int kItemSlots = 2;
constexpr int kMaxStages = 5;

template <bool kGla>
struct Layout {
    static constexpr int kStages = kGla ? 2 : 4;
    static_assert(kStages <= kMaxStages, "stage barriers");
    static constexpr uint32_t OFF_K = 0;
    static constexpr uint32_t OFF_V = OFF_K + kStages * kTile;
    static constexpr uint32_t OFF_KT = OFF_V + kStages * kTile;      // K~ hi, then lo: two buffers
    static constexpr uint32_t OFF_G = OFF_KT + 2 * 2 * kTile;        // GLA gates (then their weights)
    static constexpr uint32_t OFF_MISC = OFF_G + (kGla ? kStages * kGTile : 0);
};

struct DecSlot {
    int64_t b0, b1, obj;
    uint32_t j0;          // CTA-wide index of the item's first chunk
    int nc, layer, head;  // nc >= 0; nc < 0: the queue is exhausted
};

struct DecMisc {
    uint64_t full[kMaxStages], done[kMaxStages];  // stage landed; the MMAs that read it (and its K~) finished
    uint64_t kt_ready[2];               // K~ buffer j % 2 formed for chunk j (workers -> MMA warp)
    uint64_t acc_free;                  // the epilogue has read the accumulator (workers -> MMA warp)
    uint64_t drain;
    uint64_t slot_full[kItemSlots], slot_read[kItemSlots];
    DecSlot slots[kItemSlots];
    alignas(16) float gprod[2][kD];     // GLA: the gate product of each half chunk, per feature
    int abort_flag;
    uint32_t tmem_base;
};

struct DecArgs {
    int family, n_layers, n_heads, n_seg, n_items;
    int64_t n_tokens;
    const int32_t* cu;
    const int32_t* skip;
    const float* gamma;  // RetNet [L][H]
    const float* alpha;  // Mamba2 [L][N][H]
    float* T_out;
    float* S_out;
    const int32_t* order;
    unsigned* counter;
    unsigned* err;
    uint64_t wait_ns;
    uint32_t wait_limit;
};

// Bounded wait: sleeps until the phase completes; gives up after wait_ns of
// GPU time (or at once when the CTA already aborted), raising the abort flag
// and the device error word.
__device__ __noinline__ bool dec_wait_slow(uint64_t* bar, uint32_t parity, int* abort_flag, uint64_t wait_ns,
                                           unsigned* err) {
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
#pragma unroll 1
        for (int j = 0; j < 16; ++j)
            if (mbar_try_wait_sleep(bar, parity, 2000u)) return true;
        if (*(volatile int*)abort_flag) return false;
        if (globaltimer_ns() - t0 > wait_ns) break;
    }
    *(volatile int*)abort_flag = 1;
    set_error(err, kErrTimeout);
    return false;
}
__device__ __forceinline__ bool dec_wait(uint64_t* bar, uint32_t parity, DecMisc* ms, const DecArgs& a) {
    if (mbar_try_wait(bar, parity)) return true;
    return dec_wait_slow(bar, parity, &ms->abort_flag, a.wait_ns, a.err);
}
__device__ __forceinline__ void wsync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
__device__ __forceinline__ bool wall(bool v) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, 1, 256, p;\n selp.u32 %0, 1, 0, q;\n}\n"
        : "=r"(r)
        : "r"((uint32_t)v)
        : "memory");
    return r != 0;
}

// Warp 0: items from the queue into the slot ring (lane 0), then the tiles of
// each chunk, last chunk first, into the stage ring.  Empty bodies are the
// pair (T = 1, S = 0) and are written here.
template <bool kGla>
__device__ void dec_producer(DecMisc* ms, uint8_t* smem, const DecArgs& a, const CUtensorMap* tk, const CUtensorMap* tv,
                             const CUtensorMap* tg, int lane) {
    using Ly = Layout<kGla>;
    const int LH = a.n_layers * a.n_heads;
    uint32_t j0 = 0;
    for (int k = 0;; ++k) {
        const int s = k % kItemSlots;
        if (k >= kItemSlots && !dec_wait(&ms->slot_read[s], (k / kItemSlots - 1) & 1, ms, a)) return;
        DecSlot it;
        it.nc = -1;
        for (;;) {  // the next non-empty item (lane 0 takes it; the warp writes the empty ones)
            int item = 0;
            if (lane == 0) item = *(volatile int*)&ms->abort_flag ? a.n_items : (int)atomicAdd(a.counter, 1u);
            item = __shfl_sync(0xffffffffu, item, 0);
            if (item >= a.n_items) break;
            const int pos = item / LH, lh = item % LH;
            const int seg = a.order[pos];
            it.layer = lh / a.n_heads;
            it.head = lh % a.n_heads;
            it.b0 = (int64_t)a.cu[seg] + (a.skip ? a.skip[seg] : 0);
            it.b1 = a.cu[seg + 1];
            it.obj = ((int64_t)seg * a.n_layers + it.layer) * a.n_heads + it.head;
            it.nc = (int)((it.b1 - it.b0 + kC - 1) / kC);
            it.j0 = j0;
            if (it.nc > 0) break;
            float4* S = reinterpret_cast<float4*>(a.S_out + it.obj * kD * kD);
            for (int e = lane; e < kD * kD / 4; e += 32) S[e] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (a.family == kGLA)
                for (int i = lane; i < kD; i += 32) a.T_out[it.obj * kD + i] = 1.f;
            else if (a.family != kVANILLA && lane == 0)
                a.T_out[it.obj] = 1.f;
            it.nc = -1;
        }
        if (lane == 0) {
            ms->slots[s] = it;
            mbar_arrive(&ms->slot_full[s]);
        }
        if (it.nc < 0) return;
        for (int jj = 0; jj < it.nc; ++jj) {
            const uint32_t j = j0 + jj, st = j % Ly::kStages, u = j / Ly::kStages;
            if (u >= 1 && !dec_wait(&ms->done[st], (u - 1) & 1, ms, a)) return;
            if (lane == 0) {
                const int c = it.nc - 1 - jj;
                const int z = (int)((int64_t)it.layer * a.n_tokens + it.b0 + (int64_t)c * kC);
                mbar_expect_tx(&ms->full[st], 2 * kTile + (kGla ? kGTile : 0));
                uint8_t* kt = smem + Ly::OFF_K + st * kTile;
                uint8_t* vt = smem + Ly::OFF_V + st * kTile;
                tma_load_3d(kt, tk, &ms->full[st], 0, it.head, z);
                tma_load_3d(kt + 8192, tk, &ms->full[st], 64, it.head, z);
                tma_load_3d(vt, tv, &ms->full[st], 0, it.head, z);
                tma_load_3d(vt + 8192, tv, &ms->full[st], 64, it.head, z);
                if (kGla) {
                    uint8_t* gt = smem + Ly::OFF_G + st * kGTile;
                    for (int b = 0; b < 4; ++b) tma_load_3d(gt + b * 8192, tg, &ms->full[st], 32 * b, it.head, z);
                }
            }
        }
        j0 += (uint32_t)it.nc;
    }
}

// Weighted keys of one chunk, K~ = hi + lo (bf16 pair, same swizzled layout as
// the key tile): 16-byte chunk q of the tile holds features i0..i0+7 of token
// t.  wt(m, t, i0, f[8]) fills the eight weights of the thread's m-th piece.
// The four pieces' keys and weights are all read before any store (a store
// could alias a later read for the compiler and hold it back).
template <typename WF>
__device__ __forceinline__ void form_kt(const uint8_t* ktile, uint8_t* hi, uint8_t* lo, int w, WF wt) {
    uint4 xk[4];
    float fk[4][8];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        const int q = w + kWorkers * m, t = q >> 4, cc = q & 15;
        const uint32_t off = (cc >> 3) * 8192 + t * 128 + ((((uint32_t)cc & 7) ^ (t & 7)) << 4);
        xk[m] = *reinterpret_cast<const uint4*>(ktile + off);
        wt(m, t, 64 * (cc >> 3) + 8 * (cc & 7), fk[m]);
    }
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        const int q = w + kWorkers * m, t = q >> 4, cc = q & 15;
        const uint32_t off = (cc >> 3) * 8192 + t * 128 + ((((uint32_t)cc & 7) ^ (t & 7)) << 4);
        const uint4 x = xk[m];
        const float* f = fk[m];
        const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
        uint32_t h[4], l[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float a0 = __uint_as_float(xs[e] << 16) * f[2 * e];
            const float a1 = __uint_as_float(xs[e] & 0xffff0000u) * f[2 * e + 1];
            const __nv_bfloat162 hh = __floats2bfloat162_rn(a0, a1);
            const float2 hf = __bfloat1622float2(hh);
            const __nv_bfloat162 ll = __floats2bfloat162_rn(a0 - hf.x, a1 - hf.y);
            h[e] = *reinterpret_cast<const uint32_t*>(&hh);
            l[e] = *reinterpret_cast<const uint32_t*>(&ll);
        }
        *reinterpret_cast<uint4*>(hi + off) = make_uint4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<uint4*>(lo + off) = make_uint4(l[0], l[1], l[2], l[3]);
    }
}

constexpr uint32_t kIdesc = idesc(1, 128, 128, true, true);  // S^T += V^T K~: both operands MN-major

// Warps 1-8 (w = 0..255).  The accumulator holds S^T: its lane n is column n
// of S.  RetNet's weights are a closed form.  Mamba2 and GLA multiply: a
// token's weight is the suffix product of the gates after it in its chunk, in
// fp32, times the product over the chunks already taken, kept in double; T is
// that product at the end.  Mamba2: a shuffle scan over the 64 tokens (two a
// lane) in every warp.  GLA: thread w takes feature w % 128 over half w / 128
// of the chunk's tokens, the halves joined through shared memory.
template <bool kGla>
__device__ void dec_workers(DecMisc* ms, uint8_t* smem, const DecArgs& a, uint32_t tmem, int w) {
    using Ly = Layout<kGla>;
    const int fam = a.family;
    const int tq = (1 + (w >> 5)) & 3;  // warps 1..8 access tensor-memory lane quarters 1, 2, 3, 0, 1, 2, 3, 0
    for (int k = 0;; ++k) {
        const int s = k % kItemSlots;
        if (!wall(dec_wait(&ms->slot_full[s], (k / kItemSlots) & 1, ms, a))) return;
        const DecSlot it = ms->slots[s];
        wsync();
        if (w == 0) mbar_arrive(&ms->slot_read[s]);
        if (it.nc < 0) return;
        const float lg = fam == kRETNET ? log2f(fmaxf(a.gamma[(int64_t)it.layer * a.n_heads + it.head], FLT_MIN)) : 0.f;
        // The decay over the chunks taken so far: of feature w % 128 (GLA) or of the head (Mamba2).
        double rprod = 1.0;
        // Mamba2: the gates of tokens 2 lane + {0, 1} of the chunk taken now (acur) and of the one taken next
        // (an1); each chunk's are loaded two chunks before it is taken, and every warp scans them itself.
        // Tokens past the body end read as 1.
        float acur[2] = {1.f, 1.f}, an1[2] = {1.f, 1.f};
        auto load_gates = [&](int cc, float (&g)[2]) {
            const int64_t tc = it.b0 + (int64_t)cc * kC;
            for (int e = 0; e < 2; ++e) {
                const int64_t t = tc + 2 * (w & 31) + e;
                g[e] = t < it.b1 ? a.alpha[tok_row(it.layer, t, it.head, a.n_tokens, a.n_heads)] : 1.f;
            }
        };
        if (fam == kMAMBA2) {
            load_gates(it.nc - 1, acur);
            if (it.nc >= 2) load_gates(it.nc - 2, an1);
        }
        for (int jj = 0; jj < it.nc; ++jj) {
            const uint32_t j = it.j0 + jj, st = j % Ly::kStages, u = j / Ly::kStages;
            const int c = it.nc - 1 - jj;
            const int64_t t0 = it.b0 + (int64_t)c * kC;
            const int nvalid = (int)((it.b1 - t0) < kC ? (it.b1 - t0) : kC);
            bool ok = dec_wait(&ms->full[st], u & 1, ms, a);
            // K~ buffer j % 2 was last read by the MMAs of chunk j - 2
            ok = ok && (j < 2 || dec_wait(&ms->done[(j - 2) % Ly::kStages], ((j - 2) / Ly::kStages) & 1, ms, a));
            if (kGla ? !wall(ok) : !__all_sync(0xffffffffu, ok)) return;
            const uint8_t* ktile = smem + Ly::OFF_K + st * kTile;
            uint8_t* hi = smem + Ly::OFF_KT + (j & 1) * 2 * kTile;
            uint8_t* lo = hi + kTile;
            if (fam == kGLA) {
                // feature f, tokens [32 hf, 32 hf + 32): the gate tile (box f / 32 holds [64 t][32 features])
                // is rewritten in place with the weights
                float* gt = reinterpret_cast<float*>(smem + Ly::OFF_G + st * kGTile);
                const int f = w & (kD - 1), hf = w >> 7;
                float* col = gt + (f >> 5) * 2048 + (f & 31);
                float ph = 1.f;
#pragma unroll 8
                for (int t = 32 * hf; t < 32 * hf + 32; ++t)
                    if (t < nvalid) ph *= col[t * 32];
                ms->gprod[hf][f] = ph;
                wsync();
                const float p0 = ms->gprod[0][f], p1 = ms->gprod[1][f];
                float suf = (float)rprod * (hf == 0 ? p1 : 1.f);
#pragma unroll 8
                for (int t = 32 * hf + 31; t >= 32 * hf; --t) {
                    const float g = col[t * 32];
                    col[t * 32] = t < nvalid ? suf : 0.f;
                    if (t < nvalid) suf *= g;
                }
                rprod *= (double)p0 * (double)p1;
                wsync();
                form_kt(ktile, hi, lo, w, [&](int, int t, int i0, float (&f)[8]) {
                    const float* src = gt + (i0 >> 5) * 2048 + t * 32 + (i0 & 31);
                    const float4 x0 = *reinterpret_cast<const float4*>(src);
                    const float4 x1 = *reinterpret_cast<const float4*>(src + 4);
                    f[0] = x0.x, f[1] = x0.y, f[2] = x0.z, f[3] = x0.w;
                    f[4] = x1.x, f[5] = x1.y, f[6] = x1.z, f[7] = x1.w;
                });
            } else if (fam != kVANILLA) {
                // The scalar weights of the tokens this thread's 16-byte pieces belong to (t = (w + 256 m) / 16,
                // m = 0..3), formed by each warp itself: no barrier between the warps.
                const int lane = w & 31;
                float wm[4];
                if (fam == kRETNET) {  // gamma to the number of body tokens after t (closed form)
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        const int t = (w + kWorkers * m) >> 4;
                        wm[m] = t < nvalid ? exp2f(fmaxf(lg * (float)(it.b1 - 1 - (t0 + t)), -149.f)) : 0.f;
                    }
                } else {  // Mamba2: exclusive suffix products of a over the chunk, a shuffle scan in every warp
                    const float a0 = acur[0], a1 = acur[1];
                    acur[0] = an1[0], acur[1] = an1[1];
                    if (c >= 2) load_gates(c - 2, an1);  // (the chunk taken two after this one)
                    float suf = a0 * a1;  // inclusive suffix product over lanes >= lane
#pragma unroll
                    for (int off = 1; off < 32; off <<= 1) {
                        const float y = __shfl_down_sync(0xffffffffu, suf, off);
                        if (lane + off < 32) suf *= y;
                    }
                    const float after = __shfl_down_sync(0xffffffffu, suf, 1);
                    const float w1 = (float)rprod * (lane < 31 ? after : 1.f);  // token 2 lane + 1
                    const float wt0 = 2 * lane < nvalid ? w1 * a1 : 0.f;
                    const float wt1 = 2 * lane + 1 < nvalid ? w1 : 0.f;
                    rprod *= (double)__shfl_sync(0xffffffffu, suf, 0);
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        const int t = (w + kWorkers * m) >> 4;
                        const float x0 = __shfl_sync(0xffffffffu, wt0, t >> 1);
                        const float x1 = __shfl_sync(0xffffffffu, wt1, t >> 1);
                        wm[m] = (t & 1) ? x1 : x0;
                    }
                }
                form_kt(ktile, hi, lo, w, [&](int m, int, int, float (&f)[8]) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) f[e] = wm[m];
                });
            } else if (nvalid < kC) {
                // vanilla: the MMA reads the key tile itself, so the rows past the body end are cleared
                uint8_t* kw = smem + Ly::OFF_K + st * kTile;
                for (int e = w; e < (kC - nvalid) * 16; e += kWorkers) {
                    const int t = nvalid + e / 16, cc = e % 16;
                    const uint32_t off = (cc >> 3) * 8192 + t * 128 + ((((uint32_t)cc & 7) ^ (t & 7)) << 4);
                    *reinterpret_cast<uint4*>(kw + off) = make_uint4(0u, 0u, 0u, 0u);
                }
            }
            fence_async_smem();
            __syncwarp();
            if ((w & 31) == 0) mbar_arrive(&ms->kt_ready[j & 1]);  // one arrival per worker warp
        }
        // epilogue: thread n writes column n of S (coalesced across the warp), and T
        const uint32_t jl = it.j0 + it.nc - 1;
        if (!wall(dec_wait(&ms->done[jl % Ly::kStages], (jl / Ly::kStages) & 1, ms, a))) return;
        tc_fence_after();
        const int n = 32 * tq + (w & 31), ch = w >> 7;  // warps 1-4 write rows 0-63 of S, warps 5-8 the rest
        float* S = a.S_out + it.obj * kD * kD;
        const uint32_t tl = tmem + ((32u * tq) << 16);
#pragma unroll 1
        for (int cb = 2 * ch; cb < 2 * ch + 2; ++cb) {
            uint32_t x[32];
            tmem_ld32(tl + 32 * cb, x);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) S[(32 * cb + e) * kD + n] = __uint_as_float(x[e]);
        }
        if (fam == kGLA && w < kD) a.T_out[it.obj * kD + w] = (float)rprod;
        if (fam == kRETNET && w == 0)
            a.T_out[it.obj] = (float)pow((double)a.gamma[(int64_t)it.layer * a.n_heads + it.head], (double)(it.b1 - it.b0));
        if (fam == kMAMBA2 && w == 0) a.T_out[it.obj] = (float)rprod;
        tc_fence_before();
        wsync();  // every lane has read the accumulator before the next item's first MMA overwrites it
        if (w == 0) mbar_arrive(&ms->acc_free);
    }
}

// Warp 9, one thread: per chunk, once its K~ is formed (or, for vanilla, its
// tile has landed and been masked), S^T += V^T K~ (A = the value tile, B = K~,
// both MN-major); the first MMA of an item overwrites the accumulator once the
// previous item's epilogue has read it.  Items come from the same slot ring.
template <bool kGla>
__device__ void dec_mma(DecMisc* ms, uint8_t* smem, const DecArgs& a, uint32_t tmem) {
    using Ly = Layout<kGla>;
    const uint32_t sb = smem_u32(smem);
    for (int k = 0;; ++k) {
        const int s = k % kItemSlots;
        if (!dec_wait(&ms->slot_full[s], (k / kItemSlots) & 1, ms, a)) return;
        const DecSlot it = ms->slots[s];
        mbar_arrive(&ms->slot_read[s]);
        if (it.nc < 0) return;
        if (k > 0 && !dec_wait(&ms->acc_free, (k - 1) & 1, ms, a)) return;
        for (int jj = 0; jj < it.nc; ++jj) {
            const uint32_t j = it.j0 + jj, st = j % Ly::kStages;
            if (!dec_wait(&ms->kt_ready[j & 1], (j >> 1) & 1, ms, a)) return;
            tc_fence_after();
            const uint64_t av = sdesc_sw128(sb + Ly::OFF_V + st * kTile, 8192, 1024);
            if (a.family == kVANILLA) {
                const uint64_t bk = sdesc_sw128(sb + Ly::OFF_K + st * kTile, 8192, 1024);
#pragma unroll 1
                for (int kk = 0; kk < 4; ++kk) mma_bf16_ss(tmem, av + 128 * kk, bk + 128 * kk, kIdesc, jj > 0 || kk > 0);
            } else {
                const uint32_t hi = sb + Ly::OFF_KT + (j & 1) * 2 * kTile;
                const uint64_t bh = sdesc_sw128(hi, 8192, 1024), bl = sdesc_sw128(hi + kTile, 8192, 1024);
#pragma unroll 1
                for (int kk = 0; kk < 4; ++kk) {
                    mma_bf16_ss(tmem, av + 128 * kk, bh + 128 * kk, kIdesc, jj > 0 || kk > 0);
                    mma_bf16_ss(tmem, av + 128 * kk, bl + 128 * kk, kIdesc, true);
                }
            }
            mma_commit(&ms->done[st]);
        }
    }
}

template <bool kGla>
__global__ void __launch_bounds__(kThreads, 1)
    decay_build_tc_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                          const __grid_constant__ CUtensorMap tg, const DecArgs a) {
    using Ly = Layout<kGla>;
    extern __shared__ __align__(1024) uint8_t smem[];
    DecMisc* ms = reinterpret_cast<DecMisc*>(smem + Ly::OFF_MISC);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if ((smem_u32(smem) & 1023u) != 0) {
        if (tid == 0) set_error(a.err, kErrBadIndex);
        return;
    }
    if (tid == 0) {
        for (int s = 0; s < Ly::kStages; ++s) {
            mbar_init(&ms->full[s], 1);
            mbar_init(&ms->done[s], 1);
        }
        for (int s = 0; s < kItemSlots; ++s) {
            mbar_init(&ms->slot_full[s], 1);
            mbar_init(&ms->slot_read[s], 2);  // the workers and the MMA warp
        }
        mbar_init(&ms->kt_ready[0], kWorkers / 32);
        mbar_init(&ms->kt_ready[1], kWorkers / 32);
        mbar_init(&ms->acc_free, 1);
        mbar_init(&ms->drain, 1);
        ms->abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tk);
        tma_prefetch_desc(&tv);
        if (kGla) tma_prefetch_desc(&tg);
    }
    if (warp == 1) tmem_alloc(&ms->tmem_base, 128);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ms->tmem_base;
    if (warp == 0)
        dec_producer<kGla>(ms, smem, a, &tk, &tv, &tg, lane);
    else if (warp == kWarpMma) {
        if (lane == 0) dec_mma<kGla>(ms, smem, a, tmem);
    } else
        dec_workers<kGla>(ms, smem, a, tmem, tid - 32);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // Drain: every MMA this CTA issued has completed before tensor memory is freed (after an abort some
    // may still run).  A drain that runs out of polls is reported; the memory is freed all the same.
    if (warp == kWarpMma) {
        if (lane == 0) {
            mma_commit(&ms->drain);
            uint32_t i = 0;
            while (i < a.wait_limit && !mbar_try_wait(&ms->drain, 0)) ++i;
            if (i >= a.wait_limit) set_error(a.err, kErrTimeout);
        }
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 128);
}

// ------------------------------------------------------------------ host --
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

// [n_layers][n_tokens][n_heads][128] as a 3-D tensor (feature, head, layer-token
// row): bf16 boxes of 64 features x 64 rows with 128-byte swizzle, or fp32
// boxes of 32 features x 64 rows unswizzled.
bool make_map(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap* m, const void* base, const BuildParams& p, bool f32) {
    const cuuint64_t es = f32 ? 4 : 2;
    cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)p.n_heads, (cuuint64_t)p.n_layers * (cuuint64_t)p.n_tokens};
    cuuint64_t strides[2] = {(cuuint64_t)kD * es, (cuuint64_t)p.n_heads * kD * es};
    cuuint32_t box[3] = {f32 ? 32u : 64u, 1, (cuuint32_t)kC}, el[3] = {1, 1, 1};
    return enc(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base),
               dims, strides, box, el, CU_TENSOR_MAP_INTERLEAVE_NONE,
               f32 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool kGla>
cudaError_t launch_kind(const BuildParams& p, const DecArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                        const CUtensorMap& tg, cudaStream_t s) {
    using Ly = Layout<kGla>;
    const uint32_t smem = Ly::OFF_MISC + sizeof(DecMisc);
    static_assert(Layout<kGla>::OFF_MISC + sizeof(DecMisc) <= 232448, "shared memory budget");
    cudaError_t e = cudaFuncSetAttribute(decay_build_tc_kernel<kGla>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    const int sms = sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    const int grid = a.n_items < sms ? a.n_items : sms;
    decay_build_tc_kernel<kGla><<<grid, kThreads, smem, s>>>(tk, tv, tg, a);
    return cudaGetLastError();
}

}  // namespace

bool decay_build_tc_supported(const BuildParams& p) {
    return (p.family == kRETNET || p.family == kMAMBA2 || p.family == kGLA || p.family == kVANILLA) && p.dk == kD &&
           p.dv == kD && p.in_dtype == kBF16 && p.n_tokens > 0 && (int64_t)p.n_layers * p.n_tokens < INT32_MAX &&
           encode_fn() != nullptr;
}

cudaError_t launch_decay_build_tc(const BuildParams& p, void* workspace, unsigned* err, cudaStream_t s) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    CUtensorMap tk, tv, tg;
    if (!make_map(enc, &tk, p.k, p, false) || !make_map(enc, &tv, p.v, p, false)) return cudaErrorInvalidValue;
    const bool gla = p.family == kGLA;
    if (gla ? !make_map(enc, &tg, p.g, p, true) : !make_map(enc, &tg, p.k, p, false)) return cudaErrorInvalidValue;
    DecArgs a;
    a.family = p.family;
    a.n_layers = p.n_layers;
    a.n_heads = p.n_heads;
    a.n_seg = p.n_seg;
    a.n_items = p.n_seg * p.n_layers * p.n_heads;
    a.n_tokens = p.n_tokens;
    a.cu = p.cu;
    a.skip = p.skip;
    a.gamma = p.gamma;
    a.alpha = p.alpha;
    a.T_out = p.T_out;
    a.S_out = p.S_out;
    a.order = reinterpret_cast<const int32_t*>(workspace);
    a.counter = reinterpret_cast<unsigned*>(reinterpret_cast<char*>(workspace) + build_workspace_bytes(p.n_seg) - 256);
    a.err = err;
    a.wait_ns = 2000000000ull;
    a.wait_limit = 1u << 26;
    if (a.n_items == 0) return cudaSuccess;
    return gla ? launch_kind<true>(p, a, tk, tv, tg, s) : launch_kind<false>(p, a, tk, tv, tg, s);
}

}  // namespace hypic
