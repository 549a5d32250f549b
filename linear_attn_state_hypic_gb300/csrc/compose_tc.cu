// compose_tc.cu -- GDN chain composition on the sm_103a tensor cores (d = 128).
//
// Composition law of the aibase article on HYPIC (paragraph on the linear
// layers): S(C1.C2) = T(C2) S(C1) + S(C2).  Along a chain, for every
// (layer, head), S <- 2^e_p (T~_p S) + S_p for the pairs p in order, where
// T_p = T~_p 2^e_p is stored as an fp32 mantissa and an exponent.
//
// The product must be fp32-accurate (1e-5 on fp32 inputs), so it runs as
// three tf32 passes over a hi/lo split of both operands:
//     T S ~= Tb Sb + Ts Sb + Tb Ss,   x = xb + xs, xb = x with its low 13 mantissa bits cleared,
// dropping only Ts Ss (~2^-22 relative).  Orientation: the accumulator is
// D = (T S)^T -- TMEM lane n holds column n of the new state -- so the state
// itself is the MMA's A operand, kept in tensor memory as Sb^T and Ss^T, and
// T_p (row-major, K-major as stored) is the B operand streamed by TMA in four
// 32-column K-slices.  Per step: MMA = 3 x (M=128, N=128, K=128) tf32;
// epilogue (TMEM lane n): D row n * 2^e_p + column n of S_p (TMA-staged),
// split again into the next step's A, which is announced a K-slice at a time
// (once all of D has been read) so that the next step's MMAs start while the
// epilogue still writes.  The state never leaves the SM until the chain
// ends; the HBM traffic is the pair stream, 128 KB per step.
//
// Roles (320 threads): warp 0 TMA producer, warp 1 MMA issuer, warps 2-5
// split the T slices (hi in place, lo beside it) and, in the reuse chain,
// build the seam units' operands; warps 6-9 the epilogue.
// One CTA per SM, persistent over (chain, layer, head) items ordered
// (layer, head)-major so that chains sharing a pair table run together.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <float.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace hypic {
namespace {

using namespace tc;

constexpr int kD = 128;
constexpr int kSlices = 4;        // K-slices of 32 columns per step
constexpr int kRing = 4;          // slice buffers
constexpr int kThreads = 320;
constexpr int kWarpTMA = 0, kWarpMMA = 1, kWarpCvt0 = 2, kWarpEpi0 = 6;

constexpr uint32_t kSliceBytes = kD * 32 * 4;                    // 128 rows x 32 fp32 = 16 KB
constexpr uint32_t OFF_RING = 0;                                 // kRing x (hi 16 KB, lo 16 KB)
constexpr uint32_t OFF_SP = OFF_RING + kRing * 2 * kSliceBytes;  // S_p: 4 blocks [128 rows][32 cols] fp32
// Reuse chain only: one seam unit (up to kU seam tokens).
constexpr int kU = 8;
// B operand of the unit's dot products (M = 128 state columns, K = 128): rows
// 0..7 = -W hi, 8..15 = g_t q_t hi, 16..23 = -W lo, 24..31 = g_t q_t lo, K-major
// with the 128-byte swizzle in four 32-column slices of 4 KB.  The hi operand
// A_hi of the state takes all 32 rows (N = 32), its lo A_lo the first 16.
constexpr uint32_t kWqSlice = 4 * kU * 128;                      // 32 rows x 128 B
constexpr uint32_t kWqBytes = 4 * kWqSlice;                      // 16 KB
constexpr uint32_t OFF_WQ = OFF_SP + 4 * kSliceBytes;
// B operand of the unit's rank-kU update (N = 128 state rows, K = kU): K^T,
// K-major without swizzle (core matrices of 8 rows x 4 values; the two K halves
// 128 bytes apart, 8-row groups 256 bytes apart); hi, then lo.
constexpr uint32_t kKtBytes = kD * kU * 4;                       // 4 KB
constexpr uint32_t OFF_KT = OFF_WQ + kWqBytes;
// the unit's k and q rows, for its k.k and q.k products
constexpr int kUR = kD + 4;                                      // row stride (floats): rows fall in distinct banks
constexpr uint32_t kUnitRows = kU * kUR * 4;                     // [kU][kUR] fp32
constexpr uint32_t OFF_SK = OFF_KT + 2 * kKtBytes;
constexpr uint32_t OFF_SQ = OFF_SK + kUnitRows;
constexpr uint32_t OFF_MISC = OFF_SQ + kUnitRows;
static_assert(OFF_WQ % 1024 == 0, "128-byte swizzle atoms are 1024-byte aligned");

struct Misc {
    uint64_t full[kRing], cvt[kRing], empty[kRing];
    uint64_t sp_full, sp_empty, d_done, drain;
    uint64_t seam_ready, seam_free;  // unit operands written / consumed
    // reuse chain: the 32 A columns (state rows) 32s..32s+31 split for the next compose / for the
    // unit's dot products (one arrival per epilogue warp); the products in TM_R; C^T in TM_C;
    // the rank-kU update added to TM_D
    uint64_t a_go[kSlices], r_go[kSlices], r_done, c_go, u_done;
    // the current seam unit: tokens [tok0, tok0 + nv); g = in-unit decay prefix
    float kk[kU][kU], qk[kU][kU], th[kU][kU], thg[kU][kU];  // k.k then A, q.k, That, That Diag(g)
    float M[kU][kU];                 // (q_t . k_s) g_t / g_s, s <= t
    float g[kU], lg[kU], sc[kU];     // g_t, log2 g_t, g_w / g_s
    float beta[kU];
    int tok0, nv;
    int item;
    float red[4];  // chain transition: the warps' column maxima
    int abort_flag;
    uint32_t tmem_base;
};
constexpr uint32_t kSmemBytes = OFF_MISC + sizeof(Misc);
static_assert(kSmemBytes <= 232448, "shared memory budget");

constexpr uint32_t TM_D = 0, TM_AB = 128, TM_AS = 256;  // accumulator, A hi, A lo
// Reuse chain: the seam unit's products, lane n: u'_s = U[s][n] - W_s . x is the
// sum of columns 384 + s and 400 + s, g_s q_s . x that of 392 + s and 408 + s;
// its coefficients C^T: hi in 416..423, lo in 424..431.
constexpr uint32_t TM_R = 384, TM_C = 416;
constexpr uint32_t ID_T = idesc(2, 128, 128, false, false);
constexpr uint32_t ID_R32 = idesc(2, 128, 4 * kU, false, false), ID_R16 = idesc(2, 128, 2 * kU, false, false);

struct CtArgs {
    int n_layers, n_heads, n_pairs, n_chains, n_items;
    const int32_t* T_exp;
    const int32_t* cu_chain;
    const int32_t* seg_idx;
    const float* S0;
    float* S_out;
    float* T_out;       // chain transition: each chain's own T (mantissa) ...
    int32_t* T_exp_out;  // ... and its exponent
    unsigned* counter;
    unsigned* err;
    uint32_t wait_limit;
    // reuse chain: seam tokens before each step
    int in_bf16;
    int64_t n_tokens;
    const int32_t* cu_step;
    const void* q;
    const void* k;
    const void* v;
    const float* alpha;
    const float* beta;
    float* o_out;
};

// Seam units of step j: ceil(w / kU) for its w seam tokens.
__device__ __forceinline__ int step_units(const CtArgs& a, int j, int& tb) {
    tb = a.cu_step[j];
    return (a.cu_step[j + 1] - tb + kU - 1) / kU;
}

// Bounded wait: the fast path inline, the polling loop out of line (one copy
// of it keeps the kernel's code small in the instruction cache).
__device__ __noinline__ bool wait_bar_slow(uint64_t* bar, uint32_t parity, int* abort_flag, uint32_t limit,
                                           unsigned* err) {
    for (uint32_t i = 0; i < limit; i += 256) {
#pragma unroll 1
        for (int j = 0; j < 256; ++j)
            if (mbar_try_wait(bar, parity)) return true;
        if (*(volatile int*)abort_flag) return false;
    }
    *(volatile int*)abort_flag = 1;
    set_error(err, kErrTimeout);
    return false;
}
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, Misc* ms, const CtArgs& a) {
    if (mbar_try_wait(bar, parity)) return true;
    return wait_bar_slow(bar, parity, &ms->abort_flag, a.wait_limit, a.err);
}

__device__ __forceinline__ void named_sync(int id) { asm volatile("bar.sync %0, 128;" ::"r"(id) : "memory"); }

__device__ __forceinline__ bool wg_all(int id, bool v) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n"
        " bar.red.and.pred q, %2, 128, p;\n selp.u32 %0, 1, 0, q;\n}\n"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(id)
        : "memory");
    return r != 0;
}

// x = hi + lo with hi = x with its low 13 mantissa bits cleared (exactly a
// tf32 value); lo is exact in fp32 and is read by the MMA as tf32.
__device__ __forceinline__ void split_tf32(float x, uint32_t& hi, uint32_t& lo) {
    const uint32_t b = __float_as_uint(x) & 0xFFFFE000u;
    hi = b;
    lo = __float_as_uint(x - __uint_as_float(b));
}

// ----------------------------------------------------------------- roles --
// gs: CTA-wide slice counter, gj: CTA-wide step counter, both at the start of
// the item (barrier phases run on them across items).  c0, len: the chain's
// range in seg_idx; lh: (layer, head) index.

__device__ void producer_role(Misc* ms, uint8_t* smem, const CtArgs& a, const CUtensorMap* tmT,
                              const CUtensorMap* tmS, uint32_t gs, uint32_t gj, int c0, int len, int lh, bool load_sp) {
    const int LH = a.n_layers * a.n_heads;
    for (int j = 0; j < len; ++j) {
        const int p = a.seg_idx[c0 + j];
        const int row = (p * LH + lh) * kD;
        for (int s = 0; s < kSlices; ++s) {
            const uint32_t gsi = gs + kSlices * j + s, buf = gsi % kRing, u = gsi / kRing;
            if (u >= 1 && !wait_bar(&ms->empty[buf], (u - 1) & 1, ms, a)) return;
            mbar_expect_tx(&ms->full[buf], kSliceBytes);
            tma_load_2d(smem + OFF_RING + buf * 2 * kSliceBytes, tmT, &ms->full[buf], 32 * s, row);
        }
        if (!load_sp) continue;
        const uint32_t g = gj + j;
        if (g >= 1 && !wait_bar(&ms->sp_empty, (g - 1) & 1, ms, a)) return;
        mbar_expect_tx(&ms->sp_full, 4 * kSliceBytes);
        for (int b = 0; b < 4; ++b) tma_load_2d(smem + OFF_SP + b * kSliceBytes, tmS, &ms->sp_full, 32 * b, row);
    }
}

// Reuse chain: the MMAs of the seam units of step js (global unit counter gu).
// Per unit: the dot products TM_R += x (-W; g q)^T over the split state in
// TM_AB / TM_AS (3 x tf32 as A_hi (B_hi; B_lo) + A_lo B_hi, K = 128), a K-slice
// as soon as the epilogue has written it, then, once the epilogue has written
// C^T, the rank-kU update TM_D += C^T K (3 x tf32, K = kU).
__device__ bool mma_units(Misc* ms, uint8_t* smem, const CtArgs& a, uint32_t tmem, int js, uint32_t& gu) {
    int tb;
    const int nu = step_units(a, js, tb);
    const uint32_t wq = smem_u32(smem) + OFF_WQ, kt = smem_u32(smem) + OFF_KT;
    for (int k = 0; k < nu; ++k) {
        if (!wait_bar(&ms->seam_ready, gu & 1, ms, a)) return false;
#pragma unroll 1
        for (int s = 0; s < kSlices; ++s) {
            if (!wait_bar(&ms->r_go[s], gu & 1, ms, a)) return false;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const uint32_t acol = 32 * s + 8 * kk;
                const uint64_t b = sdesc_sw128(wq + s * kWqSlice + kk * 32, 0, 1024);
                mma_tf32_ts(tmem + TM_R, tmem + TM_AB + acol, b, ID_R32, true);
                mma_tf32_ts(tmem + TM_R, tmem + TM_AS + acol, b, ID_R16, true);
            }
        }
        mma_commit(&ms->r_done);
        if (!wait_bar(&ms->c_go, gu & 1, ms, a)) return false;
        tc_fence_after();
        const uint64_t kh = sdesc_plain(kt, 128, 256), kl = sdesc_plain(kt + kKtBytes, 128, 256);
        mma_tf32_ts(tmem + TM_D, tmem + TM_C, kh, ID_T, true);
        mma_tf32_ts(tmem + TM_D, tmem + TM_C, kl, ID_T, true);
        mma_tf32_ts(tmem + TM_D, tmem + TM_C + kU, kh, ID_T, true);
        mma_commit(&ms->u_done);
        ++gu;
    }
    return true;
}

template <bool kSeam, bool kTrans>
__device__ void mma_role(Misc* ms, uint8_t* smem, const CtArgs& a, uint32_t tmem, uint32_t gs, uint32_t gj,
                         uint32_t gu, int c0, int len) {
    const uint32_t ring = smem_u32(smem) + OFF_RING;
    if (kSeam && len > 0 && !mma_units(ms, smem, a, tmem, c0, gu)) return;
    for (int j = 0; j < len; ++j) {
        for (int s = 0; s < kSlices; ++s) {
            const uint32_t gsi = gs + kSlices * j + s, buf = gsi % kRing;
            if (!wait_bar(&ms->a_go[s], (gj + j) & 1, ms, a)) return;
            if (!wait_bar(&ms->cvt[buf], (gsi / kRing) & 1, ms, a)) return;
            tc_fence_after();
            const uint32_t hi = ring + buf * 2 * kSliceBytes, lo = hi + kSliceBytes;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const uint64_t bh = sdesc_sw128(hi + kk * 32, 0, 1024), bl = sdesc_sw128(lo + kk * 32, 0, 1024);
                const uint32_t acol = 32 * s + 8 * kk;
                mma_tf32_ts(tmem + TM_D, tmem + TM_AB + acol, bh, ID_T, !(s == 0 && kk == 0));
                mma_tf32_ts(tmem + TM_D, tmem + TM_AB + acol, bl, ID_T, true);
                mma_tf32_ts(tmem + TM_D, tmem + TM_AS + acol, bh, ID_T, true);
            }
            mma_commit(&ms->empty[buf]);
        }
        mma_commit(&ms->d_done);
        if (kSeam && j + 1 < len && !mma_units(ms, smem, a, tmem, c0 + j + 1, gu)) return;
    }
}

// ------------------------------------------------------------ seam units --
// Reuse chain: before compose step j the running state advances over the
// seam tokens of step j, taken kU at a time.  For a unit of tokens 1..w with
// in-unit decay prefix g_t = a_1 ... a_t, A[t][s] = b_t (g_t/g_s) k_t.k_s
// (s < t), That = (I + A)^-1 Diag(b), W = That Diag(g) K and U = That V (the
// WY form of the token recurrence, as in the build), the state column
// x = S[:, n] becomes, with u'_t = U[t][n] - W_t . x,
//     S_t[:, n] = g_t x + sum_{s<=t} (g_t/g_s) k_s u'_s,
//     o_t[n] = S_t[:, n] . q_t = g_t q_t . x + sum_{s<=t} (q_t . k_s)(g_t/g_s) u'_s,
// and the unit ends at t = w (the padded tokens past w have a = 1, b = 0,
// k = q = v = 0: identity steps).  The converter warpgroup builds the unit's
// operands while the MMAs of the previous compose run: -W and g q as the B
// operand of the dot products, U as their accumulator's starting value in
// tensor memory, K^T for the update and the small tables.  The dot products
// and the update g_w x + K^T c run on the tensor cores; the epilogue takes
// o and the coefficients c_s = (g_w/g_s) u'_s column by column between them.

__device__ __forceinline__ float load_tok(const void* base, int bf16, int64_t row, int i) {
    return bf16 ? __bfloat162float(__ldg(reinterpret_cast<const __nv_bfloat16*>(base) + row * kD + i))
                : __ldg(reinterpret_cast<const float*>(base) + row * kD + i);
}

// The operands of unit gu (tokens [tok0, tok0 + nv) of (layer, head) lh).
// t: converter thread 0..127 (= feature index of the k and q row loads).
__device__ bool prep_unit(Misc* ms, uint8_t* smem, const CtArgs& a, uint32_t tmem, int lh, int tok0, int nv,
                          uint32_t gu, int t) {
    if (gu >= 1 && !wg_all(3, wait_bar(&ms->seam_free, (gu - 1) & 1, ms, a))) return false;
    const int layer = lh / a.n_heads, head = lh % a.n_heads;
    // converter warp 2 + t/32 reaches the TMEM lanes of quarter (t/32 + 2) mod 4:
    // this thread starts the products of state column fl there
    const uint32_t lq = 32u * ((t / 32 + 2) & 3);
    const int fl = lq + (t & 31);
    float* Kf = reinterpret_cast<float*>(smem + OFF_SK);
    float* Qf = reinterpret_cast<float*>(smem + OFF_SQ);
    // every load is issued before any shared-memory store (the stores could
    // otherwise alias the loads for the compiler and serialise them)
    float kr[kU], qr[kU], vr[kU], ga = 1.f, gb = 0.f;
#pragma unroll
    for (int u = 0; u < kU; ++u) {
        const int64_t row = ((int64_t)layer * a.n_tokens + tok0 + (u < nv ? u : 0)) * a.n_heads + head;
        kr[u] = load_tok(a.k, a.in_bf16, row, t);
        qr[u] = load_tok(a.q, a.in_bf16, row, t);
        vr[u] = load_tok(a.v, a.in_bf16, row, fl);
    }
    if (t < kU && t < nv) {
        const int64_t row = ((int64_t)layer * a.n_tokens + tok0 + t) * a.n_heads + head;
        ga = __ldg(a.alpha + row);
        gb = __ldg(a.beta + row);
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
        const bool valid = u < nv;
        kr[u] = valid ? kr[u] : 0.f;
        qr[u] = valid ? qr[u] : 0.f;
        vr[u] = valid ? vr[u] : 0.f;
        Kf[u * kUR + t] = kr[u];
        Qf[u * kUR + t] = qr[u];
    }
    if (t < kU) {
        ms->lg[t] = log2f(fmaxf(ga, FLT_MIN));
        ms->beta[t] = gb;
    }
    named_sync(3);
    {  // k_r . k_c (threads 0..63), q_r . k_c (threads 64..127)
        const int r = (t >> 3) & 7, c = t & 7;
        const float* x = (t < 64 ? Kf : Qf) + r * kUR;
        const float* y = Kf + c * kUR;
        float d0 = 0.f, d1 = 0.f;
#pragma unroll 4
        for (int i = 0; i < kD; i += 8) {
            const float4 x0 = *reinterpret_cast<const float4*>(x + i), x1 = *reinterpret_cast<const float4*>(x + i + 4);
            const float4 y0 = *reinterpret_cast<const float4*>(y + i), y1 = *reinterpret_cast<const float4*>(y + i + 4);
            d0 = fmaf(x0.x, y0.x, fmaf(x0.y, y0.y, fmaf(x0.z, y0.z, fmaf(x0.w, y0.w, d0))));
            d1 = fmaf(x1.x, y1.x, fmaf(x1.y, y1.y, fmaf(x1.z, y1.z, fmaf(x1.w, y1.w, d1))));
        }
        (t < 64 ? ms->kk : ms->qk)[r][c] = d0 + d1;
        if (t == 0) {  // in-unit log-decay prefix
            float acc = 0.f;
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                acc += ms->lg[u];
                ms->lg[u] = acc;
            }
        }
    }
    named_sync(3);
    {  // A[r][s] = b_r (g_r/g_s) k_r.k_s (s < r) in place of k.k; M[r][s] = (g_r/g_s) q_r.k_s (s <= r)
        const int r = (t >> 3) & 7, c = t & 7;
        const float ratio = exp2f(ms->lg[r] - ms->lg[c]);
        if (t < 64) ms->kk[r][c] = c < r ? ms->beta[r] * ratio * ms->kk[r][c] : 0.f;
        else ms->M[r][c] = c <= r ? ms->qk[r][c] * ratio : 0.f;
        if (t < kU) {
            ms->g[t] = exp2f(ms->lg[t]);
            ms->sc[t] = exp2f(ms->lg[kU - 1] - ms->lg[t]);
        }
    }
    named_sync(3);
    if (t < kU) {  // column c of (I + A)^-1 by forward substitution, then That = (.) Diag(b)
        const int c = t;
        float m[kU];
#pragma unroll
        for (int r = 0; r < kU; ++r) {
            float acc = (r == c) ? 1.f : 0.f;
#pragma unroll
            for (int s2 = 0; s2 < r; ++s2) acc = fmaf(-ms->kk[r][s2], m[s2], acc);
            m[r] = acc;
        }
        const float bc = ms->beta[c], gc = ms->g[c];
#pragma unroll
        for (int r = 0; r < kU; ++r) {
            ms->th[r][c] = m[r] * bc;
            ms->thg[r][c] = m[r] * bc * gc;
        }
    }
    named_sync(3);
    uint8_t* wq = smem + OFF_WQ;
#pragma unroll
    for (int u = 0; u < kU; ++u) {  // feature t of rows u of -W and of g_u q_u, split hi/lo
        float w = 0.f;
#pragma unroll
        for (int s2 = 0; s2 <= u; ++s2) w = fmaf(ms->thg[u][s2], kr[s2], w);
        uint32_t h, l;
        split_tf32(-w, h, l);
        *reinterpret_cast<uint32_t*>(wq + sw128_offset(u, t, 4, kWqSlice)) = h;
        *reinterpret_cast<uint32_t*>(wq + sw128_offset(2 * kU + u, t, 4, kWqSlice)) = l;
        split_tf32(ms->g[u] * qr[u], h, l);
        *reinterpret_cast<uint32_t*>(wq + sw128_offset(kU + u, t, 4, kWqSlice)) = h;
        *reinterpret_cast<uint32_t*>(wq + sw128_offset(3 * kU + u, t, 4, kWqSlice)) = l;
    }
    {  // row t of K^T, split hi/lo
        uint4 h0, l0, h1, l1;
        split_tf32(kr[0], h0.x, l0.x), split_tf32(kr[1], h0.y, l0.y);
        split_tf32(kr[2], h0.z, l0.z), split_tf32(kr[3], h0.w, l0.w);
        split_tf32(kr[4], h1.x, l1.x), split_tf32(kr[5], h1.y, l1.y);
        split_tf32(kr[6], h1.z, l1.z), split_tf32(kr[7], h1.w, l1.w);
        uint8_t* kt = smem + OFF_KT + (t >> 3) * 256 + (t & 7) * 16;
        *reinterpret_cast<uint4*>(kt) = h0;
        *reinterpret_cast<uint4*>(kt + 128) = h1;
        *reinterpret_cast<uint4*>(kt + kKtBytes) = l0;
        *reinterpret_cast<uint4*>(kt + kKtBytes + 128) = l1;
    }
    {  // the products' starting value in lane fl: U[s][fl] = (That V)[s][fl], and 0 elsewhere
        uint32_t r[4 * kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            float uu = 0.f;
#pragma unroll
            for (int s2 = 0; s2 <= u; ++s2) uu = fmaf(ms->th[u][s2], vr[s2], uu);
            r[u] = __float_as_uint(uu);
            r[kU + u] = r[2 * kU + u] = r[3 * kU + u] = 0u;
        }
        tmem_st32(tmem + (lq << 16) + TM_R, r);
        tmem_wait_st();
    }
    if (t == 0) {
        ms->tok0 = tok0;
        ms->nv = nv;
    }
    fence_async_smem();
    tc_fence_before();
    named_sync(3);
    if (t == 0) mbar_arrive(&ms->seam_ready);
    return true;
}

// The units of step js (global unit counter gu) for (layer, head) lh.
__device__ bool prep_step_units(Misc* ms, uint8_t* smem, const CtArgs& a, uint32_t tmem, int lh, int js, uint32_t& gu,
                                int t) {
    int tb;
    const int nu = step_units(a, js, tb);
    const int w = a.cu_step[js + 1] - tb;
    for (int k = 0; k < nu; ++k) {
        const int nv = w - kU * k < kU ? w - kU * k : kU;
        if (!prep_unit(ms, smem, a, tmem, lh, tb + kU * k, nv, gu, t)) return false;
        ++gu;
    }
    return true;
}

// This warp's TMEM stores are complete and ordered before the MMAs that
// follow: one arrival (of the four epilogue warps') on bar.
__device__ __forceinline__ void warp_arrive(uint64_t* bar, int lane) {
    tmem_wait_st();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar);
}

// One seam unit on the state, epilogue thread n = TMEM lane n = state column
// n.  On entry TM_AB / TM_AS hold the column x split hi/lo (each K-slice
// announced on r_go as it was written) and TM_D holds g_w x.  The MMAs leave
// u'_s and g_s q_s . x in TM_R; this thread writes o_t and C^T (c_s =
// (g_w/g_s) u'_s, split hi/lo) to TM_C, and the rank-kU MMAs add K^T c to TM_D.
__device__ bool seam_unit(Misc* ms, const CtArgs& a, uint32_t tl, int layer, int head, uint32_t gu, int n) {
    if (!wg_all(4, wait_bar(&ms->r_done, gu & 1, ms, a))) return false;
    tc_fence_after();
    uint32_t r[4 * kU];
    tmem_ld32(tl + TM_R, r);
    tmem_wait_ld();
    const int nv = ms->nv, tok0 = ms->tok0;
    float up[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) up[u] = __uint_as_float(r[u]) + __uint_as_float(r[2 * kU + u]);
    uint32_t cv[2 * kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
        float o = __uint_as_float(r[kU + u]) + __uint_as_float(r[3 * kU + u]);
#pragma unroll
        for (int s2 = 0; s2 <= u; ++s2) o = fmaf(ms->M[u][s2], up[s2], o);
        if (u < nv) a.o_out[(((int64_t)layer * a.n_tokens + tok0 + u) * a.n_heads + head) * kD + n] = o;
        split_tf32(ms->sc[u] * up[u], cv[u], cv[kU + u]);
    }
    tmem_st16(tl + TM_C, cv);
    tmem_wait_st();
    tc_fence_before();
    named_sync(4);  // (also: every column has read the unit's tables)
    if (n == 0) mbar_arrive(&ms->c_go);
    if (!wg_all(4, wait_bar(&ms->u_done, gu & 1, ms, a))) return false;
    tc_fence_after();
    if (n == 0) mbar_arrive(&ms->seam_free);  // the unit's operands have been consumed
    return true;
}

// TM_D -> the A operand, split hi/lo, each K-slice announced as it is written.
// rescale (another unit follows): also TM_D <- gw TM_D, slices on r_go.
// Otherwise (the next compose follows, and its first MMA overwrites TM_D):
// all of TM_D is read first, slices on a_go.
__device__ void split_state(Misc* ms, uint32_t tl, bool rescale, float gw, int lane) {
    if (rescale) {
#pragma unroll 1
        for (int cb = 0; cb < 4; ++cb) {
            uint32_t x[32];
            tmem_ld32(tl + TM_D + 32 * cb, x);
            tmem_wait_ld();
#pragma unroll
            for (int hb = 0; hb < 2; ++hb) {
                uint32_t h[16], l[16];
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) split_tf32(__uint_as_float(x[16 * hb + jj]), h[jj], l[jj]);
                tmem_st16(tl + TM_AB + 32 * cb + 16 * hb, h);
                tmem_st16(tl + TM_AS + 32 * cb + 16 * hb, l);
            }
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) x[jj] = __float_as_uint(gw * __uint_as_float(x[jj]));
            tmem_st32(tl + TM_D + 32 * cb, x);
            warp_arrive(&ms->r_go[cb], lane);
        }
        return;
    }
#pragma unroll
    for (int half = 0; half < 2; ++half) {  // two K-slices at a time
        uint32_t x[2][32];
        tmem_ld32(tl + TM_D + 64 * half, x[0]);
        tmem_ld32(tl + TM_D + 64 * half + 32, x[1]);
        tmem_wait_ld();
        if (half == 1) {  // all of TM_D has been read
            warp_arrive(&ms->a_go[0], lane);
            warp_arrive(&ms->a_go[1], lane);
        }
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const int cb = 2 * half + c;
#pragma unroll
            for (int hb = 0; hb < 2; ++hb) {
                uint32_t h[16], l[16];
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) split_tf32(__uint_as_float(x[c][16 * hb + jj]), h[jj], l[jj]);
                tmem_st16(tl + TM_AB + 32 * cb + 16 * hb, h);
                tmem_st16(tl + TM_AS + 32 * cb + 16 * hb, l);
            }
            if (half == 1) warp_arrive(&ms->a_go[cb], lane);
        }
    }
}

// Applies the units of step js to the state; on entry as for seam_unit (the
// first unit's g_w x in TM_D), on return the A operand of the next compose,
// announced on a_go.
__device__ bool apply_step_units(Misc* ms, const CtArgs& a, uint32_t tl, int lh, int js, uint32_t& gu, int n) {
    int tb;
    const int nu = step_units(a, js, tb);
    const int layer = lh / a.n_heads, head = lh % a.n_heads;
    for (int k = 0; k < nu; ++k) {
        if (!seam_unit(ms, a, tl, layer, head, gu, n)) return false;
        ++gu;
        const bool more = k + 1 < nu;
        float gw = 0.f;
        if (more) {  // the next unit's decay over its tokens
            if (!wg_all(4, wait_bar(&ms->seam_ready, gu & 1, ms, a))) return false;
            gw = ms->g[kU - 1];
        }
        split_state(ms, tl, more, gw, n & 31);
    }
    return true;
}

// Split each T slice into hi (in place) and lo (beside it).  t: 0..127.
// Reuse chain: also the seam units, those of step 0 first and those of step
// j + 1 while the MMAs of step j run.
template <bool kSeam>
__device__ void convert_role(Misc* ms, uint8_t* smem, const CtArgs& a, uint32_t tmem, uint32_t gs, uint32_t gu, int c0,
                             int len, int lh, int t) {
    if (kSeam && len > 0 && !prep_step_units(ms, smem, a, tmem, lh, c0, gu, t)) return;
    for (int j = 0; j < len; ++j) {
        for (int s = 0; s < kSlices; ++s) {
            const uint32_t gsi = gs + kSlices * j + s, buf = gsi % kRing;
            if (!wg_all(3, wait_bar(&ms->full[buf], (gsi / kRing) & 1, ms, a))) return;
            uint8_t* hi = smem + OFF_RING + buf * 2 * kSliceBytes;
            uint8_t* lo = hi + kSliceBytes;
            float4 xs[8];  // (all read before any store: the stores could alias the reads for the compiler)
#pragma unroll
            for (int k = 0; k < 8; ++k) xs[k] = *reinterpret_cast<const float4*>(hi + k * 2048 + t * 16);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint32_t off = k * 2048 + t * 16;
                const float4 x = xs[k];
                uint4 h, l;
                split_tf32(x.x, h.x, l.x);
                split_tf32(x.y, h.y, l.y);
                split_tf32(x.z, h.z, l.z);
                split_tf32(x.w, h.w, l.w);
                *reinterpret_cast<uint4*>(hi + off) = h;
                *reinterpret_cast<uint4*>(lo + off) = l;
            }
            fence_async_smem();
            named_sync(3);
            if (t == 0) mbar_arrive(&ms->cvt[buf]);
        }
        if (kSeam && j + 1 < len && !prep_step_units(ms, smem, a, tmem, lh, c0 + j + 1, gu, t)) return;
    }
}

// Epilogue: thread n owns TMEM lane n = column n of the state.  The next
// step's A operand is announced a K-slice at a time on a_go, once all of
// TM_D has been read (the next compose's first MMA overwrites it).
__device__ void epilogue_role(Misc* ms, uint8_t* smem, const CtArgs& a, uint32_t tmem, uint32_t gj, int c0, int len,
                              int lh, int64_t obj, int q, int lane) {
    const int n = 32 * q + lane;
    const int LH = a.n_layers * a.n_heads;
    const uint32_t tl = tmem + ((32u * q) << 16);
    float* out = a.S_out + obj * kD * kD;
    const float* s0 = a.S0 ? a.S0 + obj * kD * kD : nullptr;
    if (len == 0) {  // empty chain: the start state itself
        for (int i = 0; i < kD; ++i) out[i * kD + n] = s0 ? s0[i * kD + n] : 0.f;
        return;
    }
#pragma unroll 1
    for (int cb = 0; cb < 4; ++cb) {  // A for the first step: the start state (column n), split hi/lo
        uint32_t h[32], l[32];
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) split_tf32(s0 ? s0[(32 * cb + jj) * kD + n] : 0.f, h[jj], l[jj]);
        tmem_st32(tl + TM_AB + 32 * cb, h);
        tmem_st32(tl + TM_AS + 32 * cb, l);
        warp_arrive(&ms->a_go[cb], lane);
    }
    const float* sp = reinterpret_cast<const float*>(smem + OFF_SP) + (n >> 5) * (kSliceBytes / 4) + (n & 31);
    for (int j = 0; j < len; ++j) {
        const uint32_t g = gj + j;
        const int p = a.seg_idx[c0 + j];
        const int e = a.T_exp ? a.T_exp[p * LH + lh] : 0;
        bool ok = wait_bar(&ms->d_done, g & 1, ms, a);
        ok = ok && wait_bar(&ms->sp_full, g & 1, ms, a);
        if (!wg_all(4, ok)) return;
        tc_fence_after();
        // 2^e as two factors (each exact for |e| <= 252)
        const float f1 = exp2f((float)(e / 2)), f2 = exp2f((float)(e - e / 2));
        if (j + 1 == len) {  // the end state
#pragma unroll 1
            for (int cb = 0; cb < 4; ++cb) {
                uint32_t x[32];
                tmem_ld32(tl + TM_D + 32 * cb, x);
                float spv[32];  // (all loaded before any store: the stores to out could alias them)
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) spv[jj] = sp[(32 * cb + jj) * 32];
                tmem_wait_ld();
#pragma unroll
                for (int jj = 0; jj < 32; ++jj)
                    out[(32 * cb + jj) * kD + n] = fmaf(__uint_as_float(x[jj]) * f1, f2, spv[jj]);
            }
        } else {
#pragma unroll 1
            for (int half = 0; half < 2; ++half) {  // two K-slices at a time
                uint32_t x[2][32];
                tmem_ld32(tl + TM_D + 64 * half, x[0]);
                tmem_ld32(tl + TM_D + 64 * half + 32, x[1]);
                tmem_wait_ld();
                if (half == 1) {  // all of TM_D has been read
                    warp_arrive(&ms->a_go[0], lane);
                    warp_arrive(&ms->a_go[1], lane);
                }
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const int cb = 2 * half + c;
                    float spv[32];
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj) spv[jj] = sp[(32 * cb + jj) * 32];
                    uint32_t h[32], l[32];
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj)
                        split_tf32(fmaf(__uint_as_float(x[c][jj]) * f1, f2, spv[jj]), h[jj], l[jj]);
                    tmem_st32(tl + TM_AB + 32 * cb, h);
                    tmem_st32(tl + TM_AS + 32 * cb, l);
                    if (half == 1) warp_arrive(&ms->a_go[cb], lane);
                }
            }
        }
        tmem_wait_st();
        named_sync(4);
        if (n == 0) mbar_arrive(&ms->sp_empty);  // S_p has been read
    }
}

// Reuse-chain epilogue: as epilogue_role, with the seam units of step j + 1
// applied to the composed column before it becomes the A operand of step
// j + 1 (and those of step 0 to the start state).  Before a unit the column
// goes to the A operand (split hi/lo, for the unit's dot products, a K-slice
// at a time on r_go) and, times the unit's g_w, to TM_D.  The A operand of a
// compose is announced a K-slice at a time on a_go.
__device__ void epilogue_role_seam(Misc* ms, uint8_t* smem, const CtArgs& a, uint32_t tmem, uint32_t gj, uint32_t gu,
                                   int c0, int len, int lh, int64_t obj, int q, int lane) {
    const int n = 32 * q + lane;
    const int LH = a.n_layers * a.n_heads;
    const uint32_t tl = tmem + ((32u * q) << 16);
    float* out = a.S_out + obj * kD * kD;
    const float* s0 = a.S0 ? a.S0 + obj * kD * kD : nullptr;
    if (len == 0) {
        for (int i = 0; i < kD; ++i) out[i * kD + n] = s0 ? s0[i * kD + n] : 0.f;
        return;
    }
    int tb;
    const bool seam0 = step_units(a, c0, tb) > 0;
    float gw = 0.f;
    if (seam0) {
        if (!wg_all(4, wait_bar(&ms->seam_ready, gu & 1, ms, a))) return;
        gw = ms->g[kU - 1];
    }
#pragma unroll 1
    for (int cb = 0; cb < 4; ++cb) {  // the start state, split hi/lo (and g_w S0 before a seam)
        uint32_t x[32];
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) x[jj] = __float_as_uint(s0 ? s0[(32 * cb + jj) * kD + n] : 0.f);
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
            uint32_t h[16], l[16];
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) split_tf32(__uint_as_float(x[16 * hb + jj]), h[jj], l[jj]);
            tmem_st16(tl + TM_AB + 32 * cb + 16 * hb, h);
            tmem_st16(tl + TM_AS + 32 * cb + 16 * hb, l);
        }
        if (seam0) {
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) x[jj] = __float_as_uint(gw * __uint_as_float(x[jj]));
            tmem_st32(tl + TM_D + 32 * cb, x);
        }
        warp_arrive(seam0 ? &ms->r_go[cb] : &ms->a_go[cb], lane);
    }
    if (seam0 && !apply_step_units(ms, a, tl, lh, c0, gu, n)) return;
    const float* sp = reinterpret_cast<const float*>(smem + OFF_SP) + (n >> 5) * (kSliceBytes / 4) + (n & 31);
    for (int j = 0; j < len; ++j) {
        const uint32_t g = gj + j;
        const int p = a.seg_idx[c0 + j];
        const int e = a.T_exp ? a.T_exp[p * LH + lh] : 0;
        const bool last = j + 1 == len;
        const bool seam = !last && step_units(a, c0 + j + 1, tb) > 0;
        bool ok = wait_bar(&ms->d_done, g & 1, ms, a);
        ok = ok && wait_bar(&ms->sp_full, g & 1, ms, a);
        ok = ok && (!seam || wait_bar(&ms->seam_ready, gu & 1, ms, a));
        if (!wg_all(4, ok)) return;
        tc_fence_after();
        gw = seam ? ms->g[kU - 1] : 0.f;
        // 2^e as two factors (each exact for |e| <= 252): T~ S 2^e underflows
        // only where it is negligible against S_p
        const float f1 = exp2f((float)(e / 2)), f2 = exp2f((float)(e - e / 2));
#pragma unroll 1
        for (int cb = 0; cb < 4; ++cb) {
            uint32_t x[32];
            tmem_ld32(tl + TM_D + 32 * cb, x);
            float spv[32];  // (all loaded before any store: the stores to out could alias them)
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) spv[jj] = sp[(32 * cb + jj) * 32];
            tmem_wait_ld();
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) x[jj] = __float_as_uint(fmaf(__uint_as_float(x[jj]) * f1, f2, spv[jj]));
            if (last) {
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) out[(32 * cb + jj) * kD + n] = __uint_as_float(x[jj]);
            }
            if (!last) {
#pragma unroll
                for (int hb = 0; hb < 2; ++hb) {
                    uint32_t h[16], l[16];
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) split_tf32(__uint_as_float(x[16 * hb + jj]), h[jj], l[jj]);
                    tmem_st16(tl + TM_AB + 32 * cb + 16 * hb, h);
                    tmem_st16(tl + TM_AS + 32 * cb + 16 * hb, l);
                }
            }
            if (seam) {
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) x[jj] = __float_as_uint(gw * __uint_as_float(x[jj]));
                tmem_st32(tl + TM_D + 32 * cb, x);
                warp_arrive(&ms->r_go[cb], lane);
            }
        }
        tmem_wait_st();
        if (!last && !seam)  // all of TM_D has been read: the next compose may overwrite it
            for (int cb = 0; cb < 4; ++cb) warp_arrive(&ms->a_go[cb], lane);
        named_sync(4);
        if (n == 0) mbar_arrive(&ms->sp_empty);  // S_p has been read
        if (seam && !apply_step_units(ms, a, tl, lh, c0 + j + 1, gu, n)) return;
    }
}

// Chain-transition epilogue: the state is T_chain, from I, and each step
// leaves T_p T_chain in TM_D.  The stored state is kept near unit size by a
// power of two: step j divides by 2^s_j with s_j the exponent of the largest
// entry of the previous stored state (1 for I), so the stored entries stay
// within a factor of about |T~_p| of 1, and T_chain = stored * 2^texp with
// texp += e_p + s_j.  That takes one pass over the accumulator (scale, the
// next maximum, the split into the next A, announced a K-slice at a time once
// all of TM_D has been read).  The last step instead scales by the exponent
// of its own maximum, so that T_out's largest entry lies in [1, 2), and writes
// T_out and T_exp_out.  Thread n owns column n; the four warps' maxima meet in
// shared memory.
__device__ void epilogue_role_T(Misc* ms, const CtArgs& a, uint32_t tmem, uint32_t gj, int c0, int len, int lh,
                                int64_t obj, int q, int lane) {
    const int n = 32 * q + lane;
    const int LH = a.n_layers * a.n_heads;
    const uint32_t tl = tmem + ((32u * q) << 16);
    float* out = a.T_out + obj * kD * kD;
    if (len == 0) {  // empty chain: the identity
        for (int i = 0; i < kD; ++i) out[i * kD + n] = i == n ? 1.f : 0.f;
        if (n == 0) a.T_exp_out[obj] = 0;
        return;
    }
#pragma unroll 1
    for (int cb = 0; cb < 4; ++cb) {  // A for the first step: I (column n = e_n; the lo part is 0)
        uint32_t h[32], l[32];
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
            h[jj] = 32 * cb + jj == n ? 0x3f800000u : 0u;
            l[jj] = 0u;
        }
        tmem_st32(tl + TM_AB + 32 * cb, h);
        tmem_st32(tl + TM_AS + 32 * cb, l);
        warp_arrive(&ms->a_go[cb], lane);
    }
    int texp = 0, shift = 0;  // shift: exponent of the stored state's largest entry
    for (int j = 0; j < len; ++j) {
        const uint32_t g = gj + j;
        const int p = a.seg_idx[c0 + j];
        const int e = a.T_exp ? a.T_exp[p * LH + lh] : 0;
        if (!wg_all(4, wait_bar(&ms->d_done, g & 1, ms, a))) return;
        tc_fence_after();
        float m = 0.f;
        if (j + 1 == len) {  // the exact maximum, then T_out with its largest entry in [1, 2)
#pragma unroll 1
            for (int cb = 0; cb < 4; ++cb) {
                uint32_t x[32];
                tmem_ld32(tl + TM_D + 32 * cb, x);
                tmem_wait_ld();
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) m = fmaxf(m, fabsf(__uint_as_float(x[jj])));
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
            if (lane == 0) ms->red[q] = m;
            named_sync(4);
            m = fmaxf(fmaxf(ms->red[0], ms->red[1]), fmaxf(ms->red[2], ms->red[3]));
            const int er = (m > 0.f && m < INFINITY) ? ilogbf(m) : 0;
            const float sc = ldexpf(1.f, -er);
            texp += e + er;
#pragma unroll 1
            for (int cb = 0; cb < 4; ++cb) {
                uint32_t x[32];
                tmem_ld32(tl + TM_D + 32 * cb, x);
                tmem_wait_ld();
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) out[(32 * cb + jj) * kD + n] = __uint_as_float(x[jj]) * sc;
            }
            break;
        }
        const float sc = ldexpf(1.f, -shift);
        texp += e + shift;
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {  // two K-slices at a time
            uint32_t x[2][32];
            tmem_ld32(tl + TM_D + 64 * half, x[0]);
            tmem_ld32(tl + TM_D + 64 * half + 32, x[1]);
            tmem_wait_ld();
            if (half == 1) {  // all of TM_D has been read
                warp_arrive(&ms->a_go[0], lane);
                warp_arrive(&ms->a_go[1], lane);
            }
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const int cb = 2 * half + c;
                uint32_t h[32], l[32];
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) {
                    const float y = __uint_as_float(x[c][jj]) * sc;
                    m = fmaxf(m, fabsf(y));
                    split_tf32(y, h[jj], l[jj]);
                }
                tmem_st32(tl + TM_AB + 32 * cb, h);
                tmem_st32(tl + TM_AS + 32 * cb, l);
                if (half == 1) warp_arrive(&ms->a_go[cb], lane);
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0) ms->red[q] = m;
        named_sync(4);  // (the next step's first barrier orders these reads before the next writes)
        m = fmaxf(fmaxf(ms->red[0], ms->red[1]), fmaxf(ms->red[2], ms->red[3]));
        shift = (m > 0.f && m < INFINITY) ? ilogbf(m) : 0;
    }
    if (n == 0) a.T_exp_out[obj] = texp;
}

// ---------------------------------------------------------------- kernel --
// kSeam: the fused reuse chain; kTrans: each chain's own transition instead of its state.
template <bool kSeam, bool kTrans>
__global__ void __launch_bounds__(kThreads, 1)
    compose_tc_kernel(const __grid_constant__ CUtensorMap tmT, const __grid_constant__ CUtensorMap tmS, const CtArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    Misc* ms = reinterpret_cast<Misc*>(smem + OFF_MISC);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if ((smem_u32(smem) & 1023u) != 0) {
        if (tid == 0) set_error(a.err, kErrBadIndex);
        return;
    }
    if (tid == 0) {
        for (int b = 0; b < kRing; ++b) {
            mbar_init(&ms->full[b], 1);
            mbar_init(&ms->cvt[b], 1);
            mbar_init(&ms->empty[b], 1);
        }
        mbar_init(&ms->sp_full, 1);
        mbar_init(&ms->sp_empty, 1);
        mbar_init(&ms->d_done, 1);
        mbar_init(&ms->drain, 1);
        mbar_init(&ms->seam_ready, 1);
        mbar_init(&ms->seam_free, 1);
        for (int b = 0; b < kSlices; ++b) {
            mbar_init(&ms->a_go[b], 4);
            mbar_init(&ms->r_go[b], 4);
        }
        mbar_init(&ms->r_done, 1);
        mbar_init(&ms->c_go, 1);
        mbar_init(&ms->u_done, 1);
        ms->abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kWarpTMA && lane == 0) {
        tma_prefetch_desc(&tmT);
        tma_prefetch_desc(&tmS);
    }
    if (warp == kWarpMMA) tmem_alloc(&ms->tmem_base, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ms->tmem_base;
    const int LH = a.n_layers * a.n_heads;
    uint32_t gs = 0, gj = 0, gu = 0;
    for (int item = blockIdx.x; item < a.n_items; item += gridDim.x) {
        if (*(volatile int*)&ms->abort_flag) break;
        const int lh = item / a.n_chains, chain = item % a.n_chains;
        const int c0 = a.cu_chain[chain], len = a.cu_chain[chain + 1] - c0;
        const int64_t obj = (int64_t)chain * LH + lh;
        if (warp == kWarpTMA) {
            if (lane == 0) producer_role(ms, smem, a, &tmT, &tmS, gs, gj, c0, len, lh, !kTrans);
        } else if (warp == kWarpMMA) {
            if (lane == 0) mma_role<kSeam, kTrans>(ms, smem, a, tmem, gs, gj, gu, c0, len);
        } else if (warp < kWarpEpi0) {
            convert_role<kSeam>(ms, smem, a, tmem, gs, gu, c0, len, lh, tid - 32 * kWarpCvt0);
        } else if (kSeam) {
            epilogue_role_seam(ms, smem, a, tmem, gj, gu, c0, len, lh, obj, warp & 3, lane);
        } else if (kTrans) {
            epilogue_role_T(ms, a, tmem, gj, c0, len, lh, obj, warp & 3, lane);
        } else {
            epilogue_role(ms, smem, a, tmem, gj, c0, len, lh, obj, warp & 3, lane);
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        gs += kSlices * len;
        gj += len;
        if (kSeam)
            for (int j = 0; j < len; ++j) {
                int tb;
                gu += step_units(a, c0 + j, tb);
            }
    }
    if (warp == kWarpMMA) {
        if (lane == 0) {
            // every MMA has completed before tensor memory is freed; a drain that runs out of polls is
            // reported (the result is then not to be trusted) and the memory freed all the same
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
    if (warp == kWarpMMA) tmem_dealloc(tmem, 512);
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
    static std::mutex mu;
    static int cache[128] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return 0;
    std::lock_guard<std::mutex> lk(mu);
    if (!cache[dev]) cudaDeviceGetAttribute(&cache[dev], cudaDevAttrMultiProcessorCount, dev);
    return cache[dev];
}

// A table [rows][128] fp32 as a 2-D tensor; box = 32 columns x 128 rows.
bool make_map(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap* m, const float* base, uint64_t rows, bool swz) {
    cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)kD * 4};
    cuuint32_t box[2] = {32, (cuuint32_t)kD}, es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swz ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool compose_tc_supported(const ComposeParams& p) {
    return (p.family == kGDN || p.family == kKDA) && p.dk == kD && p.dv == kD && p.n_pairs > 0 &&
           (int64_t)p.n_pairs * p.n_layers * p.n_heads * kD < INT32_MAX && encode_fn() != nullptr;
}

namespace {

template <bool kSeam, bool kTrans = false>
cudaError_t launch_tc(const ComposeParams& p, CtArgs a, cudaStream_t s) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    const uint64_t rows = (uint64_t)p.n_pairs * p.n_layers * p.n_heads * kD;
    CUtensorMap tT, tS;
    if (!make_map(enc, &tT, p.T_tab, rows, true) || !make_map(enc, &tS, p.S_tab, rows, false))
        return cudaErrorInvalidValue;
    a.n_layers = p.n_layers;
    a.n_heads = p.n_heads;
    a.n_pairs = p.n_pairs;
    a.n_chains = p.n_chains;
    a.n_items = p.n_chains * p.n_layers * p.n_heads;
    a.T_exp = p.T_exp_tab;
    a.cu_chain = p.cu_chain;
    a.seg_idx = p.seg_idx;
    a.S0 = p.S0;
    a.S_out = p.S_out;
    a.T_out = p.T_out;
    a.T_exp_out = p.T_exp_out;
    a.counter = nullptr;
    a.wait_limit = 1u << 26;
    if (a.n_items == 0) return cudaSuccess;
    const int sms = sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    cudaError_t e = cudaFuncSetAttribute(compose_tc_kernel<kSeam, kTrans>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    const int grid = a.n_items < sms ? a.n_items : sms;
    compose_tc_kernel<kSeam, kTrans><<<grid, kThreads, kSmemBytes, s>>>(tT, tS, a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_compose_tc(const ComposeParams& p, unsigned* err, cudaStream_t s) {
    CtArgs a = {};
    a.err = err;
    cudaError_t e = launch_tc<false>(p, a, s);
    if (e == cudaSuccess && p.T_out) e = launch_tc<false, true>(p, a, s);  // each chain's own transition
    return e;
}

bool chain_tc_supported(const ChainParams& p) {  // (the fused seam units run the GDN recurrence)
    return p.c.family == kGDN && compose_tc_supported(p.c) && p.c.n_pairs > 0;
}

cudaError_t launch_chain_tc(const ChainParams& p, unsigned* err, cudaStream_t s) {
    CtArgs a = {};
    a.err = err;
    a.in_bf16 = p.in_dtype == kBF16;
    a.n_tokens = p.n_tokens;
    a.cu_step = p.cu_step;
    a.q = p.q;
    a.k = p.k;
    a.v = p.v;
    a.alpha = p.alpha;
    a.beta = p.beta;
    a.o_out = p.o_out;
    return launch_tc<true>(p.c, a, s);
}

}  // namespace hypic
