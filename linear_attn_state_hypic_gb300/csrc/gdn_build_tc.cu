// gdn_build_tc.cu -- chunked GDN build of the cached pair (T_C, S(C|0)) on the
// sm_103a tensor cores (d = 128, bf16 keys/values).
//
// What it computes: for a segment C and a head, T_C = A_L ... A_1 with the
// gated-delta transition A_t = a_t (I - b_t k_t k_t^T), and S(C|0), the state
// after C from zero with the write term b_t k_t v_t^T (aibase article on
// HYPIC, paragraph on the linear layers: the cached pair of a segment).
//
// How: tokens are taken in chunks of 64.  The scalar gate a_t commutes with
// the delta projection, so the chunk's UT transform needs no decay at all:
// with A^[i][j] = b_i k_i.k_j for j < i, M = (I + A^)^-1, g_t = a_1 ... a_t
// inside the chunk and g_C its last value,
//     W^ = M Diag(b) K,   U^ = M Diag(b / g) V,
//     T <- g_C (I - K^T W^) T,   S <- g_C (S + K^T (U^ - W^ S)),
// which is the token recurrence applied 64 times (WY form of a product of
// generalised Householder transitions; the decay reaches S only through the
// per-token weights 1/g_t of the values).  The state is held transposed in
// tensor memory, D'' = [T^T ; S^T] scaled per half (256 x 128 fp32): the T
// half carries no decay (its exponent is kept apart), the S half a lazy
// power-of-two scale 2^lsS set from the gates alone.  Per chunk:
//   gram    G = K K^T                              bf16 MMA, M=64  N=64  K=128
//   solve   M from G and b                         CUDA cores + warp MMAs (block-triangular inverse)
//   W^T     -(M Diag(b) K)^T                       bf16 MMA, M=128 N=64  K=64, twice (M form as hi + lo)
//   U~      V^T (M Diag(b uf))^T into X_S          bf16 MMA, M=128 N=64  K=64 (uf = 2^(-lg2 g_t - lsS))
//   convert W^T -> tf32 operand in shared memory   (CUDA cores)
//   GEMM1   X_h (+)= D''_h (-W^)^T                 tf32 MMA, A read from tensor memory
//   pass    X_T -> bf16 hi + lo, X_S -> bf16       in place (a format conversion, nothing else)
//   GEMM2   D''_h += X_h K                         bf16 MMA, M=128 N=128 K=64 (twice for T: hi, lo),
//                                                  A read from tensor memory
// A renormalisation chunk (every 16 chunks, the last chunk of a segment, and
// chunks whose decay would push the S scale past 2^-112) first rescales the
// stored state: T by a power of two to a maximum below 2, S to its true scale
// times g_C, so that the chunk ends with S at its true scale.  The largest U~
// factor of an ordinary chunk is then below 2^112, and that of a
// renormalisation chunk below 1.
// T_C falls far below the fp32 range over long segments: it is returned as a
// mantissa and a power-of-two exponent.
//
// Roles (512 threads): warp 0 loads keys and values (TMA), writes the gate
// tables and plans each chunk's scales; three single-thread MMA issuers (a
// thread sends a small MMA only about every 60 cycles): warp 1 the prep
// stream (gram, W^T), warp 2 the S half (U~, GEMM1, GEMM2), warp 3 the T half
// (GEMM1, GEMM2); warps 4-11 (prep) turn each gram into the M forms; warps
// 12-15 (state) run the passes, convert W^ into the tf32 operand, renormalise
// and write the result.  Per chunk the state stream is serial (GEMM1, passes,
// W operand, GEMM2); the prep runs up to two chunks ahead.  The roles meet on
// mbarriers; every wait is bounded and a wait that runs out sets the device
// error word.
// One CTA per SM, persistent over (segment, layer, head) items taken from an
// atomic queue in longest-body-first order.  Warp 0 publishes them through a
// ring of item slots and each role runs through them at its own pace, so one
// item's first chunks overlap the previous item's last ones.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <float.h>
#include <stddef.h>
#include <stdint.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace hypic {
namespace {

using namespace tc;

constexpr int kD = 128;           // dk = dv
constexpr int kC = 64;            // chunk length
constexpr int kKStages = 4;       // key tiles in flight (from the gram, issued early, to GEMM2)
constexpr int kVStages = 2;
constexpr int kGateSlots = 4;     // per-chunk gate tables in flight
constexpr int kThreads = 512;
constexpr int kWarpTMA = 0, kWarpIssP = 1, kWarpIssS = 2, kWarpIssT = 3, kWarpPrep0 = 4, kWarpState0 = 12;
constexpr int kPrepThreads = 256;  // warps 4-11: two warps per tensor-memory lane quarter

// Shared memory map (byte offsets; every operand region is 1024-byte aligned).
constexpr uint32_t kTile = 16384;                        // 64 tokens x 128 (b)f16, two 64-column TMA boxes
constexpr uint32_t OFF_K = 0;                            // bf16 key ring
constexpr uint32_t OFF_V = OFF_K + kKStages * kTile;     // value ring
constexpr uint32_t kWBytes = 32768;                      // -W^: tf32 [64 t][128 i], K-major, 4 blocks of 32 i
constexpr uint32_t OFF_W = OFF_V + kVStages * kTile;     // one: rewritten only after both GEMM1s that read it
constexpr uint32_t kBT = 24576;                          // -M Diag(b) hi, lo, then M Diag(b uf): bf16 [64][64]
constexpr uint32_t OFF_BT = OFF_W + kWBytes;             // two of them: chunk gc uses buffer gc % 2
constexpr uint32_t OFF_AS = OFF_BT + 2 * kBT;            // A^ / M: fp32 [64][kAS] (padded rows)
constexpr int kAS = 68;
constexpr uint32_t OFF_PT = OFF_AS + ((64 * kAS * 4 + 1023) / 1024) * 1024;  // solve scratch: 32 x 36 fp32
constexpr uint32_t OFF_MISC = OFF_PT + 5120;

// An item of the queue as the producer publishes it to the other roles.
struct ItemSlot {
    int64_t b0, b1, obj;  // body [b0, b1) in the token index, output object
    uint32_t g;           // CTA-wide index of the item's first chunk
    int nc, layer, head;  // nc > 0, or nc < 0: the queue is exhausted
};
constexpr int kItemSlots = 4;
constexpr int kSlotReaders = 5;  // the three issuers, the prep warps, the state warps

// The scales of one chunk, planned by the producer from the gates.
struct ChunkPlan {
    float preS;    // renormalisation chunk: D''_S <- 2^preS D''_S first
    float sum_lc;  // log2 of the item's decay up to and including this chunk
    int rn;        // renormalisation chunk
    int pad;
};

struct Misc {
    uint64_t fullK[kKStages], emptyK[kKStages];  // emptyK: one commit from each half's issuer after its GEMM2
    uint64_t fullV[kVStages], emptyV[kVStages];
    uint64_t gready[kGateSlots];  // producer -> prep, state: gate tables and plan of a chunk written
    uint64_t g_done, g_read;        // gram committed; gram read by the prep warps
    // M forms of chunk gc written (that_ready[gc % 2]); the W^T and U~ MMAs that read them are done
    // (bt_free[gc % 2], one commit from each issuer).
    uint64_t that_ready[2], bt_free[2];
    // W^T committed; read from tensor memory; the tf32 operand of chunk gc written (w_cvt[gc % 2]: the
    // operand of chunk gc + 1 may be written before the issuer of one half has waited for that of chunk
    // gc, so consecutive chunks signal on different barriers)
    uint64_t w_done, w_read, w_cvt[2];
    uint64_t pre_done;               // state ready for GEMM1 (initialised or renormalised)
    uint64_t x_done_s, x_done_t;     // GEMM1 of the S / T half committed
    uint64_t y_ready_s, y_ready_t;   // pass of the S / T half done
    uint64_t d_ready_s, d_ready_t;   // GEMM2 of the S / T half committed
    uint64_t drain;
    alignas(16) float beta[kGateSlots][kC];
    alignas(16) float uf[kGateSlots][kC];  // 2^(-lg2 g_t - lsS): the U~ weight of token t
    ChunkPlan plan[kGateSlots];
    float red[4];
    uint64_t slot_full[kItemSlots], slot_read[kItemSlots];  // item slot written / copied by every reader
    ItemSlot slots[kItemSlots];
    int abort_flag;
    uint32_t tmem_base;
};
constexpr uint32_t kSmemBytes = OFF_MISC + sizeof(Misc);
static_assert(OFF_MISC % 16 == 0 && offsetof(Misc, beta) % 16 == 0 && offsetof(Misc, uf) % 16 == 0,
              "float4 accesses of the gate tables need 16-byte alignment");
static_assert(kSmemBytes <= 232448, "shared memory budget");

// Tensor-memory columns.
constexpr uint32_t TM_DT = 0, TM_DS = 128, TM_XT = 256, TM_XS = 320, TM_G = 384, TM_W = 448;

constexpr uint32_t kFmtBF16 = 1, kFmtTF32 = 2;
constexpr uint32_t ID_GRAM = idesc(kFmtBF16, 64, 64, false, false);   // G = K K^T
constexpr uint32_t ID_W = idesc(kFmtBF16, 128, 64, true, false);      // W^T: A = K^T (MN-major)
constexpr uint32_t ID_U = idesc(kFmtBF16, 128, 64, true, false);      // U~: A = V^T (MN-major)
constexpr uint32_t ID_G1 = idesc(kFmtTF32, 128, 64, false, false);    // X = D'' W^T (A in TMEM)
constexpr uint32_t ID_G2T = idesc(kFmtBF16, 128, 128, false, true);   // D''_T += X_T K (B = K, MN-major)
constexpr uint32_t ID_G2S = idesc(kFmtBF16, 128, 128, false, true);   // D''_S += X_S K

struct TcArgs {
    int n_layers, n_heads, n_seg, n_items;
    int64_t n_tokens;
    const int32_t* cu;
    const int32_t* skip;
    const float* alpha;
    const float* beta;
    float* T_out;
    int32_t* T_exp;
    float* S_out;
    const int32_t* order;
    unsigned* counter;
    unsigned* err;
    uint32_t wait_limit;  // polls of the final drain
    uint64_t wait_ns;     // time limit of every other wait
};


// Bounded wait shared by all roles: the waiting warp sleeps until the phase
// completes (re-polling at least every few microseconds); it gives up, and
// raises the CTA's abort flag and the device error word, once `wait_ns` of
// GPU time have passed, or at once when another role already gave up.
// (The slow path is a call: one copy of it instead of one per wait keeps the
// kernel's code, which every role's warps share in the instruction cache,
// small.)
__device__ __noinline__ bool wait_bar_slow(uint64_t* bar, uint32_t parity, int* abort_flag, uint64_t wait_ns,
                                           unsigned* err) {
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
#pragma unroll 1
        for (int j = 0; j < 16; ++j)
            if (mbar_try_wait_sleep(bar, parity, 4000u)) return true;
        if (*(volatile int*)abort_flag) return false;
        if (globaltimer_ns() - t0 > wait_ns) break;
    }
    *(volatile int*)abort_flag = 1;
    set_error(err, kErrTimeout);
    return false;
}
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, Misc* ms, const TcArgs& a) {
    if (mbar_try_wait(bar, parity)) return true;
    return wait_bar_slow(bar, parity, &ms->abort_flag, a.wait_ns, a.err);
}
__device__ __forceinline__ void named_sync(int id, int n = 128) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}
// Two values as bf16 pairs x = hi + lo: hi is x with its 16 low bits cleared
// (exact; two values packed by one byte permute), lo = x - hi (exact in fp32)
// rounded to bf16, so hi + lo keeps about 16 significant bits of x.
__device__ __forceinline__ void split_bf16(float x, float y, uint32_t& hi, uint32_t& lo) {
    const uint32_t hx = __float_as_uint(x) & 0xffff0000u, hy = __float_as_uint(y) & 0xffff0000u;
    hi = __byte_perm(hx, hy, 0x7632);
    lo = pack_bf16(x - __uint_as_float(hx), y - __uint_as_float(hy));
}
// x rounded to tf32 (nearest, ties away from zero) by integer arithmetic on
// its bits: add half a tf32 unit of the last place, then clear the 13 low bits.
__device__ __forceinline__ float tf32_round(float x) {
    return __uint_as_float((__float_as_uint(x) + 0x1000u) & 0xffffe000u);
}

// ------------------------------------------------------------ producer --

// Raw gates of tokens t0 + 2 lane + {0, 1} (a = 1, b = 0 past the body end:
// an identity transition, so padded rows leave the result unchanged).
__device__ __forceinline__ void gate_load(const TcArgs& a, int layer, int head, int64_t t0, int64_t t_end, int lane,
                                          float (&ra)[2], float (&rb)[2]) {
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const int64_t t = t0 + 2 * lane + u;
        ra[u] = 1.f;
        rb[u] = 0.f;
        if (t < t_end) {
            const int64_t row = tok_row(layer, t, head, a.n_tokens, a.n_heads);
            ra[u] = a.alpha[row];
            rb[u] = a.beta[row];
        }
    }
}

// The producer's running scale state of an item (identical in every lane).
struct PlanState {
    float lsS;     // log2 of the stored S scale before the next chunk
    float sum_lc;  // log2 of the decay so far
    int since;     // chunks since the last renormalisation
};
constexpr int kRenormEvery = 16;
constexpr float kLazyMax = 56.f;  // (the stored S stays below 2^112 times the true one)

// Gate tables and plan of one chunk (one warp, two tokens a lane): b_t, the
// U~ weight uf_t = 2^(-lg2 g_t - lsS) (g_t the inclusive in-chunk decay), and
// the chunk's plan.  A renormalisation chunk first brings the stored S to
// its true scale times g_C (preS = lsS + lg2 g_C) and then takes the weights
// g_C / g_t <= 1, so that it ends at the true scale (lsS = 0); an ordinary
// chunk keeps the decay in the scale (lsS += lg2 g_C).
__device__ void gate_tables(Misc* ms, int slot, const float (&ra)[2], const float (&rb)[2], bool last,
                            PlanState& st, int lane) {
    const float l0 = log2f(fmaxf(ra[0], FLT_MIN)), l1 = log2f(fmaxf(ra[1], FLT_MIN));
    float s = l0 + l1;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, s, off);
        if (lane >= off) s += y;
    }
    const float before = __shfl_up_sync(0xffffffffu, s, 1);
    const float e0 = (lane > 0 ? before : 0.f) + l0, e1 = e0 + l1;
    const float lc = __shfl_sync(0xffffffffu, e1, 31);
    const bool rn = last || st.since + 1 >= kRenormEvery || st.lsS + lc < -2.f * kLazyMax || lc < -kLazyMax;
    float ls_use, preS = 0.f;
    if (rn) {
        preS = st.lsS + lc;
        ls_use = -lc;
        st.lsS = 0.f;
        st.since = 0;
    } else {
        ls_use = st.lsS;
        st.lsS += lc;
        ++st.since;
    }
    st.sum_lc += lc;
    const int t = 2 * lane;
    auto ex = [](float x) { return exp2f(fminf(fmaxf(x, -126.f), 126.f)); };
    *reinterpret_cast<float2*>(&ms->beta[slot][t]) = make_float2(rb[0], rb[1]);
    *reinterpret_cast<float2*>(&ms->uf[slot][t]) = make_float2(ex(-e0 - ls_use), ex(-e1 - ls_use));
    if (lane == 0) {
        ChunkPlan& p = ms->plan[slot];
        p.preS = preS;
        p.sum_lc = st.sum_lc;
        p.rn = rn ? 1 : 0;
    }
}

// Warp 0: keys (ring) and values (ring) by TMA from lane 0, and the gate
// tables of each chunk from the whole warp (the loads of the next chunk's
// gates in flight meanwhile).
__device__ void producer_role(Misc* ms, uint8_t* smem, const TcArgs& a, const CUtensorMap* tmk,
                              const CUtensorMap* tmv, uint32_t g, int nc, int layer, int head, int64_t b0, int64_t b1,
                              int lane) {
    float ra[2], rb[2];
    PlanState st{0.f, 0.f, 0};
    gate_load(a, layer, head, b0, b1, lane, ra, rb);
    for (int c = 0; c < nc; ++c) {
        const uint32_t gc = g + c, s = gc % kKStages, u = gc / kKStages;
        const int z = (int)((int64_t)layer * a.n_tokens + b0 + (int64_t)c * kC);
        if (u >= 1 && !wait_bar(&ms->emptyK[s], (u - 1) & 1, ms, a)) return;
        if (lane == 0) {
            uint8_t* kt = smem + OFF_K + s * kTile;
            mbar_expect_tx(&ms->fullK[s], kTile);
            tma_load_3d(kt, tmk, &ms->fullK[s], 0, head, z);
            tma_load_3d(kt + 8192, tmk, &ms->fullK[s], 64, head, z);
        }
        // The slot of chunk gc was last read for chunk gc - 4: by the prep before its M forms, by the
        // state warps at the start of that chunk, both before GEMM2 of chunk gc - 4 (waited above).
        gate_tables(ms, gc % kGateSlots, ra, rb, c + 1 == nc, st, lane);
        if (c + 1 < nc) gate_load(a, layer, head, b0 + (int64_t)(c + 1) * kC, b1, lane, ra, rb);
        __syncwarp();
        if (lane == 0) mbar_arrive(&ms->gready[gc % kGateSlots]);
        const uint32_t vs = gc % kVStages, vu = gc / kVStages;
        if (vu >= 1 && !wait_bar(&ms->emptyV[vs], (vu - 1) & 1, ms, a)) return;
        if (lane == 0) {
            uint8_t* vt = smem + OFF_V + vs * kTile;
            mbar_expect_tx(&ms->fullV[vs], kTile);
            tma_load_3d(vt, tmv, &ms->fullV[vs], 0, head, z);
            tma_load_3d(vt + 8192, tmv, &ms->fullV[vs], 64, head, z);
        }
    }
}

// ----------------------------------------------------------- prep roles --
// p: thread index inside the prep warps (0..255); q: its tensor-memory lane
// quarter; lane: lane in the warp.

// Rows of A^ from the gram matrix in tensor memory (M=64 accumulator layout:
// row 16q + l sits in lane 32q + l, l < 16): A^[r][j] = b_r G[r][j] for
// j < r, 0 elsewhere.  Half h of the prep warps reads columns 32h..32h+31;
// lane l < 16 writes the first 16 of them in its row, lane l + 16, which holds
// no row, takes the other 16 of the same row from lane l by a shuffle.
__device__ void prep_arows(const Misc* ms, float* As, int slot, uint32_t tmem, int q, int h, int lane) {
    uint32_t g0[32];
    tmem_ld32(tmem + ((32u * q) << 16) + TM_G + 32 * h, g0);
    tmem_wait_ld();
    const bool upper = lane >= 16;
    uint32_t gv[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const uint32_t x = __shfl_xor_sync(0xffffffffu, g0[16 + j], 16);
        gv[j] = upper ? x : g0[j];
    }
    const int r = 16 * q + (lane & 15), cb = 32 * h + (upper ? 16 : 0);
    const float coef = ms->beta[slot][r];
    float* row = As + r * kAS + cb;
#pragma unroll
    for (int j = 0; j < 16; j += 4) {
        float4 v;
        v.x = (cb + j < r) ? coef * __uint_as_float(gv[j]) : 0.f;
        v.y = (cb + j + 1 < r) ? coef * __uint_as_float(gv[j + 1]) : 0.f;
        v.z = (cb + j + 2 < r) ? coef * __uint_as_float(gv[j + 2]) : 0.f;
        v.w = (cb + j + 3 < r) ? coef * __uint_as_float(gv[j + 3]) : 0.f;
        *reinterpret_cast<float4*>(row + j) = v;
    }
}

// Warp-level block products for the solve (mma.sync m16n8k8 on tf32
// operands with fp32 accumulation: the tensor cores read the fp32 values'
// upper 19 bits).  M is only needed to about tf32 precision -- the W^ it
// forms is rounded to tf32 for GEMM1 -- and products of truncated operands
// leave T_C and S where products to ~16 bits put them.
__device__ __forceinline__ void mma1688(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                        uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// C (16 x 8NT) = A (16 x 16KS, row stride lda) B (16KS x 8NT, row stride
// ldb), one warp; lane (g, t) = (lane / 4, lane % 4) holds A[g][t], A[g+8][t],
// A[g][t+4], A[g+8][t+4] and B[t][g], B[t+4][g] of each 8-wide k step, and
// rows g, g + 8, columns 2t, 2t + 1 of each 8-column tile of C.  Two
// accumulator sets alternate over the k steps (no chain through one).
template <int KS, int NT>
__device__ __forceinline__ void warp_gemm(float (&c)[NT][4], const float* A, int lda, const float* B, int ldb,
                                          int lane) {
    const int g = lane >> 2, t = lane & 3;
    float c1[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) c[nt][e] = c1[nt][e] = 0.f;
#pragma unroll
    for (int ks = 0; ks < 2 * KS; ++ks) {
        const float* a0 = A + g * lda + 8 * ks + t;
        const uint32_t x0 = __float_as_uint(a0[0]), x1 = __float_as_uint(a0[8 * lda]);
        const uint32_t x2 = __float_as_uint(a0[4]), x3 = __float_as_uint(a0[8 * lda + 4]);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const float* b = B + (8 * ks + t) * ldb + 8 * nt + g;
            const uint32_t y0 = __float_as_uint(b[0]), y1 = __float_as_uint(b[4 * ldb]);
            if (ks & 1) mma1688(c1[nt], x0, x1, x2, x3, y0, y1);
            else mma1688(c[nt], x0, x1, x2, x3, y0, y1);
        }
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) c[nt][e] += c1[nt][e];
}
template <int NT>
__device__ __forceinline__ void warp_store(const float (&c)[NT][4], float* D, int ldd, float sgn, int lane) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        *reinterpret_cast<float2*>(D + g * ldd + 8 * nt + 2 * t) = make_float2(sgn * c[nt][0], sgn * c[nt][1]);
        *reinterpret_cast<float2*>(D + (g + 8) * ldd + 8 * nt + 2 * t) = make_float2(sgn * c[nt][2], sgn * c[nt][3]);
    }
}

// The operand forms of M, K-major 64 x 64 bf16 (128-byte rows, 128-byte
// swizzle): -M Diag(b) as a hi + lo pair at bt and bt + 8192 (the W^T
// product, to about 16 bits; negated so that GEMM1 yields -X), and M Diag(b uf)
// at bt + 16384 (the U~ product).  Each block of M is written by the solve
// level that finishes it; the blocks above the diagonal are zero in every
// chunk and are written once, when the kernel starts.
__device__ __forceinline__ uint32_t form_off(int r, int j) {
    return (uint32_t)r * 128u + ((uint32_t)((j >> 3) ^ (r & 7)) << 4) + (uint32_t)(j & 7) * 2u;
}
// Elements (r, j) and (r, j + 1), j even.
__device__ __forceinline__ void form_write2(uint8_t* bt, int r, int j, float m0, float m1, const float* beta,
                                            const float* uf) {
    const float mv0 = m0 * beta[j], mv1 = m1 * beta[j + 1];
    uint32_t hi, lo;
    split_bf16(-mv0, -mv1, hi, lo);
    const uint32_t off = form_off(r, j);
    *reinterpret_cast<uint32_t*>(bt + off) = hi;
    *reinterpret_cast<uint32_t*>(bt + 8192 + off) = lo;
    *reinterpret_cast<uint32_t*>(bt + 16384 + off) = pack_bf16(mv0 * uf[j], mv1 * uf[j + 1]);
}
// A 16 x 8 tile of M from a warp_gemm fragment times sgn, rows r0.., columns c0..
__device__ __forceinline__ void form_tile(uint8_t* bt, int r0, int c0, const float (&c)[4], float sgn,
                                          const float* beta, const float* uf, int lane) {
    const int g = lane >> 2, t = lane & 3;
    form_write2(bt, r0 + g, c0 + 2 * t, sgn * c[0], sgn * c[1], beta, uf);
    form_write2(bt, r0 + g + 8, c0 + 2 * t, sgn * c[2], sgn * c[3], beta, uf);
}

// (I + A)^-1, A strictly lower triangular 64 x 64 (row stride kAS), by
// recursive doubling on the block-triangular inverse
//   [[L11, 0], [L21, L22]]^-1 = [[M11, 0], [-M22 L21 M11, M22]]:
//   level 1: the four 16 x 16 diagonal blocks, forward substitution by
//            columns (threads 0..63, one column each);
//   level 2: blocks (1,0) and (3,2), from the level-1 inverses (warps
//            w < 4: block pair w / 2, 8-column tile w % 2);
//   level 3: the lower-left 32 x 32 block, from the two 32 x 32 inverses
//            (warp w: 16 x 8 tile w of it).
// Within a level, a warp waits only for the warps whose products it reads:
// none at level 2 (each warp's second product reads only its own tile of the
// first), its partner w ^ 4 at level 3 (named barriers 4-7, 64 threads).
// The products run over full blocks: the zero upper parts of the triangular
// factors make that exact.  Levels 1 and 2 keep their blocks in place (the
// later levels read them); the forms of level 1's blocks are written by the
// warps that level 2 leaves idle, those of levels 2 and 3 from the MMA
// fragments.  Ptmp holds the left products.
__device__ void prep_solve(float* As, float* Ptmp, uint8_t* bt, const float* beta, const float* uf, int p, int bar) {
    const int w = p >> 5, lane = p & 31;
    if (p < kC) {  // level 1
        const int b = p >> 4, c = p & 15;
        const float* Ab = As + 16 * b * kAS + 16 * b;
        float s[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) s[i] = (i == c) ? 1.f : 0.f;
#pragma unroll
        for (int j = 0; j < 15; ++j) {
            const float mj = s[j];
#pragma unroll
            for (int i = j + 1; i < 16; ++i) s[i] = fmaf(-Ab[i * kAS + j], mj, s[i]);
        }
        float* Mb = As + 16 * b * kAS + 16 * b + c;
#pragma unroll
        for (int i = 0; i < 16; ++i) Mb[i * kAS] = s[i];
    }
    named_sync(bar, kPrepThreads);
    if (w >= 4) {  // the diagonal blocks' forms, two elements a thread at a time, while level 2 runs
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int q = p - 128 + 128 * e, b = q >> 7, i = (q >> 3) & 15, j = 2 * (q & 7);
            const float* m = As + (16 * b + i) * kAS + 16 * b + j;
            form_write2(bt, 16 * b + i, 16 * b + j, m[0], m[1], beta, uf);
        }
    }
    {  // level 2: P = A_{x+1,x} M_xx, then M_{x+1,x} = -M_{x+1,x+1} P, x = 0, 2
        const int x = 2 * ((w >> 1) & 1), nt = w & 1;
        float* P = Ptmp + ((w >> 1) & 1) * 320;  // 16 x 16, row stride 20
        float c[1][4];
        if (w < 4) {
            warp_gemm<1, 1>(c, As + 16 * (x + 1) * kAS + 16 * x, kAS, As + 16 * x * kAS + 16 * x + 8 * nt, kAS, lane);
            warp_store<1>(c, P + 8 * nt, 20, 1.f, lane);
            __syncwarp();  // (the second product reads only the columns of P this warp wrote)
            warp_gemm<1, 1>(c, As + 16 * (x + 1) * kAS + 16 * (x + 1), kAS, P + 8 * nt, 20, lane);
            warp_store<1>(c, As + 16 * (x + 1) * kAS + 16 * x + 8 * nt, kAS, -1.f, lane);
            form_tile(bt, 16 * (x + 1), 16 * x + 8 * nt, c[0], -1.f, beta, uf, lane);
        }
    }
    named_sync(bar, kPrepThreads);
    {  // level 3: P = A[32:64, 0:32] M[0:32, 0:32], then M[32:64, 0:32] = -M[32:64, 32:64] P
        // (8 tiles of 16 x 8, taken in turn by the group's warps; the result only goes into the forms)
        constexpr int kWarps = kPrepThreads / 32;
        float c[8 / kWarps][1][4];
#pragma unroll
        for (int i = 0; i < 8 / kWarps; ++i) {
            const int tw = w + kWarps * i, r0 = 16 * (tw >> 2), c0 = 8 * (tw & 3);
            warp_gemm<2, 1>(c[i], As + (32 + r0) * kAS, kAS, As + c0, kAS, lane);
        }
#pragma unroll
        for (int i = 0; i < 8 / kWarps; ++i) {
            const int tw = w + kWarps * i, r0 = 16 * (tw >> 2), c0 = 8 * (tw & 3);
            warp_store<1>(c[i], Ptmp + r0 * 36 + c0, 36, 1.f, lane);  // 32 x 32, row stride 36
        }
        // the second products read P's columns c0..c0+7, written by warps w and w ^ 4 (rows 0-15, 16-31)
        static_assert(kWarps == 8, "level 3's pair barriers assume eight prep warps");
        named_sync(4 + (w & 3), 64);
#pragma unroll
        for (int i = 0; i < 8 / kWarps; ++i) {
            const int tw = w + kWarps * i, r0 = 16 * (tw >> 2), c0 = 8 * (tw & 3);
            warp_gemm<2, 1>(c[i], As + (32 + r0) * kAS + 32, kAS, Ptmp + c0, 36, lane);
        }
#pragma unroll
        for (int i = 0; i < 8 / kWarps; ++i) {
            const int tw = w + kWarps * i, r0 = 16 * (tw >> 2), c0 = 8 * (tw & 3);
            form_tile(bt, 32 + r0, c0, c[i][0], -1.f, beta, uf, lane);
        }
    }
}

// ---------------------------------------------------------- state roles --
// Thread n of the state warps owns tensor-memory lane n = 32q + lane: row n
// of D''_T (column n of T) and of D''_S (column n of S).

// D'' <- (I, 0): row n of D''_T is e_n.
__device__ void state_init(uint32_t tmem, int q, int lane) {
    const uint32_t tl = tmem + ((32u * q) << 16);
    const int n = 32 * q + lane;
    uint32_t r[32];
#pragma unroll 1
    for (int cb = 0; cb < 4; ++cb) {
#pragma unroll
        for (int j = 0; j < 32; ++j) r[j] = (32 * cb + j == n) ? 0x3f800000u : 0u;
        tmem_st32(tl + TM_DT + 32 * cb, r);
    }
#pragma unroll
    for (int j = 0; j < 32; ++j) r[j] = 0u;
#pragma unroll 1
    for (int cb = 0; cb < 4; ++cb) tmem_st32(tl + TM_DS + 32 * cb, r);
    tmem_wait_st();
}

// Max |.| of this thread's row of a 128-column tensor-memory block.
__device__ __noinline__ float row_absmax(uint32_t addr) {
    float m = 0.f;
#pragma unroll 1
    for (int cb = 0; cb < 4; ++cb) {
        uint32_t x[32];
        tmem_ld32(addr + 32 * cb, x);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) m = fmaxf(m, fabsf(__uint_as_float(x[j])));
    }
    return m;
}
// This thread's row of a 128-column tensor-memory block times sc.
__device__ __noinline__ void row_scale(uint32_t addr, float sc) {
#pragma unroll 1
    for (int cb = 0; cb < 4; ++cb) {
        uint32_t x[32];
        tmem_ld32(addr + 32 * cb, x);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) x[j] = __float_as_uint(__uint_as_float(x[j]) * sc);
        tmem_st32(addr + 32 * cb, x);
    }
    tmem_wait_st();
}

// Warp max, then the 4 state warps through shared memory.
__device__ float state_reduce_max(float v, float* slot, int q, int lane) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    named_sync(2);  // (the slots' previous values have been read)
    if (lane == 0) slot[q] = v;
    named_sync(2);
    return fmaxf(fmaxf(slot[0], slot[1]), fmaxf(slot[2], slot[3]));
}

// The pass of one half after GEMM1: X (64 fp32 columns) rewritten in place as
// the A operand of GEMM2, two tokens per column (the lower token in the low
// half).  S half: bf16 (its lazy scale spans up to 2^112), tokens 2j, 2j + 1 in
// column j.  T half: a bf16 hi + lo pair (about 16 bits; T_C over long
// segments needs more than one bf16), tokens 16k..16k+15 as hi in columns
// 16k..16k+7 and lo in 16k+8..16k+15, each group of 16 columns read and then
// rewritten in place.
template <bool kHalfT>
__device__ __forceinline__ void state_pass(uint32_t addr) {
    if (kHalfT) {
#pragma unroll 1
        for (int k = 0; k < 4; ++k) {
            uint32_t x[16], y[16];
            tmem_ld16(addr + 16 * k, x);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 8; ++j)
                split_bf16(__uint_as_float(x[2 * j]), __uint_as_float(x[2 * j + 1]), y[j], y[8 + j]);
            tmem_st16(addr + 16 * k, y);
        }
    } else {
#pragma unroll 1
        for (int m = 0; m < 2; ++m) {
            uint32_t x[32], y[16];
            tmem_ld32(addr + 32 * m, x);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j) y[j] = pack_bf16(__uint_as_float(x[2 * j]), __uint_as_float(x[2 * j + 1]));
            tmem_st16(addr + 16 * m, y);
        }
    }
    tmem_wait_st();
}

// -W^T of the next chunk (lane i holds column i of it, in the W columns) ->
// the tf32 K-major [64 t][128 i] operand of GEMM1.
__device__ void convert_w(uint8_t* smem, uint32_t tmem, int q, int lane) {
    const int i = 32 * q + lane;
    const uint32_t tl = tmem + ((32u * q) << 16);
    uint8_t* bw = smem + OFF_W + (i >> 5) * 8192 + (i & 3) * 4;
    const uint32_t c4 = (uint32_t)((i & 31) >> 2);
#pragma unroll 1
    for (int half = 0; half < 2; ++half) {
        uint32_t w[32];
        tmem_ld32(tl + TM_W + 32 * half, w);
        tmem_wait_ld();
        uint8_t* b = bw + 32 * half * 128;
#pragma unroll
        for (int j = 0; j < 32; ++j)
            *reinterpret_cast<float*>(b + j * 128 + ((c4 ^ (uint32_t)(j & 7)) << 4)) =
                tf32_round(__uint_as_float(w[j]));
    }
}

// End of an item, T half: T_C = mantissa * 2^exp with the mantissa's largest
// entry in [1, 2), from D''_T and its scale 2^F.  Each 32-column chunk of
// D''_T is reset to the identity's as soon as it has been read, so that the
// next item may start on it.  Thread n writes column n (coalesced across the
// warp).
__device__ void state_epilogue_T(Misc* ms, const TcArgs& a, int64_t obj, float F, uint32_t tmem, int q, int lane) {
    const int n = 32 * q + lane;
    const uint32_t tl = tmem + ((32u * q) << 16);
    const float m = state_reduce_max(row_absmax(tl + TM_DT), ms->red, q, lane);
    const float Fi = floorf(F);
    const float sc = exp2f(F - Fi);  // in [1, 2)
    const float ms_ = m * sc;
    const int ef = (ms_ > 0.f && ms_ < INFINITY) ? ilogbf(ms_) : 0;
    const float f = ldexpf(sc, -ef);
    float* T = a.T_out + obj * kD * kD;
#pragma unroll 1
    for (int cb = 0; cb < 4; ++cb) {
        uint32_t x[32], id[32];
        tmem_ld32(tl + TM_DT + 32 * cb, x);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) id[j] = (32 * cb + j == n) ? 0x3f800000u : 0u;
        tmem_st32(tl + TM_DT + 32 * cb, id);
#pragma unroll
        for (int j = 0; j < 32; ++j) T[(32 * cb + j) * kD + n] = __uint_as_float(x[j]) * f;
    }
    tmem_wait_st();
    if (n == 0) a.T_exp[obj] = (int)Fi + ef;
}
// S half: S(C|0) as is (the last chunk ends at the true scale).  D''_S is not
// reset: an item's first chunk skips GEMM1 of the S half (X_S = U~, as S
// starts at 0) and its first GEMM2 MMA overwrites D''_S.
__device__ void state_epilogue_S(const TcArgs& a, int64_t obj, uint32_t tmem, int q, int lane) {
    const int n = 32 * q + lane;
    const uint32_t tl = tmem + ((32u * q) << 16);
    float* S = a.S_out + obj * kD * kD;
#pragma unroll 1
    for (int cb = 0; cb < 4; ++cb) {
        uint32_t x[32];
        tmem_ld32(tl + TM_DS + 32 * cb, x);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) S[(32 * cb + j) * kD + n] = __uint_as_float(x[j]);
    }
}

// All n threads of named barrier `id` agree: true only if every one passed true.
__device__ __forceinline__ bool wg_all(int id, bool v, int n = 128) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n"
        " bar.red.and.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}\n"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}

// --------------------------------------------------------- role drivers --
// g: CTA-wide index of the item's first chunk (barrier phases run on it
// across items); nc: chunks of this item's body.  Every barrier completes
// once per chunk (the ring and gate-slot barriers once per use of their
// slot).  A thread waits for phase k of a barrier only once it has seen
// phase k - 1 complete, or knows it from the order of the other roles.

// An issuer's idle step: the start of its idle time (t_idle, 0 if it was
// busy), or 0 once the CTA aborted or this wait ran out (which sets the abort
// flag and the device error word).
__device__ __forceinline__ uint64_t issuer_idle(Misc* ms, const TcArgs& a, uint64_t t_idle) {
    if (*(volatile int*)&ms->abort_flag) return 0;
    const uint64_t now = globaltimer_ns();
    if (t_idle != 0 && now - t_idle > a.wait_ns) {
        *(volatile int*)&ms->abort_flag = 1;
        set_error(a.err, kErrTimeout);
        return 0;
    }
    return t_idle != 0 ? t_idle : now;
}

// Warp 1, one thread: the prep stream.  The gram of a chunk as soon as its
// keys are in and the prep warps have read the previous gram (up to three
// chunks ahead of W^T), and W^T = -(M Diag(b) K)^T of a chunk as soon as its
// M forms, its fp16 keys and a free W block are there.
__device__ void issue_prep_role(Misc* ms, uint8_t* smem, const TcArgs& a, uint32_t tmem, uint32_t g, int nc) {
    const uint32_t sb = smem_u32(smem);
    int ig = 0, iw = 0;
    uint64_t t_idle = 0;
    while (iw < nc) {
        bool any = false;
        if (ig < nc && ig <= iw + 3) {  // G = K K^T (K-major view of the key tile, two 64-wide boxes)
            const uint32_t gc = g + ig;
            if (mbar_test(&ms->fullK[gc % kKStages], (gc / kKStages) & 1) &&
                (gc == 0 || mbar_test(&ms->g_read, (gc - 1) & 1))) {
                tc_fence_after();
                const uint64_t d0 = sdesc_sw128(sb + OFF_K + (gc % kKStages) * kTile, 0, 1024);
#pragma unroll 2
                for (int k = 0; k < 8; ++k) {
                    const uint64_t d = d0 + 512 * (k >> 2) + 2 * (k & 3);
                    mma_bf16_ss(tmem + TM_G, d, d, ID_GRAM, k > 0);
                }
                mma_commit(&ms->g_done);
                ++ig;
                any = true;
            }
        }
        if (iw < ig) {  // W^T = K^T (-M Diag(b))^T (hi + lo) into the W columns (a descriptor's address counts 16 B)
            const uint32_t gc = g + iw;
            if (mbar_test(&ms->that_ready[gc & 1], (gc >> 1) & 1) &&
                (gc == 0 || mbar_test(&ms->w_read, (gc - 1) & 1))) {
                tc_fence_after();
                const uint64_t a0 = sdesc_sw128(sb + OFF_K + (gc % kKStages) * kTile, 8192, 1024),
                               bh = sdesc_sw128(sb + OFF_BT + (gc & 1) * kBT, 0, 1024),
                               bl = sdesc_sw128(sb + OFF_BT + (gc & 1) * kBT + 8192, 0, 1024);
#pragma unroll 1
                for (int k = 0; k < 4; ++k) {
                    mma_bf16_ss(tmem + TM_W, a0 + 128 * k, bh + 2 * k, ID_W, k > 0);
                    mma_bf16_ss(tmem + TM_W, a0 + 128 * k, bl + 2 * k, ID_W, true);
                }
                mma_commit(&ms->w_done);
                mma_commit(&ms->bt_free[gc & 1]);
                ++iw;
                any = true;
            }
        }
        if (any) {
            t_idle = 0;
        } else if ((t_idle = issuer_idle(ms, a, t_idle)) == 0) {
            return;
        }
    }
}

// The state-stream issuers' wait: a spin on the phase (a suspended thread
// answers a completed phase late, and these threads' MMAs are the chain).
__device__ __noinline__ bool issuer_wait_slow(uint64_t* bar, uint32_t parity, int* abort_flag, uint64_t wait_ns,
                                              unsigned* err) {
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
#pragma unroll 1
        for (int j = 0; j < 64; ++j)
            if (mbar_test(bar, parity)) return true;
        if (*(volatile int*)abort_flag) return false;
        if (globaltimer_ns() - t0 > wait_ns) break;
    }
    *(volatile int*)abort_flag = 1;
    set_error(err, kErrTimeout);
    return false;
}
__device__ __forceinline__ bool issuer_wait(uint64_t* bar, uint32_t parity, Misc* ms, const TcArgs& a) {
    if (mbar_test(bar, parity)) return true;
    return issuer_wait_slow(bar, parity, &ms->abort_flag, a.wait_ns, a.err);
}

// Warp 2, one thread: the S half in chunk order -- U~ into X_S, GEMM1, then
// (after the S pass) GEMM2.  A thread issues a small MMA only every ~60
// cycles, so the two halves have an issuer each; every accumulator's MMAs
// come from one thread, in order.
__device__ void issue_s_role(Misc* ms, uint8_t* smem, const TcArgs& a, uint32_t tmem, uint32_t g, int nc) {
    const uint32_t sb = smem_u32(smem);
    for (int c = 0; c < nc; ++c) {
        const uint32_t gc = g + c;
        const uint64_t bw = sdesc_sw128(sb + OFF_W, 0, 1024);
        // U~ = V^T (M Diag(b uf))^T: needs the M forms, the values and a free X_S (GEMM2 of the previous
        // chunk has read it)
        if (!issuer_wait(&ms->that_ready[gc & 1], (gc >> 1) & 1, ms, a)) return;
        if (!issuer_wait(&ms->fullV[gc % kVStages], (gc / kVStages) & 1, ms, a)) return;
        if (gc >= 1 && !issuer_wait(&ms->d_ready_s, (gc - 1) & 1, ms, a)) return;
        tc_fence_after();
        {
            const uint64_t a0 = sdesc_sw128(sb + OFF_V + (gc % kVStages) * kTile, 8192, 1024),
                           b0 = sdesc_sw128(sb + OFF_BT + (gc & 1) * kBT + 16384, 0, 1024);
#pragma unroll 1
            for (int k = 0; k < 4; ++k) mma_bf16_ss(tmem + TM_XS, a0 + 128 * k, b0 + 2 * k, ID_U, k > 0);
        }
        mma_commit(&ms->emptyV[gc % kVStages]);
        mma_commit(&ms->bt_free[gc & 1]);
        // GEMM1 (tf32, A = the state in tensor memory): X_S += D''_S (-W^)^T; not in an item's first
        // chunk, where S is 0 (and D''_S may still be being written out)
        if (c > 0) {
            if (!issuer_wait(&ms->w_cvt[gc & 1], (gc >> 1) & 1, ms, a)) return;
            if (!issuer_wait(&ms->pre_done, gc & 1, ms, a)) return;
            tc_fence_after();
#pragma unroll 4
            for (int k = 0; k < 16; ++k)
                mma_tf32_ts(tmem + TM_XS, tmem + TM_DS + 8 * k, bw + 512 * (k >> 2) + 2 * (k & 3), ID_G1, true);
        }
        mma_commit(&ms->x_done_s);
        // GEMM2 (bf16, A = the pass's output in tensor memory): D''_S += X_S K
        if (!issuer_wait(&ms->y_ready_s, gc & 1, ms, a)) return;
        tc_fence_after();
        {
            const uint64_t kt = sdesc_sw128(sb + OFF_K + (gc % kKStages) * kTile, 8192, 1024);
#pragma unroll 1
            for (int k = 0; k < 4; ++k)
                mma_bf16_ts(tmem + TM_DS, tmem + TM_XS + 8 * k, kt + 128 * k, ID_G2S, c > 0 || k > 0);
        }
        mma_commit(&ms->d_ready_s);
        mma_commit(&ms->emptyK[gc % kKStages]);
    }
}

// Warp 3, one thread: the T half in chunk order -- GEMM1, then (after the T
// pass) GEMM2.
__device__ void issue_t_role(Misc* ms, uint8_t* smem, const TcArgs& a, uint32_t tmem, uint32_t g, int nc) {
    const uint32_t sb = smem_u32(smem);
    for (int c = 0; c < nc; ++c) {
        const uint32_t gc = g + c;
        const uint64_t bw = sdesc_sw128(sb + OFF_W, 0, 1024);
        // GEMM1 (tf32): X_T = D''_T (-W^)^T; X_T is free once GEMM2 of the previous chunk has read it
        if (!issuer_wait(&ms->w_cvt[gc & 1], (gc >> 1) & 1, ms, a)) return;
        if (!issuer_wait(&ms->pre_done, gc & 1, ms, a)) return;
        if (gc >= 1 && !issuer_wait(&ms->d_ready_t, (gc - 1) & 1, ms, a)) return;
        tc_fence_after();
#pragma unroll 4
        for (int k = 0; k < 16; ++k)
            mma_tf32_ts(tmem + TM_XT, tmem + TM_DT + 8 * k, bw + 512 * (k >> 2) + 2 * (k & 3), ID_G1, k > 0);
        mma_commit(&ms->x_done_t);
        // GEMM2 (bf16, hi + lo): D''_T += X_T K
        if (!issuer_wait(&ms->y_ready_t, gc & 1, ms, a)) return;
        tc_fence_after();
        {
            const uint64_t kt = sdesc_sw128(sb + OFF_K + (gc % kKStages) * kTile, 8192, 1024);
#pragma unroll 1
            for (int k = 0; k < 4; ++k) {
                mma_bf16_ts(tmem + TM_DT, tmem + TM_XT + 16 * k, kt + 128 * k, ID_G2T, true);
                mma_bf16_ts(tmem + TM_DT, tmem + TM_XT + 16 * k + 8, kt + 128 * k, ID_G2T, true);
            }
        }
        mma_commit(&ms->d_ready_t);
        mma_commit(&ms->emptyK[gc % kKStages]);
    }
}

// Warps 4-11: gram -> A^ -> M = (I + A^)^-1 and its operand forms, chunk
// after chunk (p: thread index among them).
__device__ void prep_role(Misc* ms, uint8_t* smem, const TcArgs& a, uint32_t tmem, uint32_t g, int nc, int p, int q,
                          int lane) {
    float* As = reinterpret_cast<float*>(smem + OFF_AS);
    float* Ptmp = reinterpret_cast<float*>(smem + OFF_PT);
    for (int c = 0; c < nc; ++c) {
        const uint32_t gc = g + c;
        const int slot = gc % kGateSlots;
        bool ok = wait_bar(&ms->gready[slot], (gc / kGateSlots) & 1, ms, a);
        ok = ok && wait_bar(&ms->g_done, gc & 1, ms, a);
        // the forms buffer's previous forms (chunk gc - 2) have been read (its phases are waited in order;
        // waited here rather than before the solve: one barrier of the prep warps fewer per chunk)
        ok = ok && (gc < 2 || wait_bar(&ms->bt_free[gc & 1], ((gc >> 1) - 1) & 1, ms, a));
        if (!wg_all(1, ok, kPrepThreads)) return;
        tc_fence_after();
        prep_arows(ms, As, slot, tmem, q, p >> 7, lane);
        tc_fence_before();
        named_sync(1, kPrepThreads);
        if (p == 0) mbar_arrive(&ms->g_read);
        prep_solve(As, Ptmp, smem + OFF_BT + (gc & 1) * kBT, ms->beta[slot], ms->uf[slot], p, 1);
        fence_async_smem();
        named_sync(1, kPrepThreads);
        if (p == 0) mbar_arrive(&ms->that_ready[gc & 1]);
    }
}

// Producer, lane 0: the next non-empty item of this CTA into slot s (nc = -1
// once the queue is exhausted or the CTA aborted); the slot's previous item
// has been copied by every reader.  Items are (segment, layer, head),
// segments in longest-body-first order.  An item with an empty body is the
// identity pair (I, 0): the whole warp writes it here and takes the next.
__device__ void publish_item(Misc* ms, const TcArgs& a, int k, int s, int lane) {
    const int LH = a.n_layers * a.n_heads;
    uint32_t g = 0;
    if (k > 0) {
        const ItemSlot& prev = ms->slots[(s + kItemSlots - 1) % kItemSlots];
        g = prev.g + (uint32_t)prev.nc;
    }
    for (;;) {
        int item = 0;
        if (lane == 0) item = *(volatile int*)&ms->abort_flag ? a.n_items : (int)atomicAdd(a.counter, 1u);
        item = __shfl_sync(0xffffffffu, item, 0);
        if (item >= a.n_items) {
            if (lane == 0) ms->slots[s].nc = -1;
            break;
        }
        const int pos = item / LH, lh = item % LH;
        const int seg = a.order[pos];
        const int64_t b0 = (int64_t)a.cu[seg] + (a.skip ? a.skip[seg] : 0), b1 = a.cu[seg + 1];
        const int64_t obj = ((int64_t)seg * a.n_layers + lh / a.n_heads) * a.n_heads + lh % a.n_heads;
        const int nc = (int)((b1 - b0 + kC - 1) / kC);
        if (nc <= 0) {
            float4* T = reinterpret_cast<float4*>(a.T_out + obj * kD * kD);
            float4* S = reinterpret_cast<float4*>(a.S_out + obj * kD * kD);
            for (int e = lane; e < kD * kD / 4; e += 32) {
                const int i = (4 * e) / kD, j = (4 * e) % kD;  // row i, columns j..j+3
                T[e] = make_float4(i == j, i == j + 1, i == j + 2, i == j + 3);
                S[e] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
            if (lane == 0) a.T_exp[obj] = 0;
            continue;
        }
        if (lane == 0) {
            ItemSlot& it = ms->slots[s];
            it.layer = lh / a.n_heads;
            it.head = lh % a.n_heads;
            it.b0 = b0;
            it.b1 = b1;
            it.nc = nc;
            it.obj = obj;
            it.g = g;
        }
        break;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&ms->slot_full[s]);  // (release: the slot is visible to the readers that wait on it)
}

// Warps 12-15, per chunk: the renormalisation (if planned), the S and T
// passes, then the next chunk's W operand (converted while GEMM2 of this chunk
// runs; the buffers alternate); the epilogue at the end of an item.  Unless the
// next chunk renormalises, its state is ready for GEMM1 once GEMM2 of this one
// is done (its issuers wait for that themselves), so pre_done is signalled as
// soon as the W operand is written.  Returns false once the CTA aborted.
// (Converting the next W before the passes, to overlap GEMM1, measured slower:
// the next W^T is then seldom ready and the passes wait for it.)
__device__ void convert_next_w(Misc* ms, uint8_t* smem, const TcArgs& a, uint32_t tmem, uint32_t ng, int q, int lane,
                               bool& ok) {
    // (the buffer was last read by GEMM1 of chunk ng - 1, whose completion the passes of that chunk waited for)
    ok = wg_all(2, wait_bar(&ms->w_done, ng & 1, ms, a));
    if (!ok) return;
    tc_fence_after();
    convert_w(smem, tmem, q, lane);
    fence_async_smem();
    tc_fence_before();
    named_sync(2);
    if (q == 0 && lane == 0) {
        mbar_arrive(&ms->w_cvt[ng & 1]);
        mbar_arrive(&ms->w_read);
    }
}

// first_ready: pre_done of the item's first chunk already signalled (by the
// previous item's epilogue); on return, whether this item's epilogue signalled
// that of the next item's first chunk.
__device__ bool state_item(Misc* ms, uint8_t* smem, const TcArgs& a, uint32_t tmem, const ItemSlot& it, ItemSlot& next,
                           int k, int q, int lane, bool& first_ready) {
    const int n = 32 * q + lane;
    const uint32_t tl = tmem + ((32u * q) << 16);
    int E = 0;
    float sum_lc = 0.f;
    bool ready = first_ready;  // pre_done of the current chunk already signalled
    for (int c = 0; c < it.nc; ++c) {
        const uint32_t gc = it.g + c;
        const int slot = gc % kGateSlots;
        if (!wg_all(2, wait_bar(&ms->gready[slot], (gc / kGateSlots) & 1, ms, a))) return false;
        const ChunkPlan pl = ms->plan[slot];
        sum_lc = pl.sum_lc;
        if (!ready) {
            if (pl.rn && c > 0) {  // renormalise the state GEMM2 of the previous chunk left
                bool ok = wait_bar(&ms->d_ready_s, (gc - 1) & 1, ms, a);
                ok = ok && wait_bar(&ms->d_ready_t, (gc - 1) & 1, ms, a);
                if (!wg_all(2, ok)) return false;
                tc_fence_after();
                row_scale(tl + TM_DS, exp2f(fmaxf(pl.preS, -149.f)));
                const float m = state_reduce_max(row_absmax(tl + TM_DT), ms->red, q, lane);
                const int e = (m > 0.f && m < INFINITY) ? ilogbf(m) : 0;
                row_scale(tl + TM_DT, ldexpf(1.f, -e));
                E += e;
            }
            tc_fence_before();
            named_sync(2);
            if (n == 0) mbar_arrive(&ms->pre_done);
        }
        if (!wg_all(2, wait_bar(&ms->x_done_s, gc & 1, ms, a))) return false;
        tc_fence_after();
        state_pass<false>(tl + TM_XS);
        tc_fence_before();
        named_sync(2);
        if (n == 0) mbar_arrive(&ms->y_ready_s);
        if (!wg_all(2, wait_bar(&ms->x_done_t, gc & 1, ms, a))) return false;
        tc_fence_after();
        state_pass<true>(tl + TM_XT);
        tc_fence_before();
        named_sync(2);
        if (n == 0) mbar_arrive(&ms->y_ready_t);
        // The W operand of the next chunk: the next chunk of this item, or the first of the next item.
        uint32_t ng = gc + 1;
        bool has_next = c + 1 < it.nc;
        if (!has_next) {
            const int s = (k + 1) % kItemSlots;
            if (!wg_all(2, wait_bar(&ms->slot_full[s], ((k + 1) / kItemSlots) & 1, ms, a))) return false;
            next = ms->slots[s];
            named_sync(2);
            if (n == 0) mbar_arrive(&ms->slot_read[s]);
            has_next = next.nc > 0;
            ng = next.g;
        }
        if (has_next) {
            bool ok;
            convert_next_w(ms, smem, a, tmem, ng, q, lane, ok);
            if (!ok) return false;
        }
        ready = false;
        if (c + 1 < it.nc) {  // the next chunk of this item: ready at once unless it renormalises
            const uint32_t g1 = gc + 1;
            const int s1 = g1 % kGateSlots;
            if (!wg_all(2, wait_bar(&ms->gready[s1], (g1 / kGateSlots) & 1, ms, a))) return false;
            if (!ms->plan[s1].rn) {
                if (n == 0) mbar_arrive(&ms->pre_done);
                ready = true;
            }
        }
    }
    const uint32_t last = it.g + it.nc - 1;
    bool ok = wait_bar(&ms->d_ready_s, last & 1, ms, a);
    ok = ok && wait_bar(&ms->d_ready_t, last & 1, ms, a);
    if (!wg_all(2, ok)) return false;
    tc_fence_after();
    state_epilogue_T(ms, a, it.obj, (float)E + sum_lc, tmem, q, lane);
    // D''_T is the identity's again: the next item's first chunk may start (its first chunk never
    // renormalises), while S is written out
    tc_fence_before();
    named_sync(2);
    first_ready = next.nc > 0;
    if (first_ready && n == 0) mbar_arrive(&ms->pre_done);
    state_epilogue_S(a, it.obj, tmem, q, lane);
    return true;
}

// ---------------------------------------------------------------- kernel --
__global__ void __launch_bounds__(kThreads, 1)
    gdn_build_tc_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                        const TcArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    Misc* ms = reinterpret_cast<Misc*>(smem + OFF_MISC);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if ((smem_u32(smem) & 1023u) != 0) {  // the swizzled operand layouts need 1024-byte alignment
        if (tid == 0) set_error(a.err, kErrBadIndex);
        return;
    }
    if (tid == 0) {
        for (int s = 0; s < kKStages; ++s) {
            mbar_init(&ms->fullK[s], 1);
            mbar_init(&ms->emptyK[s], 2);  // GEMM2 of both halves read the key tile
        }
        for (int s = 0; s < kVStages; ++s) {
            mbar_init(&ms->fullV[s], 1);
            mbar_init(&ms->emptyV[s], 1);
        }
        // gready .. drain are consecutive in Misc: one arrival each, but bt_free (two issuers read the M
        // forms) takes two and drain (every issuer's MMAs) three
        for (uint64_t* b = &ms->gready[0]; b <= &ms->drain; ++b)
            mbar_init(b, b == &ms->bt_free[0] || b == &ms->bt_free[1] ? 2 : b == &ms->drain ? 3 : 1);
        for (int s = 0; s < kItemSlots; ++s) {
            mbar_init(&ms->slot_full[s], 1);
            mbar_init(&ms->slot_read[s], kSlotReaders);
        }
        ms->abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kWarpTMA && lane == 0) {
        tma_prefetch_desc(&tmk);
        tma_prefetch_desc(&tmv);
    }
    if (warp == kWarpIssP) tmem_alloc(&ms->tmem_base, 512);
    for (uint32_t e = tid; e < 2 * kBT / 16; e += kThreads)  // the forms' zero blocks (written once)
        *reinterpret_cast<uint4*>(smem + OFF_BT + 16 * e) = make_uint4(0u, 0u, 0u, 0u);
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ms->tmem_base;
    const bool is_state = warp >= kWarpState0;
    const bool is_prep = warp >= kWarpPrep0 && warp < kWarpState0;
    const int q = warp & 3;  // tensor-memory lane quarter a warp may access
    if (is_state) state_init(tmem, q, lane);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (is_state) {
        // The state warps read item k + 1 from the ring during the last chunk of item k (to convert its
        // first W operand early); the first item before the loop.
        ItemSlot it, next;
        bool ok = wg_all(2, wait_bar(&ms->slot_full[0], 0, ms, a));
        if (ok) {
            it = ms->slots[0];
            named_sync(2);
            if (tid == 32 * kWarpState0) mbar_arrive(&ms->slot_read[0]);
            if (it.nc > 0) convert_next_w(ms, smem, a, tmem, it.g, q, lane, ok);
        }
        bool first_ready = false;
        for (int k = 0; ok && it.nc > 0; ++k) {
            if (!state_item(ms, smem, a, tmem, it, next, k, q, lane, first_ready)) break;
            it = next;
            if (*(volatile int*)&ms->abort_flag) break;
        }
    } else {
        // Every other role runs through the items at its own pace: the producer takes them from the
        // queue into a ring of kItemSlots slots, and the other roles copy them from there, so the next
        // item's loads, gram, solve and W^T overlap this item's last chunks and epilogue.  Across items
        // the roles meet on the same barriers as within one (chunks are numbered CTA-wide).
        for (int k = 0;; ++k) {
            const int s = k % kItemSlots;
            ItemSlot it;
            if (warp == kWarpTMA) {
                if (k >= kItemSlots && !wait_bar(&ms->slot_read[s], (k / kItemSlots - 1) & 1, ms, a)) break;
                publish_item(ms, a, k, s, lane);
                __syncwarp();
                it = ms->slots[s];
            } else if (is_prep) {
                const bool ok = wait_bar(&ms->slot_full[s], (k / kItemSlots) & 1, ms, a);
                if (!wg_all(1, ok, kPrepThreads)) break;
                it = ms->slots[s];
                named_sync(1, kPrepThreads);
                if (tid == 32 * kWarpPrep0) mbar_arrive(&ms->slot_read[s]);
            } else {  // the issuers, one thread each
                if (lane != 0) break;
                if (!wait_bar(&ms->slot_full[s], (k / kItemSlots) & 1, ms, a)) break;
                it = ms->slots[s];
                mbar_arrive(&ms->slot_read[s]);
            }
            if (it.nc < 0) break;
            if (warp == kWarpTMA) {
                producer_role(ms, smem, a, &tmk, &tmv, it.g, it.nc, it.layer, it.head, it.b0, it.b1, lane);
            } else if (warp == kWarpIssP) {
                issue_prep_role(ms, smem, a, tmem, it.g, it.nc);
            } else if (warp == kWarpIssS) {
                issue_s_role(ms, smem, a, tmem, it.g, it.nc);
            } else if (warp == kWarpIssT) {
                issue_t_role(ms, smem, a, tmem, it.g, it.nc);
            } else {
                prep_role(ms, smem, a, tmem, it.g, it.nc, tid - 32 * kWarpPrep0, q, lane);
            }
            if (*(volatile int*)&ms->abort_flag) break;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // Drain: every MMA this CTA issued (from every issuer) has completed before tensor memory is freed.  A
    // drain that runs out of polls is reported (the result is then not to be trusted); the memory is freed
    // all the same, since the kernel is about to exit either way.
    if (warp == kWarpIssP || warp == kWarpIssS || warp == kWarpIssT) {
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
    if (warp == kWarpIssP) tmem_dealloc(tmem, 512);
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

// [n_layers][n_tokens][n_heads][128] bf16 as a 3-D tensor (feature, head,
// layer-token row); box = 64 features x 1 head x 64 rows, 128-byte swizzle.
bool make_map(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap* m, const void* base, const BuildParams& p) {
    cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)p.n_heads, (cuuint64_t)p.n_layers * (cuuint64_t)p.n_tokens};
    cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)p.n_heads * kD * 2};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)kC}, es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool gdn_build_tc_supported(const BuildParams& p) {
    return p.family == kGDN && p.dk == kD && p.dv == kD && p.in_dtype == kBF16 && p.n_tokens > 0 &&
           (int64_t)p.n_layers * p.n_tokens < INT32_MAX && encode_fn() != nullptr;
}

cudaError_t launch_gdn_build_tc(const BuildParams& p, void* workspace, unsigned* err, cudaStream_t s) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    CUtensorMap tk, tv;
    if (!make_map(enc, &tk, p.k, p) || !make_map(enc, &tv, p.v, p)) return cudaErrorInvalidValue;
    TcArgs a;
    a.n_layers = p.n_layers;
    a.n_heads = p.n_heads;
    a.n_seg = p.n_seg;
    a.n_items = p.n_seg * p.n_layers * p.n_heads;
    a.n_tokens = p.n_tokens;
    a.cu = p.cu;
    a.skip = p.skip;
    a.alpha = p.alpha;
    a.beta = p.beta;
    a.T_out = p.T_out;
    a.T_exp = p.T_exp;
    a.S_out = p.S_out;
    a.order = reinterpret_cast<const int32_t*>(workspace);
    a.counter = reinterpret_cast<unsigned*>(reinterpret_cast<char*>(workspace) + build_workspace_bytes(p.n_seg) - 256);
    a.err = err;
    a.wait_limit = 1u << 26;
    a.wait_ns = 2000000000ull;  // 2 s
    if (a.n_items == 0) return cudaSuccess;
    const int sms = sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    cudaError_t e = cudaFuncSetAttribute(gdn_build_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    const int grid = a.n_items < sms ? a.n_items : sms;
    gdn_build_tc_kernel<<<grid, kThreads, kSmemBytes, s>>>(tk, tv, a);
    return cudaGetLastError();
}

}  // namespace hypic
