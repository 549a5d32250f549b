// gdn_build_tc.cu -- chunked GDN build of the cached pair (T_C, S(C|0)) on the
// sm_103a tensor cores (d = 128, bf16 keys/values).
//
// What it computes: for a segment C and a head, T_C = A_L ... A_1 with the
// gated-delta transition A_t = a_t (I - b_t k_t k_t^T), and S(C|0), the state
// after C from zero with the write term b_t k_t v_t^T (aibase article on
// HYPIC, paragraph on the linear layers: the cached pair of a segment).
//
// How: tokens are taken in chunks of 64.  With g_i = a_1 ... a_i inside a
// chunk (g_C its last value), A[i][j] = b_i (g_i/g_j) k_i.k_j for j < i,
// That = (I + A)^-1 Diag(b), W = That Diag(g) K and U = That V, the chunk
// maps the running pair D = [T | S] (dk x 2dk) to
//     D <- g_C D + K^T Diag(g_C/g_t) ([0 | U] - W D),
// which is the token recurrence applied 64 times (WY / UT form of a product
// of generalised Householder transitions).  The state is held transposed,
// D'' = D^T / sigma (256 x 128 fp32, sigma a per-half scale, see "Lazy
// decay" below), in tensor memory; per chunk:
//   gram      G = K K^T                      bf16 MMA, M=64  N=64  K=128
//   solve     That from G and the gates      CUDA cores + warp MMAs (block-triangular inverse)
//   W'^T, U^T K^T (That Diag(up))^T, V^T That^T   bf16 MMA, M=128 N=64 K=64
//   GEMM1     X''_h = D''_h W'^T             tf32 MMA, A read from tensor memory
//   pass      Y''_T = Diag(f_T) X''_T^T (bf16, in place of X''_T in tensor memory),
//             Y''_S = Diag(f_S) X''_S^T + U~ (bf16, smem)
//   GEMM2     D''_h += Y''_h K                bf16 MMA, M=128 N=128 K=64 (A of the T half
//                                             read from tensor memory)
// with up_t = g_t / g_C^(1/2) in W' = W / g_C^(1/2) and f_h = -g_C^(1/2)/g_t
// (times the renormalisation factor): the in-chunk decay is centred on the
// middle of its range so that neither factor leaves the float32 range for
// chunk decays down to 2^-252.
// Two operands are carried as a pair of bf16 values (x = hi + lo, hi the
// truncation of x and lo the rest): That Diag(up) in the W product and Y''_T
// in the T half of GEMM2.  Rounding either to a single bf16 alone costs T_C about
// 7e-3 relative error over 2048-token segments with strong decay; the pair
// brings it to ~2e-3.  Keys and values are bf16 inputs and need no split.
// T_C falls far below the fp32 range over long segments: it is returned as a
// mantissa and a power-of-two exponent.
//
// Roles (480 threads): warp 0 loads keys and values (TMA) and writes the gate
// tables.  Two single-thread issuers send the MMAs as their inputs become
// ready: warp 1 W'^T, GEMM1 of the T half and GEMM2, warp 14 GEMM1 of the S
// half, U^T and the gram (one thread issues a small MMA only about every 60
// cycles; two come closer to the tensor pipe's own rate).  Warps 6-13 (the
// prep warps) turn each gram into That; warps 2-5 (the state warpgroup) run
// the pass between GEMM1 and GEMM2, convert W into an MMA operand and write
// the result.  The prep warps run ahead of the state chain: only the pass,
// the W conversion and the two state GEMMs are serial per chunk.  The roles
// meet on mbarriers; every wait is bounded and a wait that runs out sets the
// device error word.
// One CTA per SM, persistent over (segment, layer, head) items taken from an
// atomic queue in longest-body-first order.  Warp 0 publishes them through a
// ring of item slots and each role runs through them at its own pace, so one
// item's first chunks overlap the previous item's last ones.
#include <cuda.h>
#include <cuda_bf16.h>
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
constexpr int kKStages = 3;       // K ring depth (the gram of a chunk wants its keys early)
constexpr int kGateSlots = 4;     // per-chunk gate tables in flight
constexpr int kThreads = 480;
constexpr int kWarpTMA = 0, kWarpMMA = 1, kWarpState0 = 2, kWarpPrep0 = 6, kWarpMMA2 = 14;
constexpr int kPrepThreads = 256;  // warps 6-13: two warps per tensor-memory lane quarter

// Shared memory map (byte offsets; every operand region is 1024-byte aligned).
constexpr uint32_t kTile = 16384;                       // 64 tokens x 128 bf16, two 64-column TMA boxes
constexpr uint32_t OFF_K = 0;                           // K ring
constexpr uint32_t OFF_V = OFF_K + kKStages * kTile;    // V (one chunk: read only by the U^T MMA)
constexpr uint32_t OFF_BW = OFF_V + kTile;              // W: fp32 [64 t][128 i], K-major, 4 blocks of 32 i
constexpr uint32_t OFF_AY = OFF_BW + 32768;             // Y''_S (with U~): bf16 [128 n][64 t], K-major
constexpr uint32_t kBT = 24576;                         // That Diag(g) hi, That, That Diag(g) lo: bf16 [64][64]
constexpr uint32_t OFF_BT = OFF_AY + 16384;             // two of them: chunk gc uses buffer gc % 2
constexpr uint32_t OFF_AS = OFF_BT + 2 * kBT;           // A / (I+A)^-1: fp32 [64][kAS] (padded rows)
constexpr int kAS = 68;                                 // row stride (floats) of that scratch
constexpr uint32_t OFF_PT = OFF_AS + ((64 * kAS * 4 + 1023) / 1024) * 1024;  // solve scratch: 32 x 36 fp32
constexpr uint32_t OFF_MISC = OFF_PT + 5120;

// An item of the queue as the producer publishes it to the other roles.
struct ItemSlot {
    int64_t b0, b1, obj;  // body [b0, b1) in the token index, output object
    uint32_t g;           // CTA-wide index of the item's first chunk
    int nc, layer, head;  // nc < 0: the queue is exhausted
};
constexpr int kItemSlots = 4;
constexpr int kSlotReaders = 4;  // warp 1, warp 14, the state warpgroup, the prep warps

struct Misc {
    uint64_t fullK[kKStages], emptyK[kKStages], fullV, emptyV;
    uint64_t gready[kGateSlots];  // producer -> prep, state: gate tables of a chunk written
    uint64_t g_done, g_read;      // gram committed; gram read by the prep warpgroup
    // That of chunk gc written (that_ready[gc % 2]); the W/U MMAs that read it are done (bt_free[gc % 2],
    // one commit from each issuer).  One barrier per That buffer: the prep may run two chunks ahead of
    // an issuer, and an issuer one chunk ahead of the other, so a shared barrier could be two phases
    // ahead of a parity wait or mix the commits of two chunks in one phase.
    uint64_t that_ready[2], bt_free[2];
    uint64_t u_done, w_done;      // U^T, W^T committed
    uint64_t w_cvt;               // W operand written
    uint64_t x_done_s, x_done, xs_free, y_ready, d_ready, drain;  // GEMM1 S half / T half done; X''_S read
    alignas(16) float lg2[kGateSlots][kC];  // slot gc % kGateSlots; every table is read as float4
    alignas(16) float beta[kGateSlots][kC];
    alignas(16) float up[kGateSlots][kC];
    alignas(16) float wn[kGateSlots][kC];  // 2^(lg2_t - lg2_C/2), 2^(lg2_C/2 - lg2_t): g_r/g_j = up_r wn_j
    alignas(16) float fT[kC];    // state pass: Y'' = f X'' for the T and S halves
    alignas(16) float fS[kC];
    alignas(16) float uf[kC];    // U~ = Diag(uf) U
    float red[2][4];
    float red_ep[4];
    uint64_t slot_full[kItemSlots], slot_read[kItemSlots];  // item slot written / copied by every reader
    ItemSlot slots[kItemSlots];
    int abort_flag;
    uint32_t tmem_base;
};
constexpr uint32_t kSmemBytes = OFF_MISC + sizeof(Misc);
static_assert(OFF_MISC % 16 == 0 && offsetof(Misc, lg2) % 16 == 0 && offsetof(Misc, beta) % 16 == 0 &&
                  offsetof(Misc, up) % 16 == 0 && offsetof(Misc, wn) % 16 == 0 && offsetof(Misc, fT) % 16 == 0,
              "float4 / float2 accesses of the gate tables need 16-byte alignment");
static_assert(kSmemBytes <= 232448, "shared memory budget");

// Tensor-memory columns.
// W^T is staged in the X_S columns: it is converted before GEMM1 writes X.
constexpr uint32_t TM_DT = 0, TM_DS = 128, TM_XT = 256, TM_XS = 320, TM_U = 384, TM_G = 448;

constexpr uint32_t ID_GRAM = idesc(1, 64, 64, false, false);  // G = K K^T
constexpr uint32_t ID_WU = idesc(1, 128, 64, true, false);    // W^T, U^T: A = K^T / V^T (MN-major)
constexpr uint32_t ID_G1 = idesc(2, 128, 64, false, false);   // X' = D' W^T (tf32, A in TMEM)
constexpr uint32_t ID_G2 = idesc(1, 128, 128, false, true);   // D' += Y' K (B = K, MN-major)

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
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}
__device__ __forceinline__ float bf16_round(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }
// Two values as bf16 pairs x = hi + lo: hi is x with its low 16 bits cleared
// (exact; two values packed by one byte permute) and lo = x - hi (exact in
// fp32) rounded to bf16, so hi + lo keeps about 16 significant bits of x.
__device__ __forceinline__ void split2_bf16(float x, float y, uint32_t& hi, uint32_t& lo) {
    const uint32_t hx = __float_as_uint(x) & 0xffff0000u, hy = __float_as_uint(y) & 0xffff0000u;
    hi = __byte_perm(hx, hy, 0x7632);
    lo = pack_bf16(x - __uint_as_float(hx), y - __uint_as_float(hy));
}
__device__ __forceinline__ float tf32_rna(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

// ----------------------------------------------------------- prep roles --
// p: thread index inside the prep warpgroup (0..127); q: its tensor-memory
// lane quarter; lane: lane in the warp.

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

// Gate tables of one chunk (one warp, two tokens a lane): lg2[t] = sum_{s<=t}
// log2 a_s (inclusive prefix inside the chunk), beta[t], and
// up[t] = g_t / g_C^(1/2), wn[t] = g_C^(1/2) / g_t: the in-chunk decay
// centred on the middle of its range, so that both stay in float32 range for
// chunk decays g_C down to 2^-252 (g_t itself underflows below 2^-126).  The
// exponents are clamped to +-126, which only matters beyond that.
__device__ void gate_tables(Misc* ms, int slot, const float (&ra)[2], const float (&rb)[2], int lane) {
    const float l0 = log2f(fmaxf(ra[0], FLT_MIN)), l1 = log2f(fmaxf(ra[1], FLT_MIN));
    float s = l0 + l1;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, s, off);
        if (lane >= off) s += y;
    }
    const float before = __shfl_up_sync(0xffffffffu, s, 1);
    const float e0 = (lane > 0 ? before : 0.f) + l0, e1 = e0 + l1;
    const float h = 0.5f * __shfl_sync(0xffffffffu, e1, 31);
    const int t = 2 * lane;
    *reinterpret_cast<float2*>(&ms->lg2[slot][t]) = make_float2(e0, e1);
    *reinterpret_cast<float2*>(&ms->beta[slot][t]) = make_float2(rb[0], rb[1]);
    auto ex = [](float x) { return exp2f(fminf(fmaxf(x, -126.f), 126.f)); };
    *reinterpret_cast<float2*>(&ms->up[slot][t]) = make_float2(ex(e0 - h), ex(e1 - h));
    *reinterpret_cast<float2*>(&ms->wn[slot][t]) = make_float2(ex(h - e0), ex(h - e1));
}

// Rows of A from the gram matrix in tensor memory (M=64 accumulator layout:
// row 16q + l sits in lane 32q + l, l < 16):
// A[r][j] = b_r 2^(lg2_r - lg2_j) G[r][j] for j < r, 0 elsewhere.
// Half h of the prep warps reads columns 32h..32h+31; lane l < 16 writes the
// first 16 of them in its row, lane l + 16, which holds no row, takes the
// other 16 of the same row from lane l by a shuffle.
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
    const float coef = ms->beta[slot][r] * ms->up[slot][r];
    const float* wn = ms->wn[slot] + cb;
    float* row = As + r * kAS + cb;
#pragma unroll
    for (int j = 0; j < 16; j += 4) {
        const float4 w = *reinterpret_cast<const float4*>(wn + j);
        float4 v;
        v.x = (cb + j < r) ? coef * w.x * __uint_as_float(gv[j]) : 0.f;
        v.y = (cb + j + 1 < r) ? coef * w.y * __uint_as_float(gv[j + 1]) : 0.f;
        v.z = (cb + j + 2 < r) ? coef * w.z * __uint_as_float(gv[j + 2]) : 0.f;
        v.w = (cb + j + 3 < r) ? coef * w.w * __uint_as_float(gv[j + 3]) : 0.f;
        *reinterpret_cast<float4*>(row + j) = v;
    }
}

// Warp-level block products for the solve (mma.sync m16n8k16, bf16 with
// fp32 accumulation).  Each fp32 operand is carried as a pair of bf16 values
// (x = hi + lo, lo the rounding residual of hi) and a product as
// hi*hi + hi*lo + lo*hi, which keeps about 16 bits of every operand: the
// solve then matches an fp32 one to ~3e-6 relative.
__device__ __forceinline__ void split_bf16(float x, float y, uint32_t& hi, uint32_t& lo) {
    const float hx = bf16_round(x), hy = bf16_round(y);
    hi = pack_bf16(hx, hy);
    lo = pack_bf16(x - hx, y - hy);
}
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// C (16 x 8NT) = A (16 x 16KS, row stride lda) B (16KS x 8NT, row stride
// ldb), one warp; lane (g, t) = (lane / 4, lane % 4) holds rows g, g + 8 and
// columns 2t, 2t + 1 of each 8-column tile (the m16n8k16 layouts).
template <int KS, int NT>
__device__ __forceinline__ void warp_gemm(float (&c)[NT][4], const float* A, int lda, const float* B, int ldb,
                                          int lane) {
    const int g = lane >> 2, t = lane & 3;
    float c1[NT][4], c2[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) c[nt][e] = c1[nt][e] = c2[nt][e] = 0.f;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
        uint32_t ah[4], al[4];
        const float* a0 = A + g * lda + 16 * ks + 2 * t;
        const float2 x0 = *reinterpret_cast<const float2*>(a0);
        const float2 x1 = *reinterpret_cast<const float2*>(a0 + 8 * lda);
        const float2 x2 = *reinterpret_cast<const float2*>(a0 + 8);
        const float2 x3 = *reinterpret_cast<const float2*>(a0 + 8 * lda + 8);
        split_bf16(x0.x, x0.y, ah[0], al[0]);
        split_bf16(x1.x, x1.y, ah[1], al[1]);
        split_bf16(x2.x, x2.y, ah[2], al[2]);
        split_bf16(x3.x, x3.y, ah[3], al[3]);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const float* b = B + (16 * ks + 2 * t) * ldb + 8 * nt + g;
            uint32_t bh0, bl0, bh1, bl1;
            split_bf16(b[0], b[ldb], bh0, bl0);
            split_bf16(b[8 * ldb], b[9 * ldb], bh1, bl1);
            mma16816(c1[nt], al, bh0, bh1);  // three accumulators: no chain through one register set
            mma16816(c2[nt], ah, bl0, bl1);
            mma16816(c[nt], ah, bh0, bh1);
        }
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) c[nt][e] += c1[nt][e] + c2[nt][e];
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

// (I + A)^-1 in place, A strictly lower triangular 64 x 64 (row stride kAS),
// by recursive doubling on the block-triangular inverse
//   [[L11, 0], [L21, L22]]^-1 = [[M11, 0], [-M22 L21 M11, M22]]:
//   level 1: the four 16 x 16 diagonal blocks, forward substitution by
//            columns (threads 0..63, one column each);
//   level 2: blocks (1,0) and (3,2), from the level-1 inverses (warps
//            w < 4: block pair w / 2, 8-column tile w % 2);
//   level 3: the lower-left 32 x 32 block, from the two 32 x 32 inverses
//            (warp w: 16 x 8 tile w of it).
// The products run over full blocks: the zero upper parts of the triangular
// factors make that exact.  Ptmp holds the left products.
__device__ void prep_solve(float* As, float* Ptmp, int p) {
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
    named_sync(1, kPrepThreads);
    {  // level 2: P = A_{x+1,x} M_xx, then M_{x+1,x} = -M_{x+1,x+1} P, x = 0, 2
        const int x = 2 * ((w >> 1) & 1), nt = w & 1;
        float* P = Ptmp + ((w >> 1) & 1) * 320;  // 16 x 16, row stride 20
        float c[1][4];
        if (w < 4) {
            warp_gemm<1, 1>(c, As + 16 * (x + 1) * kAS + 16 * x, kAS, As + 16 * x * kAS + 16 * x + 8 * nt, kAS, lane);
            warp_store<1>(c, P + 8 * nt, 20, 1.f, lane);
        }
        named_sync(1, kPrepThreads);
        if (w < 4) {
            warp_gemm<1, 1>(c, As + 16 * (x + 1) * kAS + 16 * (x + 1), kAS, P + 8 * nt, 20, lane);
            warp_store<1>(c, As + 16 * (x + 1) * kAS + 16 * x + 8 * nt, kAS, -1.f, lane);
        }
    }
    named_sync(1, kPrepThreads);
    {  // level 3: P = A[32:64, 0:32] M[0:32, 0:32], then M[32:64, 0:32] = -M[32:64, 32:64] P
        const int r0 = 16 * (w >> 2), c0 = 8 * (w & 3);
        float c[1][4];
        warp_gemm<2, 1>(c, As + (32 + r0) * kAS, kAS, As + c0, kAS, lane);
        warp_store<1>(c, Ptmp + r0 * 36 + c0, 36, 1.f, lane);  // 32 x 32, row stride 36
        named_sync(1, kPrepThreads);
        warp_gemm<2, 1>(c, As + (32 + r0) * kAS + 32, kAS, Ptmp + c0, 36, lane);
        warp_store<1>(c, As + (32 + r0) * kAS + c0, kAS, -1.f, lane);
    }
    named_sync(1, kPrepThreads);
}

// That Diag(up) (bf16 hi at bt, residual lo at bt + 16384; up = g / g_C^(1/2))
// and That = (I+A)^-1 Diag(b) (bf16 at bt + 8192) as K-major 64 x 64 operands
// (128-byte rows, 128-byte swizzle).  Thread p writes a quarter of a row.
__device__ void prep_write_that(const Misc* ms, const float* As, uint32_t bt, int par, int p) {
    const int t = p >> 2, qr = p & 3;
    const float* row = As + t * kAS + 16 * qr;
    const float* beta = ms->beta[par] + 16 * qr;
    const float* gam = ms->up[par] + 16 * qr;  // That Diag(g / g_C^(1/2))
#pragma unroll
    for (int ch = 0; ch < 2; ++ch) {
        const float4 x0 = *reinterpret_cast<const float4*>(row + 8 * ch);
        const float4 x1 = *reinterpret_cast<const float4*>(row + 8 * ch + 4);
        const float4 b0 = *reinterpret_cast<const float4*>(beta + 8 * ch);
        const float4 b1 = *reinterpret_cast<const float4*>(beta + 8 * ch + 4);
        const float4 y0 = *reinterpret_cast<const float4*>(gam + 8 * ch);
        const float4 y1 = *reinterpret_cast<const float4*>(gam + 8 * ch + 4);
        const float mv[8] = {x0.x * b0.x, x0.y * b0.y, x0.z * b0.z, x0.w * b0.w,
                             x1.x * b1.x, x1.y * b1.y, x1.z * b1.z, x1.w * b1.w};
        const float gv[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
        uint32_t w1[4], w2[4], w3[4];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            const float m0 = mv[2 * jj], m1 = mv[2 * jj + 1];
            const float z0 = m0 * gv[2 * jj], z1 = m1 * gv[2 * jj + 1];
            split2_bf16(z0, z1, w1[jj], w3[jj]);
            w2[jj] = pack_bf16(m0, m1);
        }
        const uint32_t off = t * 128u + ((uint32_t)((2 * qr + ch) ^ (t & 7)) << 4);
        st_shared_v4(bt + off, w1[0], w1[1], w1[2], w1[3]);
        st_shared_v4(bt + 8192u + off, w2[0], w2[1], w2[2], w2[3]);
        st_shared_v4(bt + 16384u + off, w3[0], w3[1], w3[2], w3[3]);
    }
}

// W^T (lane i holds W[.][i], staged in the X_S columns) -> W as a tf32
// K-major [64 t][128 i] operand.
__device__ void convert_w(uint8_t* smem, uint32_t tmem, int q, int lane) {
    const int i = 32 * q + lane;
    const uint32_t tl = tmem + ((32u * q) << 16);
    uint8_t* bw = smem + OFF_BW + (i >> 5) * 8192;
#pragma unroll 1
    for (int half = 0; half < 2; ++half) {
        uint32_t w[32];
        tmem_ld32(tl + TM_XS + 32 * half, w);
        tmem_wait_ld();
        uint8_t* b = bw + 32 * half * 128;
#pragma unroll
        for (int j = 0; j < 32; ++j)
            *reinterpret_cast<float*>(b + sw128_offset(j, i & 31, 4, 0)) = tf32_rna(__uint_as_float(w[j]));
    }
}

// ---------------------------------------------------------- state roles --
// Thread n of the state warpgroup owns tensor-memory lane n = 32q + lane:
// row n of D'_T (column n of T) and of D'_S (column n of S).

// D' <- (I, 0): row n of D'_T is e_n.
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

// D''_h <- sc D''_h in tensor memory (this thread's row), returning the max
// |.| of the new row when want_max: the rescale of a renormalisation chunk.
// (Rare: out of line, so that it stays out of the pass's instruction stream.)
__device__ __noinline__ float state_rescale(uint32_t addr, float sc, bool want_max) {
    float mloc = 0.f;
#pragma unroll 1
    for (int cb = 0; cb < 4; ++cb) {
        uint32_t x[32];
        tmem_ld32(addr + 32 * cb, x);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const float v = __uint_as_float(x[j]) * sc;
            if (want_max) mloc = fmaxf(mloc, fabsf(v));
            x[j] = __float_as_uint(v);
        }
        tmem_st32(addr + 32 * cb, x);
    }
    tmem_wait_st();
    return mloc;
}

// After GEMM1 of a chunk, half h (0 = T, 1 = S), the A operand of GEMM2:
//   Y''_T[n][t] = fT[t] X''_T[n][t] as bf16 hi + lo, written over X''_T in
//     tensor memory: lane n, tokens 16k..16k+15 in columns 16k..16k+7 (hi)
//     and 16k+8..16k+15 (lo), two tokens per column, so that each group of
//     16 columns is read and then rewritten in place;
//   Y''_S[n][t] = fS[t] X''_S[n][t] + uf[t] U^T[n][t] as bf16 into shared
//     memory (K-major [128 n][64 t]); the S half of GEMM2 multiplies both
//     terms by the same keys, so U~ rides in Y''_S, rounded once.
// On a renormalisation chunk the stored state is also rescaled in tensor
// memory, D''_T <- dT D''_T and D''_S <- dS D''_S, and the max |.| of the new
// T rows is returned (else 0).
template <int h>
__device__ float state_pass(const Misc* ms, uint32_t ay, bool rn, float dT, float dS, uint32_t tmem, int q,
                            int lane) {
    const int n = 32 * q + lane;
    const uint32_t tl = tmem + ((32u * q) << 16);
#pragma unroll 1
    for (int qt = 0; qt < 4; ++qt) {  // 16 columns (tokens) at a time
        const float* f = (h ? ms->fS : ms->fT) + 16 * qt;
        const float* uf = ms->uf + 16 * qt;
        uint32_t x[16], u[16];
        tmem_ld16(tl + (h ? TM_XS : TM_XT) + 16 * qt, x);
        if (h) tmem_ld16(tl + TM_U + 16 * qt, u);
        tmem_wait_ld();
        uint32_t hl[16];  // (T half: hi in [0, 8), lo in [8, 16))
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
            uint32_t pk[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int t = 8 * jj + 2 * k;
                float y0 = f[t] * __uint_as_float(x[t]);
                float y1 = f[t + 1] * __uint_as_float(x[t + 1]);
                if (h) {
                    y0 = fmaf(uf[t], __uint_as_float(u[t]), y0);
                    y1 = fmaf(uf[t + 1], __uint_as_float(u[t + 1]), y1);
                    pk[k] = pack_bf16(y0, y1);
                } else {
                    split2_bf16(y0, y1, hl[4 * jj + k], hl[8 + 4 * jj + k]);
                }
            }
            if (h) {
                const uint32_t off = n * 128u + ((uint32_t)((2 * qt + jj) ^ (n & 7)) << 4);
                st_shared_v4(ay + off, pk[0], pk[1], pk[2], pk[3]);
            }
        }
        if (!h) tmem_st16(tl + TM_XT + 16 * qt, hl);
    }
    if (!h) tmem_wait_st();
    return rn ? state_rescale(tl + (h ? TM_DS : TM_DT), h ? dS : dT, !h) : 0.f;
}

// Warp max, then the 4 warps of the state warpgroup through shared memory.
__device__ float state_reduce_max(float v, float* slot, int q, int lane) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (lane == 0) slot[q] = v;
    named_sync(2);
    return fmaxf(fmaxf(slot[0], slot[1]), fmaxf(slot[2], slot[3]));
}

// End of an item: T_C = mantissa * 2^exp with the mantissa's largest entry in
// [1, 2); S(C|0) as is.  Thread n writes column n (coalesced across the warp).
__device__ void state_epilogue(Misc* ms, const TcArgs& a, int64_t obj, int E, uint32_t tmem, int q, int lane) {
    const int n = 32 * q + lane;
    const uint32_t tl = tmem + ((32u * q) << 16);
    uint32_t x[32];
    float m = 0.f;
#pragma unroll 1
    for (int cb = 0; cb < 4; ++cb) {
        tmem_ld32(tl + TM_DT + 32 * cb, x);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) m = fmaxf(m, fabsf(__uint_as_float(x[j])));
    }
    m = state_reduce_max(m, ms->red_ep, q, lane);
    const int ef = (m > 0.f && m < INFINITY) ? ilogbf(m) : 0;
    float* T = a.T_out + obj * kD * kD;
    float* S = a.S_out + obj * kD * kD;
#pragma unroll 1
    for (int cb = 0; cb < 4; ++cb) {
        tmem_ld32(tl + TM_DT + 32 * cb, x);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) T[(32 * cb + j) * kD + n] = ldexpf(__uint_as_float(x[j]), -ef);
    }
#pragma unroll 1
    for (int cb = 0; cb < 4; ++cb) {
        tmem_ld32(tl + TM_DS + 32 * cb, x);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) S[(32 * cb + j) * kD + n] = __uint_as_float(x[j]);
    }
    if (n == 0) a.T_exp[obj] = E + ef;
}

// Empty body: the identity pair.
__device__ void state_identity(const TcArgs& a, int64_t obj, int n) {
    float* T = a.T_out + obj * kD * kD;
    float* S = a.S_out + obj * kD * kD;
    for (int i = 0; i < kD; ++i) {
        T[i * kD + n] = (i == n) ? 1.f : 0.f;
        S[i * kD + n] = 0.f;
    }
    if (n == 0) a.T_exp[obj] = 0;
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
// g: global chunk counter at the start of the item (barrier phases run on it
// across items); nc: chunks of this item's body.  Every barrier completes
// once per chunk (the ring and gate-slot barriers once per use of their slot).

// Warp 0: keys (3-deep ring) and values (one buffer) by TMA from lane 0, and
// the gate tables of each chunk from the whole warp (a chunk ahead of the
// prep warpgroup, the loads of the next chunk's gates in flight meanwhile).
__device__ void producer_role(Misc* ms, uint8_t* smem, const TcArgs& a, const CUtensorMap* tmk,
                              const CUtensorMap* tmv, uint32_t g, int nc, int layer, int head, int64_t b0, int64_t b1,
                              int lane) {
    float ra[2], rb[2];
    if (nc > 0) gate_load(a, layer, head, b0, b1, lane, ra, rb);
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
        // The slot of chunk gc was last read for chunk gc - 4, whose GEMM2
        // completed before that of gc - 3 (waited above).
        gate_tables(ms, gc % kGateSlots, ra, rb, lane);
        if (c + 1 < nc) gate_load(a, layer, head, b0 + (int64_t)(c + 1) * kC, b1, lane, ra, rb);
        __syncwarp();
        if (lane == 0) mbar_arrive(&ms->gready[gc % kGateSlots]);
        if (gc >= 1 && !wait_bar(&ms->emptyV, (gc - 1) & 1, ms, a)) return;
        if (lane == 0) {
            uint8_t* vt = smem + OFF_V;
            mbar_expect_tx(&ms->fullV, kTile);
            tma_load_3d(vt, tmv, &ms->fullV, 0, head, z);
            tma_load_3d(vt + 8192, tmv, &ms->fullV, 64, head, z);
        }
    }
}

// The MMA issuers.  W^T of the next chunk reuses the X''_S columns and waits
// only for the S half of this chunk's pass, so it runs while the pass does the
// T half.  A readiness test of a barrier's phase k is only made once its phase
// k - 1 is known to be complete (by an earlier test or an earlier item), so a
// parity test cannot mistake an old phase for a new one.

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

// Warp 1, one thread: the state chain's MMAs, each group as soon as its
// inputs are ready (a dataflow loop that tests barrier phases without
// blocking); priority W'^T, GEMM2, GEMM1 (T half).
__device__ void mma_role(Misc* ms, uint8_t* smem, const TcArgs& a, uint32_t tmem, uint32_t g, int nc) {
    if (nc == 0) return;
    const uint32_t sb = smem_u32(smem);
    const uint32_t bw = sb + OFF_BW, ay = sb + OFF_AY, bt = sb + OFF_BT;
    auto ktile = [&](uint32_t gc) { return sb + OFF_K + (gc % kKStages) * kTile; };
    int iw = 0, i1 = 0, i2 = 0;
    uint64_t t_idle = 0;
    while (i2 < nc) {
        bool any = false;
        if (iw < nc && i1 == iw) {  // W^T = K^T (That Diag(g))^T (hi + lo) into the X_S columns
            const uint32_t gc = g + iw;
            if (mbar_test(&ms->that_ready[gc & 1], (gc >> 1) & 1) &&
                (gc == 0 || mbar_test(&ms->xs_free, (gc - 1) & 1))) {  // the pass has read the previous X''_S
                tc_fence_after();
                const uint32_t btc = bt + (gc & 1) * kBT;
                const uint64_t a0 = sdesc_sw128(ktile(gc), 8192, 1024), bh = sdesc_sw128(btc, 0, 1024),
                               bl = sdesc_sw128(btc + 16384, 0, 1024);
#pragma unroll 2
                for (int k = 0; k < 4; ++k) {  // (a descriptor's address field counts 16-byte units)
                    mma_bf16_ss(tmem + TM_XS, a0 + 128 * k, bh + 2 * k, ID_WU, k > 0);
                    mma_bf16_ss(tmem + TM_XS, a0 + 128 * k, bl + 2 * k, ID_WU, true);
                }
                mma_commit(&ms->w_done);
                mma_commit(&ms->bt_free[gc & 1]);
                ++iw;
                any = true;
            }
        }
        if (i2 < i1) {  // GEMM2 (bf16): D''_T += Y''_T K (hi + lo, A in the X_T columns); D''_S += Y''_S K
            const uint32_t gc = g + i2;
            if (mbar_test(&ms->y_ready, gc & 1)) {
                tc_fence_after();
                const uint64_t b0 = sdesc_sw128(ktile(gc), 8192, 1024), ys = sdesc_sw128(ay, 0, 1024);
#pragma unroll 2
                for (int k = 0; k < 4; ++k) {
                    const uint64_t bk = b0 + 128 * k;
                    mma_bf16_ts(tmem + TM_DT, tmem + TM_XT + 16 * k, bk, ID_G2, true);
                    mma_bf16_ts(tmem + TM_DT, tmem + TM_XT + 16 * k + 8, bk, ID_G2, true);
                    mma_bf16_ss(tmem + TM_DS, ys + 2 * k, bk, ID_G2, true);
                }
                // (the gram of this K tile completed before That, hence before W'^T and this GEMM2)
                mma_commit(&ms->d_ready);
                mma_commit(&ms->emptyK[gc % kKStages]);
                ++i2;
                any = true;
            }
        }
        if (i1 < iw && i2 == i1) {  // GEMM1 (tf32), T half: X''_T = D''_T W^T, A = the state in tensor memory
            const uint32_t gc = g + i1;
            if (mbar_test(&ms->w_cvt, gc & 1) && (i1 == 0 || mbar_test(&ms->d_ready, (gc - 1) & 1))) {
                tc_fence_after();
                const uint64_t b0 = sdesc_sw128(bw, 0, 1024);
#pragma unroll 4  // (a measured balance of issue rate and code size)
                for (int k = 0; k < 16; ++k)
                    mma_tf32_ts(tmem + TM_XT, tmem + TM_DT + 8 * k, b0 + 512 * (k >> 2) + 2 * (k & 3), ID_G1, k > 0);
                mma_commit(&ms->x_done);
                ++i1;
                any = true;
            }
        }
        if (any) {  // (no sleep when idle: a sleeping issuer answers its barriers late)
            t_idle = 0;
        } else if ((t_idle = issuer_idle(ms, a, t_idle)) == 0) {
            return;
        }
    }
}

// Warp 14, one thread: GEMM1 of the S half (on the state chain), then the
// prep chain's U^T and gram.  Its commits cover only its own MMAs: every
// reader of their results waits on its barriers (x_done_s, u_done, g_done,
// and bt_free, which takes one commit from each issuer).
__device__ void mma_role2(Misc* ms, uint8_t* smem, const TcArgs& a, uint32_t tmem, uint32_t g, int nc) {
    if (nc == 0) return;
    const uint32_t sb = smem_u32(smem);
    const uint32_t bw = sb + OFF_BW, bt = sb + OFF_BT, vt = sb + OFF_V;
    int ig = 0, iu = 0, i1 = 0;
    uint64_t t_idle = 0;
    while (i1 < nc || ig < nc) {
        bool any = false;
        if (i1 < iu) {  // GEMM1 (tf32), S half: X''_S = D''_S W^T (the W^T staged in X_S has been converted)
            const uint32_t gc = g + i1;
            if (mbar_test(&ms->w_cvt, gc & 1) && (i1 == 0 || mbar_test(&ms->d_ready, (gc - 1) & 1))) {
                tc_fence_after();
                const uint64_t b0 = sdesc_sw128(bw, 0, 1024);
#pragma unroll 4
                for (int k = 0; k < 16; ++k)
                    mma_tf32_ts(tmem + TM_XS, tmem + TM_DS + 8 * k, b0 + 512 * (k >> 2) + 2 * (k & 3), ID_G1, k > 0);
                mma_commit(&ms->x_done_s);
                ++i1;
                any = true;
            }
        }
        if (iu < ig) {  // U^T = V^T That^T
            const uint32_t gc = g + iu;
            if (mbar_test(&ms->that_ready[gc & 1], (gc >> 1) & 1) && mbar_test(&ms->fullV, gc & 1) &&
                (gc == 0 || mbar_test(&ms->xs_free, (gc - 1) & 1))) {  // the S pass has read the previous U^T
                tc_fence_after();
                const uint64_t a0 = sdesc_sw128(vt, 8192, 1024), b0 = sdesc_sw128(bt + (gc & 1) * kBT + 8192, 0, 1024);
#pragma unroll 1
                for (int k = 0; k < 4; ++k) mma_bf16_ss(tmem + TM_U, a0 + 128 * k, b0 + 2 * k, ID_WU, k > 0);
                mma_commit(&ms->u_done);
                mma_commit(&ms->emptyV);
                mma_commit(&ms->bt_free[gc & 1]);
                ++iu;
                any = true;
            }
        }
        // G = K K^T (K-major view of the K tile, K = feature index, two 64-wide boxes); the gram of
        // chunk c + 3 waits until GEMM1 (S half) of chunk c is issued, so that it fills a gap of the
        // pipe (measured: one chunk less lookahead +0.7 %, two less +16 %)
        if (ig < nc && ig <= i1 + 2) {
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
        if (any) {
            t_idle = 0;
        } else if ((t_idle = issuer_idle(ms, a, t_idle)) == 0) {
            return;
        }
    }
}

// Warps 6-13: gram -> A -> (I + A)^-1 -> That, chunk after chunk.
__device__ void prep_role(Misc* ms, uint8_t* smem, const TcArgs& a, uint32_t tmem, uint32_t g, int nc, int p, int q,
                          int lane) {
    float* As = reinterpret_cast<float*>(smem + OFF_AS);
    float* Ptmp = reinterpret_cast<float*>(smem + OFF_PT);
    const uint32_t bt = smem_u32(smem) + OFF_BT;
    for (int c = 0; c < nc; ++c) {
        const uint32_t gc = g + c;
        const int slot = gc % kGateSlots;
        bool ok = wait_bar(&ms->gready[slot], (gc / kGateSlots) & 1, ms, a);
        ok = ok && wait_bar(&ms->g_done, gc & 1, ms, a);
        if (!wg_all(1, ok, kPrepThreads)) return;
        tc_fence_after();
        prep_arows(ms, As, slot, tmem, q, p >> 7, lane);
        tc_fence_before();
        named_sync(1, kPrepThreads);
        if (p == 0) mbar_arrive(&ms->g_read);
        prep_solve(As, Ptmp, p);
        // the buffer's previous That (chunk gc - 2) has been read (the buffer's phases are waited in order)
        if (!wg_all(1, gc < 2 || wait_bar(&ms->bt_free[gc & 1], ((gc >> 1) - 1) & 1, ms, a), kPrepThreads))
            return;
        prep_write_that(ms, As, bt + (gc & 1) * kBT, slot, p);
        fence_async_smem();
        named_sync(1, kPrepThreads);
        if (p == 0) mbar_arrive(&ms->that_ready[gc & 1]);
    }
}

// Lazy decay.  The true state is D = sigma_h D''_h per half (h = T, S); the
// stored D'' is not rescaled on an ordinary chunk: its decay g_C goes into
// sigma (sigma_T = 2^(E + lsT), sigma_S = 2^lsS), so that with g_t the
// in-chunk decay prefix and X''_h = D''_h W'^T,
//   D''_T += sum_t -(g_C^(1/2)/g_t) X''_T[:, t] k_t,
//   D''_S += sum_t -(g_C^(1/2)/g_t) X''_S[:, t] k_t + (1/(g_t sigma_S)) u_t k_t.
// A renormalisation chunk folds sigma back: D''_T <- 2^(lsT + lc - e) D''_T
// with e = ilogb(max |D''_T|) + floor(lsT + lc) (E += e), D''_S <- 2^(lsS + lc)
// D''_S, and the factors of that chunk carry the same scales.  It comes on an
// item's last chunk, every kRenormEvery chunks (which bounds how far T's
// stored magnitude drifts between exponent updates), when the chunk's own
// decay passes 2^-kLazyMax, and when sigma_S times the chunk's decay would pass
// 2^-(2 kLazyMax).  The largest factor of an ordinary chunk, U~'s
// 2^(-lg2_t - lsS), then stays below 2^(2 kLazyMax), and so does the growth
// of D''_S.  (Bounding sigma_S and the chunk decay by 2^-kLazyMax each, and
// renormalising every 8 chunks, gave the same bound with twice the
// renormalisations: 1.7 % slower.)
constexpr int kRenormEvery = 16;
constexpr float kLazyMax = 56.f;  // (2^112 x the state stays far inside float32 range)

struct StatePlan {
    bool rn;
    int e;
    float dT, dS, lc;
};

// The factor tables of chunk gc (threads n < 64 write entry n) and its plan.
__device__ __forceinline__ StatePlan state_plan(Misc* ms, uint32_t gc, bool last, int since, float lsT, float lsS,
                                                float m, int n) {
    const int slot = gc % kGateSlots;
    StatePlan pl;
    pl.lc = ms->lg2[slot][kC - 1];
    pl.rn = last || since + 1 >= kRenormEvery || lsS + pl.lc < -2.f * kLazyMax || pl.lc < -kLazyMax;
    pl.e = pl.rn ? ((m > 0.f && m < INFINITY) ? ilogbf(m) : 0) + (int)floorf(lsT + pl.lc) : 0;
    pl.dT = exp2f(lsT + pl.lc - (float)pl.e);
    pl.dS = exp2f(lsS + pl.lc);
    if (n < kC) {  // (W carries g_t / g_C^(1/2), so the Y factors carry g_C^(1/2) / g_t)
        const float l = ms->lg2[slot][n], h = 0.5f * pl.lc;
        if (pl.rn) {
            ms->fT[n] = -exp2f(fminf(lsT + pl.lc - (float)pl.e + h - l, 126.f));
            ms->fS[n] = -exp2f(fminf(lsS + pl.lc + h - l, 126.f));
            ms->uf[n] = exp2f(pl.lc - l);
        } else {
            const float r = ms->wn[slot][n];
            ms->fT[n] = -r;
            ms->fS[n] = -r;
            ms->uf[n] = exp2f(-l - lsS);
        }
    }
    return pl;
}

// Chunk gc's factor tables and plan, then its W operand (on the chain to
// GEMM1).
__device__ __forceinline__ bool state_prepare(Misc* ms, uint8_t* smem, const TcArgs& a, uint32_t tmem, uint32_t gc,
                                              bool last, int since, float lsT, float lsS, float m, int q, int lane,
                                              StatePlan& pl) {
    const int slot = gc % kGateSlots;
    bool ok = wait_bar(&ms->gready[slot], (gc / kGateSlots) & 1, ms, a);
    if (!wg_all(2, ok)) return false;  // (and every thread is past the previous pass)
    pl = state_plan(ms, gc, last, since, lsT, lsS, m, 32 * q + lane);
    if (!wg_all(2, wait_bar(&ms->w_done, gc & 1, ms, a))) return false;  // (also publishes the factor tables)
    tc_fence_after();
    convert_w(smem, tmem, q, lane);
    fence_async_smem();
    tc_fence_before();
    named_sync(2);
    if (q == 0 && lane == 0) mbar_arrive(&ms->w_cvt);
    return true;
}

// Warps 2-5: per chunk the pass (Y'' and, on renormalisation chunks, the
// state rescale), then the next chunk's operands; the epilogue at the end.
__device__ void state_role(Misc* ms, uint8_t* smem, const TcArgs& a, uint32_t tmem, uint32_t g, int nc,
                           int64_t obj, int q, int lane) {
    const int n = 32 * q + lane;
    if (nc == 0) {
        state_identity(a, obj, n);
        return;
    }
    const uint32_t ay = smem_u32(smem) + OFF_AY;
    int E = 0, since = 0;
    float m = 1.f, lsT = 0.f, lsS = 0.f;
    StatePlan pl;
    // Step c runs the pass of chunk c - 1 (none for c = 0), then prepares
    // chunk c (none for c = nc): one call site per stage keeps the code small.
    for (int c = 0; c <= nc; ++c) {
        const uint32_t gc = g + c;
        if (c > 0) {
            const uint32_t gp = gc - 1;
            bool ok = wait_bar(&ms->x_done_s, gp & 1, ms, a);
            ok = ok && wait_bar(&ms->u_done, gp & 1, ms, a);
            if (!wg_all(2, ok)) return;
            tc_fence_after();
            state_pass<1>(ms, ay, pl.rn, pl.dT, pl.dS, tmem, q, lane);
            tc_fence_before();
            named_sync(2);  // every lane has read X''_S and U^T: the next W'^T and U^T may overwrite them
            if (n == 0) mbar_arrive(&ms->xs_free);
            if (!wg_all(2, wait_bar(&ms->x_done, gp & 1, ms, a))) return;
            tc_fence_after();
            const float mloc = state_pass<0>(ms, ay, pl.rn, pl.dT, pl.dS, tmem, q, lane);
            fence_async_smem();
            tc_fence_before();
            if (pl.rn) {
                m = state_reduce_max(mloc, ms->red[gp & 1], q, lane);
                E += pl.e;
                lsT = 0.f;
                lsS = 0.f;
                since = 0;
            } else {
                named_sync(2);
                lsT += pl.lc;
                lsS += pl.lc;
                ++since;
            }
            if (n == 0) mbar_arrive(&ms->y_ready);
        }
        if (c < nc && !state_prepare(ms, smem, a, tmem, gc, c + 1 == nc, since, lsT, lsS, m, q, lane, pl)) return;
    }
    if (!wg_all(2, wait_bar(&ms->d_ready, (g + nc - 1) & 1, ms, a))) return;
    tc_fence_after();
    state_epilogue(ms, a, obj, E, tmem, q, lane);
    state_init(tmem, q, lane);  // (I, 0) for the next item
}

// Producer, lane 0: the k-th item of this CTA into slot s (nc = -1 once the
// queue is exhausted or the CTA aborted); the slot's previous item has been
// copied by every reader.  Items are (segment, layer, head), segments in
// longest-body-first order.
__device__ __forceinline__ void publish_item(Misc* ms, const TcArgs& a, int k, int s) {
    const int LH = a.n_layers * a.n_heads;
    const ItemSlot& prev = ms->slots[(s + kItemSlots - 1) % kItemSlots];
    const uint32_t g = k == 0 ? 0u : prev.g + (uint32_t)(prev.nc > 0 ? prev.nc : 0);
    const int item = *(volatile int*)&ms->abort_flag ? a.n_items : (int)atomicAdd(a.counter, 1u);
    ItemSlot& it = ms->slots[s];
    if (item >= a.n_items) {
        it.nc = -1;
    } else {
        const int pos = item / LH, lh = item % LH;
        const int seg = a.order[pos];
        it.layer = lh / a.n_heads;
        it.head = lh % a.n_heads;
        it.b0 = (int64_t)a.cu[seg] + (a.skip ? a.skip[seg] : 0);
        it.b1 = a.cu[seg + 1];
        it.nc = (int)((it.b1 - it.b0 + kC - 1) / kC);
        it.obj = ((int64_t)seg * a.n_layers + it.layer) * a.n_heads + it.head;
        it.g = g;
    }
    mbar_arrive(&ms->slot_full[s]);  // (release: the slot is visible to the readers that wait on it)
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
            mbar_init(&ms->emptyK[s], 1);
        }
        // fullV .. drain (gready included) are consecutive in Misc: one arrival each, but bt_free (both
        // issuers read That) and drain (both issuers' MMAs) take two
        for (uint64_t* b = &ms->fullV; b <= &ms->drain; ++b)
            mbar_init(b, b == &ms->bt_free[0] || b == &ms->bt_free[1] || b == &ms->drain ? 2 : 1);
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
    if (warp == kWarpMMA) tmem_alloc(&ms->tmem_base, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ms->tmem_base;
    const bool is_state = warp >= kWarpState0 && warp < kWarpState0 + 4;
    const int q = warp & 3;  // tensor-memory lane quarter a warp may access
    if (is_state) state_init(tmem, q, lane);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // Every role runs through the items at its own pace: the producer takes
    // them from the queue into a ring of kItemSlots slots, and the other roles
    // copy them from there, so the next item's loads, gram, solve and W'^T
    // overlap this item's last chunks and epilogue.  Across items the roles
    // meet on the same barriers as within one (chunks are numbered CTA-wide).
    for (int k = 0;; ++k) {
        const int s = k % kItemSlots;
        ItemSlot it;
        if (warp == kWarpTMA) {
            if (k >= kItemSlots && !wait_bar(&ms->slot_read[s], (k / kItemSlots - 1) & 1, ms, a)) break;
            if (lane == 0) publish_item(ms, a, k, s);
            __syncwarp();
            it = ms->slots[s];
        } else {
            const bool one = warp == kWarpMMA || warp == kWarpMMA2;
            if (one && lane != 0) break;
            const int id = is_state ? 2 : 1, cnt = is_state ? 128 : kPrepThreads;
            const bool ok = wait_bar(&ms->slot_full[s], (k / kItemSlots) & 1, ms, a);
            if (one ? !ok : !wg_all(id, ok, cnt)) break;
            it = ms->slots[s];
            if (!one) named_sync(id, cnt);
            if (one || (tid & (cnt - 1)) == ((32 * (is_state ? kWarpState0 : kWarpPrep0)) & (cnt - 1)))
                mbar_arrive(&ms->slot_read[s]);
        }
        if (it.nc < 0) break;
        if (warp == kWarpTMA) {
            producer_role(ms, smem, a, &tmk, &tmv, it.g, it.nc, it.layer, it.head, it.b0, it.b1, lane);
        } else if (warp == kWarpMMA) {
            mma_role(ms, smem, a, tmem, it.g, it.nc);
        } else if (warp == kWarpMMA2) {
            mma_role2(ms, smem, a, tmem, it.g, it.nc);
        } else if (is_state) {
            state_role(ms, smem, a, tmem, it.g, it.nc, it.obj, q, lane);
        } else {
            prep_role(ms, smem, a, tmem, it.g, it.nc, tid - 32 * kWarpPrep0, q, lane);
        }
        if (*(volatile int*)&ms->abort_flag) break;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // Drain: every MMA this CTA issued (from both issuers) has completed before tensor memory is freed.
    if (warp == kWarpMMA || warp == kWarpMMA2) {
        if (lane == 0) {
            mma_commit(&ms->drain);
            for (uint32_t i = 0; i < a.wait_limit && !mbar_try_wait(&ms->drain, 0); ++i) {
            }
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
