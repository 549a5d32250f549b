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
// split again into the next step's A.  The state never leaves the SM until
// the chain ends; the HBM traffic is the pair stream, 128 KB per step.
//
// Roles (320 threads): warp 0 TMA producer, warp 1 MMA issuer, warps 2-5
// split the T slices (hi in place, lo beside it), warps 6-9 the epilogue.
// One CTA per SM, persistent over (chain, layer, head) items ordered
// (layer, head)-major so that chains sharing a pair table run together.
#include <cuda.h>
#include <cuda_runtime.h>
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
constexpr uint32_t OFF_MISC = OFF_SP + 4 * kSliceBytes;

struct Misc {
    uint64_t full[kRing], cvt[kRing], empty[kRing];
    uint64_t sp_full, sp_empty, d_done, a_ready, drain;
    int item;
    int abort_flag;
    uint32_t tmem_base;
};
constexpr uint32_t kSmemBytes = OFF_MISC + sizeof(Misc);
static_assert(kSmemBytes <= 232448, "shared memory budget");

constexpr uint32_t TM_D = 0, TM_AB = 128, TM_AS = 256;  // accumulator, A hi, A lo
constexpr uint32_t ID_T = idesc(2, 128, 128, false, false);

struct CtArgs {
    int n_layers, n_heads, n_pairs, n_chains, n_items;
    const int32_t* T_exp;
    const int32_t* cu_chain;
    const int32_t* seg_idx;
    const float* S0;
    float* S_out;
    unsigned* counter;
    unsigned* err;
    uint32_t wait_limit;
};

__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, Misc* ms, const CtArgs& a) {
    for (uint32_t i = 0; i < a.wait_limit; i += 256) {
        for (int j = 0; j < 256; ++j)
            if (mbar_try_wait(bar, parity)) return true;
        if (*(volatile int*)&ms->abort_flag) return false;
    }
    *(volatile int*)&ms->abort_flag = 1;
    set_error(a.err, kErrTimeout);
    return false;
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
                              const CUtensorMap* tmS, uint32_t gs, uint32_t gj, int c0, int len, int lh) {
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
        const uint32_t g = gj + j;
        if (g >= 1 && !wait_bar(&ms->sp_empty, (g - 1) & 1, ms, a)) return;
        mbar_expect_tx(&ms->sp_full, 4 * kSliceBytes);
        for (int b = 0; b < 4; ++b) tma_load_2d(smem + OFF_SP + b * kSliceBytes, tmS, &ms->sp_full, 32 * b, row);
    }
}

__device__ void mma_role(Misc* ms, uint8_t* smem, const CtArgs& a, uint32_t tmem, uint32_t gs, uint32_t gj, int len) {
    const uint32_t ring = smem_u32(smem) + OFF_RING;
    for (int j = 0; j < len; ++j) {
        if (!wait_bar(&ms->a_ready, (gj + j) & 1, ms, a)) return;
        tc_fence_after();
        for (int s = 0; s < kSlices; ++s) {
            const uint32_t gsi = gs + kSlices * j + s, buf = gsi % kRing;
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
    }
}

// Split each T slice into hi (in place) and lo (beside it).  t: 0..127.
__device__ void convert_role(Misc* ms, uint8_t* smem, const CtArgs& a, uint32_t gs, int len, int t) {
    for (int j = 0; j < len; ++j) {
        for (int s = 0; s < kSlices; ++s) {
            const uint32_t gsi = gs + kSlices * j + s, buf = gsi % kRing;
            if (!wg_all(3, wait_bar(&ms->full[buf], (gsi / kRing) & 1, ms, a))) return;
            uint8_t* hi = smem + OFF_RING + buf * 2 * kSliceBytes;
            uint8_t* lo = hi + kSliceBytes;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint32_t off = k * 2048 + t * 16;
                const float4 x = *reinterpret_cast<const float4*>(hi + off);
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
    }
}

// Epilogue: thread n owns TMEM lane n = column n of the state.
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
    // A for the first step: the start state (column n), split hi/lo.
#pragma unroll
    for (int cb = 0; cb < 4; ++cb) {
        uint32_t h[32], l[32];
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) split_tf32(s0 ? s0[(32 * cb + jj) * kD + n] : 0.f, h[jj], l[jj]);
        tmem_st32(tl + TM_AB + 32 * cb, h);
        tmem_st32(tl + TM_AS + 32 * cb, l);
    }
    tmem_wait_st();
    tc_fence_before();
    named_sync(4);
    if (n == 0) mbar_arrive(&ms->a_ready);
    const float* sp = reinterpret_cast<const float*>(smem + OFF_SP) + (n >> 5) * (kSliceBytes / 4) + (n & 31);
    for (int j = 0; j < len; ++j) {
        const uint32_t g = gj + j;
        const int p = a.seg_idx[c0 + j];
        const int e = a.T_exp ? a.T_exp[p * LH + lh] : 0;
        bool ok = wait_bar(&ms->d_done, g & 1, ms, a);
        ok = ok && wait_bar(&ms->sp_full, g & 1, ms, a);
        if (!wg_all(4, ok)) return;
        tc_fence_after();
        const bool last = j + 1 == len;
#pragma unroll
        for (int cb = 0; cb < 4; ++cb) {
            uint32_t x[32];
            tmem_ld32(tl + TM_D + 32 * cb, x);
            tmem_wait_ld();
            uint32_t h[32], l[32];
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
                const int i = 32 * cb + jj;
                const float v = ldexpf(__uint_as_float(x[jj]), e) + sp[i * 32];
                if (last) out[i * kD + n] = v;
                else split_tf32(v, h[jj], l[jj]);
            }
            if (!last) {
                tmem_st32(tl + TM_AB + 32 * cb, h);
                tmem_st32(tl + TM_AS + 32 * cb, l);
            }
        }
        tmem_wait_st();
        tc_fence_before();
        named_sync(4);
        if (n == 0) {
            mbar_arrive(&ms->sp_empty);
            if (!last) mbar_arrive(&ms->a_ready);
        }
    }
}

// ---------------------------------------------------------------- kernel --
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
        mbar_init(&ms->a_ready, 1);
        mbar_init(&ms->drain, 1);
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
    uint32_t gs = 0, gj = 0;
    for (int item = blockIdx.x; item < a.n_items; item += gridDim.x) {
        if (*(volatile int*)&ms->abort_flag) break;
        const int lh = item / a.n_chains, chain = item % a.n_chains;
        const int c0 = a.cu_chain[chain], len = a.cu_chain[chain + 1] - c0;
        const int64_t obj = (int64_t)chain * LH + lh;
        if (warp == kWarpTMA) {
            if (lane == 0) producer_role(ms, smem, a, &tmT, &tmS, gs, gj, c0, len, lh);
        } else if (warp == kWarpMMA) {
            if (lane == 0) mma_role(ms, smem, a, tmem, gs, gj, len);
        } else if (warp < kWarpEpi0) {
            convert_role(ms, smem, a, gs, len, tid - 32 * kWarpCvt0);
        } else {
            epilogue_role(ms, smem, a, tmem, gj, c0, len, lh, obj, warp & 3, lane);
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        gs += kSlices * len;
        gj += len;
    }
    if (warp == kWarpMMA) {
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
    return p.family == kGDN && p.dk == kD && p.dv == kD && p.n_pairs > 0 &&
           (int64_t)p.n_pairs * p.n_layers * p.n_heads * kD < INT32_MAX && encode_fn() != nullptr;
}

cudaError_t launch_compose_tc(const ComposeParams& p, unsigned* err, cudaStream_t s) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    const uint64_t rows = (uint64_t)p.n_pairs * p.n_layers * p.n_heads * kD;
    CUtensorMap tT, tS;
    if (!make_map(enc, &tT, p.T_tab, rows, true) || !make_map(enc, &tS, p.S_tab, rows, false))
        return cudaErrorInvalidValue;
    CtArgs a;
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
    a.counter = nullptr;
    a.err = err;
    a.wait_limit = 1u << 26;
    if (a.n_items == 0) return cudaSuccess;
    const int sms = sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    cudaError_t e = cudaFuncSetAttribute(compose_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    const int grid = a.n_items < sms ? a.n_items : sms;
    compose_tc_kernel<<<grid, kThreads, kSmemBytes, s>>>(tT, tS, a);
    return cudaGetLastError();
}

}  // namespace hypic
