// kernels.h -- internal interface between the C ABI (api.cu) and the kernels.
// Arguments reaching these launchers have already been validated on the host.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace hypic {

struct BuildParams {
    int family, in_dtype, n_layers, n_heads, dk, dv, n_seg;
    int64_t n_tokens;
    const int32_t* cu;    // [n_seg+1]
    const int32_t* skip;  // [n_seg] or null
    const int32_t* cu_host = nullptr;    // host copies of cu and skip (batch planning)
    const int32_t* skip_host = nullptr;
    const void* k;
    const void* v;
    const float* alpha;
    const float* beta;
    const float* gamma;
    const float* g;
    float* T_out;
    int32_t* T_exp;
    float* S_out;
};

struct ComposeParams {
    int family, n_layers, n_heads, dk, dv, n_pairs, n_chains;
    const float* T_tab;
    const int32_t* T_exp_tab;
    const float* S_tab;
    const int32_t* cu_chain;
    const int32_t* seg_idx;
    const float* S0;
    float* S_out;
    float* T_out = nullptr;        // optional: each chain's own transition (T_chain)
    int32_t* T_exp_out = nullptr;  // its exponent (dense families)
};

struct SeamParams {
    int family, in_dtype, n_layers, n_heads, dk, dv, n_seams;
    int64_t n_tokens;
    const int32_t* cu_seam;
    const void* q;
    const void* k;
    const void* v;
    const float* alpha;
    const float* beta;
    const float* gamma;
    const float* g;
    const float* state_in;
    float* state_out;
    float* o_out;
};

// Workspace layout of the build: [order: n_seg int32][pad to 256 B][counter: 256 B].
size_t build_workspace_bytes(int n_seg);

// Sort segments by body length, longest first (ties: lower index first), into
// `order`, and zero the work counter.
cudaError_t launch_build_plan(const BuildParams& p, void* workspace, cudaStream_t s);

// Token-loop build on CUDA cores (every family, every supported d).
cudaError_t launch_build_simt(const BuildParams& p, const void* workspace, unsigned* err, cudaStream_t s);

// Chunked GDN build on the tensor cores (d = 128, bf16 k/v).  Returns
// cudaErrorNotSupported when the shape is not covered.
cudaError_t launch_gdn_build_tc(const BuildParams& p, void* workspace, unsigned* err, cudaStream_t s);
bool gdn_build_tc_supported(const BuildParams& p);

// The decay families (RetNet, Mamba2, GLA, vanilla) on the tensor cores (d =
// 128, bf16 k/v): the closed form S = sum_t Diag(w_t) k_t v_t^T as a
// contraction.  Returns cudaErrorNotSupported when the shape is not covered.
cudaError_t launch_decay_build_tc(const BuildParams& p, void* workspace, unsigned* err, cudaStream_t s);
bool decay_build_tc_supported(const BuildParams& p);

// KDA (d = 128, bf16 k/v) on the tensor cores: every 64-token chunk's own pair,
// then the chunk pairs of each segment chained by the tensor-core compose.
// The chunk tables live in the workspace, whose size kda_build_tc_workspace_bytes
// reports (segments are taken in batches whose tables fit it).
bool kda_build_tc_supported(const BuildParams& p);
size_t kda_build_tc_workspace_bytes(const BuildParams& p);
cudaError_t launch_kda_build_tc(const BuildParams& p, void* workspace, size_t workspace_bytes, unsigned* err,
                                cudaStream_t s);

cudaError_t launch_compose(const ComposeParams& p, unsigned* err, cudaStream_t s);
cudaError_t launch_compose_simt(const ComposeParams& p, unsigned* err, cudaStream_t s);
cudaError_t launch_compose_tc(const ComposeParams& p, unsigned* err, cudaStream_t s);
bool compose_tc_supported(const ComposeParams& p);
cudaError_t launch_seam(const SeamParams& p, unsigned* err, cudaStream_t s);

// Reuse chain: the compose chain of `c` with, before step j, a seam advance
// over the seam tokens [cu_step[j], cu_step[j+1]) (layouts as SeamParams).
struct ChainParams {
    ComposeParams c;
    int in_dtype;
    int64_t n_tokens;
    const int32_t* cu_step;
    const void* q;
    const void* k;
    const void* v;
    const float* alpha;
    const float* beta;
    float* o_out;
};
// GDN, d = 128: one fused tensor-core kernel (state on chip for the whole chain).
bool chain_tc_supported(const ChainParams& p);
cudaError_t launch_chain_tc(const ChainParams& p, unsigned* err, cudaStream_t s);

// State re-rotation of cached pairs (rope.cu), in place.
struct RopeParams {
    int n_layers, n_heads, dk, dv, n_pairs, rotary_dim;
    double base;
    const int64_t* delta;  // [n_pairs] position shift
    float* T;              // [n_pairs][L][H][dk][dk] (dense families) or nullptr
    float* S;              // [n_pairs][L][H][dk][dv]
};
cudaError_t launch_rope(const RopeParams& p, cudaStream_t s);

// Conv-state warm-up of seam windows (conv.cu).
struct ConvParams {
    int n_layers, C, K, n_seams, act;
    int64_t n_tokens;
    const int32_t* cu_seam;
    const float* x;     // [L][n_tokens][C]
    const float* hist;  // [n_seams][L][K-1][C] or nullptr
    const float* w;     // [L][C][K]
    const float* bias;  // [L][C] or nullptr
    float* y;           // [L][n_tokens][C]
};
cudaError_t launch_conv_warmup(const ConvParams& p, cudaStream_t s);

}  // namespace hypic
