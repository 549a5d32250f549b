// api.cu -- the C ABI of libhypic.so (declared in include/hypic.h): host-side
// argument checks, work dispatch and error reporting.  No call allocates
// memory; all checks happen before the first launch.
#include <cuda_runtime.h>
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>

#include "../../include/hypic.h"
#include "common.cuh"
#include "kernels.h"

namespace hypic {
cudaError_t launch_compose_simt(const ComposeParams& p, unsigned* err, cudaStream_t s);
cudaError_t launch_compose_tc(const ComposeParams& p, unsigned* err, cudaStream_t s);
bool compose_tc_supported(const ComposeParams& p);
}  // namespace hypic

using namespace hypic;

// Device error word: set (first writer wins) by kernels whose bounded waits
// ran out; read and cleared by hypic_check_device().
__device__ unsigned g_hypic_err_word;

namespace {

thread_local char t_detail[512] = "";

hypic_status fail(hypic_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_detail, sizeof(t_detail), fmt, ap);
    va_end(ap);
    return st;
}

hypic_status cuda_fail(cudaError_t e, const char* where) {
    return fail(HYPIC_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

// Address of the device error word on the current device.  Host code cannot
// take the address of a __device__ variable itself, so it is looked up on every
// call (a cheap host-side query): an address cached per device ordinal would go
// stale once the device's primary context is reset and the module reloaded.
unsigned* err_word(cudaError_t* e_out) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_hypic_err_word);
    *e_out = e;
    return e == cudaSuccess ? static_cast<unsigned*>(p) : nullptr;
}

bool dim_ok(int d) { return d == 16 || d == 32 || d == 64 || d == 128; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// [a, a + na) and [b, b + nb) (bytes) share a byte.
bool overlap(const void* a, size_t na, const void* b, size_t nb) {
    if (!a || !b || !na || !nb) return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

const char* fam_name(int f) {
    static const char* n[] = {"GDN", "RETNET", "GLA", "VANILLA", "KDA", "MAMBA2"};
    return (f >= 0 && f <= 5) ? n[f] : "?";
}

// T_C is a dense dk x dk matrix (stored with an exponent) / a scalar.
bool dense_T(int family) { return family == HYPIC_GDN || family == HYPIC_KDA; }

// Checks shared by the three calls: family, dtype, dims and the family's
// gate pointers.  `has_tokens` is false when no token is read.
hypic_status check_family(int family, int in_dtype, int n_layers, int n_heads, int dk, int dv, bool has_tokens,
                          const float* alpha, const float* beta, const float* gamma, const float* g,
                          bool check_dtype) {
    if (family < HYPIC_GDN || family > HYPIC_MAMBA2) return fail(HYPIC_ERR_INVALID_ARG, "family %d", family);
    if (check_dtype && in_dtype != HYPIC_F32 && in_dtype != HYPIC_BF16)
        return fail(HYPIC_ERR_INVALID_ARG, "in_dtype %d", in_dtype);
    if (n_layers < 1 || n_heads < 1) return fail(HYPIC_ERR_INVALID_ARG, "n_layers %d n_heads %d", n_layers, n_heads);
    if (dk < 1 || dv < 1) return fail(HYPIC_ERR_INVALID_ARG, "dk %d dv %d", dk, dv);
    if (!dim_ok(dk) || !dim_ok(dv))
        return fail(HYPIC_ERR_UNSUPPORTED, "dk %d dv %d (supported: 16, 32, 64, 128)", dk, dv);
    if (dense_T(family) && dk != dv)
        return fail(HYPIC_ERR_UNSUPPORTED, "%s needs dk == dv (%d, %d)", fam_name(family), dk, dv);
    const bool want_alpha = family == HYPIC_GDN || family == HYPIC_MAMBA2;
    const bool want_beta = family == HYPIC_GDN || family == HYPIC_KDA;
    const bool want_gamma = family == HYPIC_RETNET, want_g = family == HYPIC_GLA || family == HYPIC_KDA;
    if (!want_alpha && alpha) return fail(HYPIC_ERR_INVALID_ARG, "alpha must be NULL for %s", fam_name(family));
    if (!want_beta && beta) return fail(HYPIC_ERR_INVALID_ARG, "beta must be NULL for %s", fam_name(family));
    if (!want_gamma && gamma) return fail(HYPIC_ERR_INVALID_ARG, "gamma must be NULL for %s", fam_name(family));
    if (!want_g && g) return fail(HYPIC_ERR_INVALID_ARG, "g must be NULL for %s", fam_name(family));
    if (has_tokens) {  // gates are read only when tokens are
        if (want_alpha && !alpha) return fail(HYPIC_ERR_INVALID_ARG, "%s needs alpha", fam_name(family));
        if (want_beta && !beta) return fail(HYPIC_ERR_INVALID_ARG, "%s needs beta", fam_name(family));
        if (want_gamma && !gamma) return fail(HYPIC_ERR_INVALID_ARG, "RETNET needs gamma");
        if (want_g && !g) return fail(HYPIC_ERR_INVALID_ARG, "%s needs g", fam_name(family));
    }
    const void* ptrs[] = {alpha, beta, gamma, g};
    for (const void* q : ptrs)
        if (q && !aligned16(q)) return fail(HYPIC_ERR_INVALID_ARG, "gate pointer %p not 16-byte aligned", q);
    return HYPIC_OK;
}

}  // namespace

// ------------------------------------------------------------------ build --

namespace {

hypic_status check_build(const hypic_build_args* a) {
    if (!a) return fail(HYPIC_ERR_INVALID_ARG, "args is NULL");
    if (a->n_segments < 0) return fail(HYPIC_ERR_INVALID_ARG, "n_segments %d", a->n_segments);
    if (a->n_tokens < 0 || a->n_tokens > INT32_MAX)
        return fail(HYPIC_ERR_INVALID_ARG, "n_tokens %lld", (long long)a->n_tokens);
    if (!a->cu_seqlens || !a->cu_seqlens_host) return fail(HYPIC_ERR_INVALID_ARG, "cu_seqlens (device and host) required");
    if ((a->seam_skip == nullptr) != (a->seam_skip_host == nullptr))
        return fail(HYPIC_ERR_INVALID_ARG, "seam_skip and seam_skip_host must both be set or both NULL");
    const int32_t* cu = a->cu_seqlens_host;
    if (cu[0] < 0) return fail(HYPIC_ERR_INVALID_ARG, "cu_seqlens[0] = %d", cu[0]);
    for (int s = 0; s < a->n_segments; ++s) {
        if (cu[s + 1] < cu[s]) return fail(HYPIC_ERR_INVALID_ARG, "cu_seqlens decreases at %d", s);
        if (a->seam_skip_host) {
            const int sk = a->seam_skip_host[s];
            if (sk < 0 || sk > cu[s + 1] - cu[s])
                return fail(HYPIC_ERR_INVALID_ARG, "seam_skip[%d] = %d outside [0, %d]", s, sk, cu[s + 1] - cu[s]);
        }
    }
    if ((int64_t)cu[a->n_segments] > a->n_tokens)
        return fail(HYPIC_ERR_INVALID_ARG, "cu_seqlens[n_segments] = %d > n_tokens %lld", cu[a->n_segments],
                    (long long)a->n_tokens);
    const bool has_tokens = cu[a->n_segments] > cu[0];
    hypic_status st = check_family(a->family, a->in_dtype, a->n_layers, a->n_heads, a->dk, a->dv, has_tokens, a->alpha,
                                   a->beta, a->gamma, a->g, true);
    if (st != HYPIC_OK) return st;
    if (has_tokens && (!a->k || !a->v)) return fail(HYPIC_ERR_INVALID_ARG, "k and v required");
    const bool any = a->n_segments > 0;
    if (any && !a->S_out) return fail(HYPIC_ERR_INVALID_ARG, "S_out required");
    const bool want_T = a->family != HYPIC_VANILLA, want_exp = dense_T(a->family);
    if (!want_T && a->T_out) return fail(HYPIC_ERR_INVALID_ARG, "T_out must be NULL for VANILLA");
    if (!want_exp && a->T_exp_out) return fail(HYPIC_ERR_INVALID_ARG, "T_exp_out must be NULL for %s", fam_name(a->family));
    if (any && want_T && !a->T_out) return fail(HYPIC_ERR_INVALID_ARG, "T_out required for %s", fam_name(a->family));
    if (any && want_exp && !a->T_exp_out)
        return fail(HYPIC_ERR_INVALID_ARG, "T_exp_out required for %s", fam_name(a->family));
    const void* ptrs[] = {a->k, a->v, a->T_out, a->T_exp_out, a->S_out};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return fail(HYPIC_ERR_INVALID_ARG, "pointer %p not 16-byte aligned", p);
    return HYPIC_OK;
}

BuildParams to_params(const hypic_build_args* a) {
    BuildParams p;
    p.family = a->family;
    p.in_dtype = a->in_dtype;
    p.n_layers = a->n_layers;
    p.n_heads = a->n_heads;
    p.dk = a->dk;
    p.dv = a->dv;
    p.n_seg = a->n_segments;
    p.n_tokens = a->n_tokens;
    p.cu = a->cu_seqlens;
    p.skip = a->seam_skip;
    p.cu_host = a->cu_seqlens_host;
    p.skip_host = a->seam_skip_host;
    p.k = a->k;
    p.v = a->v;
    p.alpha = a->alpha;
    p.beta = a->beta;
    p.gamma = a->gamma;
    p.g = a->g;
    p.T_out = a->T_out;
    p.T_exp = a->T_exp_out;
    p.S_out = a->S_out;
    return p;
}

}  // namespace

extern "C" size_t hypic_build_workspace_size(const hypic_build_args* args) {
    if (check_build(args) != HYPIC_OK) return 0;
    const BuildParams p = to_params(args);
    if (args->n_segments > 0 && kda_build_tc_supported(p)) return kda_build_tc_workspace_bytes(p);
    return build_workspace_bytes(args->n_segments);
}

namespace hypic {
// The build with `tables` = false needs only the plan and counter in its
// workspace: KDA then runs its CUDA-core kernel (the no-alloc build).
hypic_status segment_build_impl(const hypic_build_args* args, void* workspace, size_t workspace_bytes,
                                hypic_stream_t stream, bool tables) {
    hypic_status st = check_build(args);
    if (st != HYPIC_OK) return st;
    if (args->n_segments == 0) return HYPIC_OK;
    const size_t need = tables ? hypic_build_workspace_size(args) : build_workspace_bytes(args->n_segments);
    if (!workspace || workspace_bytes < need)
        return fail(HYPIC_ERR_WORKSPACE, "workspace %p of %zu bytes, need %zu", workspace, workspace_bytes, need);
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return fail(HYPIC_ERR_WORKSPACE, "workspace %p not 256-byte aligned", workspace);
    cudaError_t e;
    unsigned* err = err_word(&e);
    if (!err) return cuda_fail(e, "device error word");
    const BuildParams p = to_params(args);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    e = launch_build_plan(p, workspace, s);
    if (e != cudaSuccess) return cuda_fail(e, "build plan launch");
    if (gdn_build_tc_supported(p)) {
        e = launch_gdn_build_tc(p, workspace, err, s);
        if (e != cudaSuccess) return cuda_fail(e, "tensor-core build launch");
    } else if (decay_build_tc_supported(p)) {
        e = launch_decay_build_tc(p, workspace, err, s);
        if (e != cudaSuccess) return cuda_fail(e, "tensor-core decay-family build launch");
    } else if (tables && kda_build_tc_supported(p)) {
        e = launch_kda_build_tc(p, workspace, workspace_bytes, err, s);
        if (e != cudaSuccess) return cuda_fail(e, "tensor-core KDA build launch");
    } else {
        e = launch_build_simt(p, workspace, err, s);
        if (e != cudaSuccess) return cuda_fail(e, "build launch");
    }
    return HYPIC_OK;
}
}  // namespace hypic

extern "C" hypic_status hypic_segment_build(const hypic_build_args* args, void* workspace, size_t workspace_bytes,
                                            hypic_stream_t stream) {
    return segment_build_impl(args, workspace, workspace_bytes, stream, true);
}

// ---------------------------------------------------------------- compose --

namespace {

size_t T_bytes_per_obj(int family, int dk) {
    switch (family) {
        case HYPIC_GDN:
        case HYPIC_KDA: return sizeof(float) * (size_t)dk * dk;
        case HYPIC_RETNET:
        case HYPIC_MAMBA2: return sizeof(float);
        case HYPIC_GLA: return sizeof(float) * (size_t)dk;
    }
    return 0;
}

hypic_status check_compose(const hypic_compose_args* a) {
    if (!a) return fail(HYPIC_ERR_INVALID_ARG, "args is NULL");
    if (a->n_pairs < 0 || a->n_chains < 0)
        return fail(HYPIC_ERR_INVALID_ARG, "n_pairs %d n_chains %d", a->n_pairs, a->n_chains);
    hypic_status st = check_family(a->family, 0, a->n_layers, a->n_heads, a->dk, a->dv, false, nullptr, nullptr,
                                   nullptr, nullptr, false);
    if (st != HYPIC_OK) return st;
    if (!a->cu_chain || !a->cu_chain_host) return fail(HYPIC_ERR_INVALID_ARG, "cu_chain (device and host) required");
    const int32_t* cu = a->cu_chain_host;
    if (cu[0] != 0) return fail(HYPIC_ERR_INVALID_ARG, "cu_chain[0] = %d (must be 0)", cu[0]);
    for (int r = 0; r < a->n_chains; ++r)
        if (cu[r + 1] < cu[r]) return fail(HYPIC_ERR_INVALID_ARG, "cu_chain decreases at %d", r);
    const int total = cu[a->n_chains];
    if (total > 0) {
        if (!a->seg_idx || !a->seg_idx_host) return fail(HYPIC_ERR_INVALID_ARG, "seg_idx (device and host) required");
        for (int j = 0; j < total; ++j)
            if (a->seg_idx_host[j] < 0 || a->seg_idx_host[j] >= a->n_pairs)
                return fail(HYPIC_ERR_INVALID_ARG, "seg_idx[%d] = %d outside [0, %d)", j, a->seg_idx_host[j], a->n_pairs);
        if (!a->S_tab) return fail(HYPIC_ERR_INVALID_ARG, "S_tab required");
        if (a->family != HYPIC_VANILLA && !a->T_tab) return fail(HYPIC_ERR_INVALID_ARG, "T_tab required for %s", fam_name(a->family));
    }
    if (a->family == HYPIC_VANILLA && a->T_tab) return fail(HYPIC_ERR_INVALID_ARG, "T_tab must be NULL for VANILLA");
    if (!dense_T(a->family) && a->T_exp_tab)
        return fail(HYPIC_ERR_INVALID_ARG, "T_exp_tab must be NULL for %s", fam_name(a->family));
    if (a->n_chains > 0 && !a->S_out) return fail(HYPIC_ERR_INVALID_ARG, "S_out required");
    if (a->family == HYPIC_VANILLA && a->T_out) return fail(HYPIC_ERR_INVALID_ARG, "T_out must be NULL for VANILLA");
    if (a->T_exp_out && !(a->T_out && dense_T(a->family)))
        return fail(HYPIC_ERR_INVALID_ARG, "T_exp_out goes with T_out for GDN / KDA only");
    if (a->T_out && dense_T(a->family) && !a->T_exp_out)
        return fail(HYPIC_ERR_INVALID_ARG, "T_out for %s needs T_exp_out", fam_name(a->family));
    const void* ptrs[] = {a->T_tab, a->T_exp_tab, a->S_tab, a->S0, a->S_out, a->T_out, a->T_exp_out};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return fail(HYPIC_ERR_INVALID_ARG, "pointer %p not 16-byte aligned", p);
    const size_t LH = (size_t)a->n_layers * a->n_heads;
    const size_t state = sizeof(float) * (size_t)a->dk * a->dv * LH;
    const size_t out_b = state * a->n_chains;
    if (overlap(a->S_out, out_b, a->S_tab, state * a->n_pairs) ||
        overlap(a->S_out, out_b, a->T_tab, T_bytes_per_obj(a->family, a->dk) * LH * a->n_pairs) ||
        overlap(a->S_out, out_b, a->T_exp_tab, sizeof(int32_t) * LH * a->n_pairs) ||
        overlap(a->S_out, out_b, a->S0, out_b))
        return fail(HYPIC_ERR_INVALID_ARG, "S_out overlaps an input");
    if (a->T_out) {  // the chain transition outputs overlap nothing else
        const size_t tb = T_bytes_per_obj(a->family, a->dk) * LH * a->n_chains, eb = sizeof(int32_t) * LH * a->n_chains;
        const void* ins[] = {a->T_tab, a->T_exp_tab, a->S_tab, a->S0, a->S_out};
        const size_t in_b[] = {T_bytes_per_obj(a->family, a->dk) * LH * a->n_pairs, sizeof(int32_t) * LH * a->n_pairs,
                               state * a->n_pairs, out_b, out_b};
        for (int i = 0; i < 5; ++i)
            if (overlap(a->T_out, tb, ins[i], in_b[i]) || overlap(a->T_exp_out, eb, ins[i], in_b[i]))
                return fail(HYPIC_ERR_INVALID_ARG, "T_out / T_exp_out overlaps another buffer");
        if (overlap(a->T_out, tb, a->T_exp_out, eb)) return fail(HYPIC_ERR_INVALID_ARG, "T_out overlaps T_exp_out");
    }
    return HYPIC_OK;
}

}  // namespace

extern "C" hypic_status hypic_compose(const hypic_compose_args* args, hypic_stream_t stream) {
    hypic_status st = check_compose(args);
    if (st != HYPIC_OK) return st;
    if (args->n_chains == 0) return HYPIC_OK;
    cudaError_t e;
    unsigned* err = err_word(&e);
    if (!err) return cuda_fail(e, "device error word");
    ComposeParams p;
    p.family = args->family;
    p.n_layers = args->n_layers;
    p.n_heads = args->n_heads;
    p.dk = args->dk;
    p.dv = args->dv;
    p.n_pairs = args->n_pairs;
    p.n_chains = args->n_chains;
    p.T_tab = args->T_tab;
    p.T_exp_tab = args->T_exp_tab;
    p.S_tab = args->S_tab;
    p.cu_chain = args->cu_chain;
    p.seg_idx = args->seg_idx;
    p.S0 = args->S0;
    p.S_out = args->S_out;
    p.T_out = args->T_out;
    p.T_exp_out = args->T_exp_out;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    e = compose_tc_supported(p) ? launch_compose_tc(p, err, s) : launch_compose_simt(p, err, s);
    if (e != cudaSuccess) return cuda_fail(e, "compose launch");
    return HYPIC_OK;
}

// ------------------------------------------------------------------- seam --

namespace {

hypic_status check_seam(const hypic_seam_args* a) {
    if (!a) return fail(HYPIC_ERR_INVALID_ARG, "args is NULL");
    if (a->n_seams < 0) return fail(HYPIC_ERR_INVALID_ARG, "n_seams %d", a->n_seams);
    if (a->n_tokens < 0 || a->n_tokens > INT32_MAX)
        return fail(HYPIC_ERR_INVALID_ARG, "n_tokens %lld", (long long)a->n_tokens);
    if (!a->cu_seam || !a->cu_seam_host) return fail(HYPIC_ERR_INVALID_ARG, "cu_seam (device and host) required");
    const int32_t* cu = a->cu_seam_host;
    if (cu[0] != 0) return fail(HYPIC_ERR_INVALID_ARG, "cu_seam[0] = %d (must be 0)", cu[0]);
    for (int r = 0; r < a->n_seams; ++r)
        if (cu[r + 1] < cu[r]) return fail(HYPIC_ERR_INVALID_ARG, "cu_seam decreases at %d", r);
    if ((int64_t)cu[a->n_seams] != a->n_tokens)
        return fail(HYPIC_ERR_INVALID_ARG, "cu_seam[n_seams] = %d != n_tokens %lld", cu[a->n_seams], (long long)a->n_tokens);
    const bool has_tokens = a->n_tokens > 0;
    hypic_status st = check_family(a->family, a->in_dtype, a->n_layers, a->n_heads, a->dk, a->dv, has_tokens, a->alpha,
                                   a->beta, a->gamma, a->g, true);
    if (st != HYPIC_OK) return st;
    if (has_tokens && (!a->q || !a->k || !a->v || !a->o_out))
        return fail(HYPIC_ERR_INVALID_ARG, "q, k, v and o_out required");
    if (a->n_seams > 0 && !a->state_out) return fail(HYPIC_ERR_INVALID_ARG, "state_out required");
    const void* ptrs[] = {a->q, a->k, a->v, a->state_in, a->state_out, a->o_out};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return fail(HYPIC_ERR_INVALID_ARG, "pointer %p not 16-byte aligned", p);
    const size_t state = sizeof(float) * (size_t)a->dk * a->dv * a->n_layers * a->n_heads * a->n_seams;
    const size_t o_b = sizeof(float) * (size_t)a->n_layers * a->n_tokens * a->n_heads * a->dv;
    if (a->state_in != a->state_out && overlap(a->state_in, state, a->state_out, state))
        return fail(HYPIC_ERR_INVALID_ARG, "state_in and state_out partially overlap");
    if (overlap(a->o_out, o_b, a->state_out, state) || overlap(a->o_out, o_b, a->state_in, state))
        return fail(HYPIC_ERR_INVALID_ARG, "o_out overlaps a state buffer");
    return HYPIC_OK;
}

}  // namespace

extern "C" hypic_status hypic_seam_advance(const hypic_seam_args* args, hypic_stream_t stream) {
    hypic_status st = check_seam(args);
    if (st != HYPIC_OK) return st;
    if (args->n_seams == 0) return HYPIC_OK;
    cudaError_t e;
    unsigned* err = err_word(&e);
    if (!err) return cuda_fail(e, "device error word");
    SeamParams p;
    p.family = args->family;
    p.in_dtype = args->in_dtype;
    p.n_layers = args->n_layers;
    p.n_heads = args->n_heads;
    p.dk = args->dk;
    p.dv = args->dv;
    p.n_seams = args->n_seams;
    p.n_tokens = args->n_tokens;
    p.cu_seam = args->cu_seam;
    p.q = args->q;
    p.k = args->k;
    p.v = args->v;
    p.alpha = args->alpha;
    p.beta = args->beta;
    p.gamma = args->gamma;
    p.g = args->g;
    p.state_in = args->state_in;
    p.state_out = args->state_out;
    p.o_out = args->o_out;
    e = launch_seam(p, err, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "seam launch");
    return HYPIC_OK;
}

// ------------------------------------------------------------ reuse chain --

namespace {

// The chain as the compose call it contains (same tables and chains).
hypic_compose_args chain_compose_view(const hypic_chain_args* a) {
    hypic_compose_args c;
    c.family = a->family;
    c.n_layers = a->n_layers;
    c.n_heads = a->n_heads;
    c.dk = a->dk;
    c.dv = a->dv;
    c.n_pairs = a->n_pairs;
    c.T_tab = a->T_tab;
    c.T_exp_tab = a->T_exp_tab;
    c.S_tab = a->S_tab;
    c.n_chains = a->n_chains;
    c.cu_chain = a->cu_chain;
    c.cu_chain_host = a->cu_chain_host;
    c.seg_idx = a->seg_idx;
    c.seg_idx_host = a->seg_idx_host;
    c.S0 = a->S0;
    c.S_out = a->S_out;
    c.T_out = nullptr;
    c.T_exp_out = nullptr;
    return c;
}

hypic_status check_chain(const hypic_chain_args* a) {
    if (!a) return fail(HYPIC_ERR_INVALID_ARG, "args is NULL");
    const hypic_compose_args c = chain_compose_view(a);
    hypic_status st = check_compose(&c);
    if (st != HYPIC_OK) return st;
    const int n_steps = a->cu_chain_host[a->n_chains];
    if (a->n_tokens < 0 || a->n_tokens > INT32_MAX)
        return fail(HYPIC_ERR_INVALID_ARG, "n_tokens %lld", (long long)a->n_tokens);
    if (!a->cu_step || !a->cu_step_host) return fail(HYPIC_ERR_INVALID_ARG, "cu_step (device and host) required");
    const int32_t* cu = a->cu_step_host;
    if (cu[0] != 0) return fail(HYPIC_ERR_INVALID_ARG, "cu_step[0] = %d (must be 0)", cu[0]);
    for (int j = 0; j < n_steps; ++j)
        if (cu[j + 1] < cu[j]) return fail(HYPIC_ERR_INVALID_ARG, "cu_step decreases at %d", j);
    if ((int64_t)cu[n_steps] != a->n_tokens)
        return fail(HYPIC_ERR_INVALID_ARG, "cu_step[n_steps] = %d != n_tokens %lld", cu[n_steps], (long long)a->n_tokens);
    const bool has_tokens = a->n_tokens > 0;
    st = check_family(a->family, a->in_dtype, a->n_layers, a->n_heads, a->dk, a->dv, has_tokens, a->alpha, a->beta,
                      a->gamma, a->g, true);
    if (st != HYPIC_OK) return st;
    if (has_tokens && (!a->q || !a->k || !a->v || !a->o_out))
        return fail(HYPIC_ERR_INVALID_ARG, "q, k, v and o_out required");
    const void* ptrs[] = {a->q, a->k, a->v, a->o_out};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return fail(HYPIC_ERR_INVALID_ARG, "pointer %p not 16-byte aligned", p);
    const size_t LH = (size_t)a->n_layers * a->n_heads;
    const size_t state = sizeof(float) * (size_t)a->dk * a->dv * LH;
    const size_t o_b = sizeof(float) * (size_t)a->n_layers * a->n_tokens * a->n_heads * a->dv;
    if (overlap(a->o_out, o_b, a->S_out, state * a->n_chains) || overlap(a->o_out, o_b, a->S0, state * a->n_chains) ||
        overlap(a->o_out, o_b, a->S_tab, state * a->n_pairs) ||
        overlap(a->o_out, o_b, a->T_tab, T_bytes_per_obj(a->family, a->dk) * LH * a->n_pairs))
        return fail(HYPIC_ERR_INVALID_ARG, "o_out overlaps another buffer");
    return HYPIC_OK;
}

ChainParams chain_params(const hypic_chain_args* a) {
    ChainParams p;
    p.c.family = a->family;
    p.c.n_layers = a->n_layers;
    p.c.n_heads = a->n_heads;
    p.c.dk = a->dk;
    p.c.dv = a->dv;
    p.c.n_pairs = a->n_pairs;
    p.c.n_chains = a->n_chains;
    p.c.T_tab = a->T_tab;
    p.c.T_exp_tab = a->T_exp_tab;
    p.c.S_tab = a->S_tab;
    p.c.cu_chain = a->cu_chain;
    p.c.seg_idx = a->seg_idx;
    p.c.S0 = a->S0;
    p.c.S_out = a->S_out;
    p.in_dtype = a->in_dtype;
    p.n_tokens = a->n_tokens;
    p.cu_step = a->cu_step;
    p.q = a->q;
    p.k = a->k;
    p.v = a->v;
    p.alpha = a->alpha;
    p.beta = a->beta;
    p.o_out = a->o_out;
    return p;
}

size_t chain_state_floats(const hypic_chain_args* a) {
    return (size_t)a->dk * a->dv * a->n_layers * a->n_heads;
}

// Step-by-step path: two ping-pong states of one chain, then the indices
// 0..n_steps (each step's compose is a one-step chain [j, j + 1) of seg_idx).
size_t chain_ws_bytes(const hypic_chain_args* a) {
    const size_t st = (sizeof(float) * chain_state_floats(a) + 255) / 256 * 256;
    const size_t n_steps = (size_t)a->cu_chain_host[a->n_chains];
    return 2 * st + (sizeof(int32_t) * (n_steps + 1) + 255) / 256 * 256;
}

__global__ void iota_kernel(int32_t* x, int n) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) x[i] = i;
}

}  // namespace

extern "C" size_t hypic_chain_workspace_size(const hypic_chain_args* args) {
    if (check_chain(args) != HYPIC_OK) return 0;
    if (args->n_chains == 0 || chain_tc_supported(chain_params(args))) return 0;
    return chain_ws_bytes(args);
}

extern "C" hypic_status hypic_reuse_chain(const hypic_chain_args* args, void* workspace, size_t workspace_bytes,
                                          hypic_stream_t stream) {
    hypic_status st = check_chain(args);
    if (st != HYPIC_OK) return st;
    if (args->n_chains == 0) return HYPIC_OK;
    const ChainParams cp = chain_params(args);
    const bool fused = chain_tc_supported(cp);
    const size_t need = fused ? 0 : chain_ws_bytes(args);
    if (!fused && (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u)))
        return fail(HYPIC_ERR_WORKSPACE, "workspace of %zu bytes (256-byte aligned) required, got %zu at %p", need,
                    workspace_bytes, workspace);
    cudaError_t e;
    unsigned* err = err_word(&e);
    if (!err) return cuda_fail(e, "device error word");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (fused) {
        e = launch_chain_tc(cp, err, s);
        if (e != cudaSuccess) return cuda_fail(e, "reuse chain launch");
        return HYPIC_OK;
    }
    const size_t sf = chain_state_floats(args);
    const size_t st_b = (sizeof(float) * sf + 255) / 256 * 256;
    float* buf[2] = {reinterpret_cast<float*>(workspace),
                     reinterpret_cast<float*>(reinterpret_cast<char*>(workspace) + st_b)};
    int32_t* iota = reinterpret_cast<int32_t*>(reinterpret_cast<char*>(workspace) + 2 * st_b);
    const int n_steps = args->cu_chain_host[args->n_chains];
    iota_kernel<<<(n_steps + 1 + 255) / 256, 256, 0, s>>>(iota, n_steps + 1);
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e, "reuse chain launch");
    for (int r = 0; r < args->n_chains; ++r) {
        const float* cur = args->S0 ? args->S0 + r * sf : nullptr;
        float* out = args->S_out + r * sf;
        const int c0 = args->cu_chain_host[r], c1 = args->cu_chain_host[r + 1];
        if (c0 == c1) {  // no steps: the start state
            e = cur ? cudaMemcpyAsync(out, cur, sizeof(float) * sf, cudaMemcpyDeviceToDevice, s)
                    : cudaMemsetAsync(out, 0, sizeof(float) * sf, s);
            if (e != cudaSuccess) return cuda_fail(e, "reuse chain copy");
            continue;
        }
        int nb = 0;
        for (int j = c0; j < c1; ++j) {
            if (args->cu_step_host[j + 1] > args->cu_step_host[j]) {  // seam tokens of step j
                SeamParams sp;
                sp.family = args->family;
                sp.in_dtype = args->in_dtype;
                sp.n_layers = args->n_layers;
                sp.n_heads = args->n_heads;
                sp.dk = args->dk;
                sp.dv = args->dv;
                sp.n_seams = 1;
                sp.n_tokens = args->n_tokens;
                sp.cu_seam = args->cu_step + j;  // tokens [cu_step[j], cu_step[j+1])
                sp.q = args->q;
                sp.k = args->k;
                sp.v = args->v;
                sp.alpha = args->alpha;
                sp.beta = args->beta;
                sp.gamma = args->gamma;
                sp.g = args->g;
                sp.state_in = cur;
                sp.state_out = buf[nb];
                sp.o_out = args->o_out;
                if ((e = launch_seam(sp, err, s)) != cudaSuccess) return cuda_fail(e, "reuse chain seam");
                cur = buf[nb];
                nb ^= 1;
            }
            ComposeParams cp1 = cp.c;
            cp1.n_chains = 1;
            cp1.cu_chain = iota + j;  // the one-step chain [j, j + 1)
            cp1.S0 = cur;
            cp1.S_out = j + 1 == c1 ? out : buf[nb];
            e = compose_tc_supported(cp1) ? launch_compose_tc(cp1, err, s) : launch_compose_simt(cp1, err, s);
            if (e != cudaSuccess) return cuda_fail(e, "reuse chain compose");
            cur = cp1.S_out;
            nb ^= 1;
        }
    }
    return HYPIC_OK;
}

// ------------------------------------------------------------ re-rotation --

namespace {

hypic_status check_rope(const hypic_rope_args* a) {
    if (!a) return fail(HYPIC_ERR_INVALID_ARG, "args is NULL");
    if (a->n_pairs < 0) return fail(HYPIC_ERR_INVALID_ARG, "n_pairs %d", a->n_pairs);
    hypic_status st = check_family(a->family, 0, a->n_layers, a->n_heads, a->dk, a->dv, false, nullptr, nullptr,
                                   nullptr, nullptr, false);
    if (st != HYPIC_OK) return st;
    if (a->family == HYPIC_GLA || a->family == HYPIC_KDA)
        return fail(HYPIC_ERR_UNSUPPORTED, "%s: per-channel gates do not commute with the rotation", fam_name(a->family));
    if (a->rotary_dim < 2 || a->rotary_dim > a->dk || (a->rotary_dim & 1))
        return fail(HYPIC_ERR_INVALID_ARG, "rotary_dim %d (even, in [2, dk = %d])", a->rotary_dim, a->dk);
    if (!(a->base > 0.0) || !isfinite(a->base)) return fail(HYPIC_ERR_INVALID_ARG, "base %g", a->base);
    if (a->n_pairs > 0) {
        if (!a->delta || !a->S) return fail(HYPIC_ERR_INVALID_ARG, "delta and S required");
        if (dense_T(a->family) != (a->T != nullptr))
            return fail(HYPIC_ERR_INVALID_ARG, "T must be given for GDN and only for GDN");
    }
    const void* ptrs[] = {a->delta, a->T, a->S};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return fail(HYPIC_ERR_INVALID_ARG, "pointer %p not 16-byte aligned", p);
    const size_t LH = (size_t)a->n_layers * a->n_heads * a->n_pairs;
    if (overlap(a->T, sizeof(float) * LH * a->dk * a->dk, a->S, sizeof(float) * LH * a->dk * a->dv) ||
        overlap(a->delta, sizeof(int64_t) * a->n_pairs, a->S, sizeof(float) * LH * a->dk * a->dv) ||
        overlap(a->delta, sizeof(int64_t) * a->n_pairs, a->T, sizeof(float) * LH * a->dk * a->dk))
        return fail(HYPIC_ERR_INVALID_ARG, "T, S and delta overlap");
    return HYPIC_OK;
}

}  // namespace

extern "C" hypic_status hypic_rope_rerotate(const hypic_rope_args* args, hypic_stream_t stream) {
    hypic_status st = check_rope(args);
    if (st != HYPIC_OK) return st;
    if (args->n_pairs == 0) return HYPIC_OK;
    RopeParams p;
    p.n_layers = args->n_layers;
    p.n_heads = args->n_heads;
    p.dk = args->dk;
    p.dv = args->dv;
    p.n_pairs = args->n_pairs;
    p.rotary_dim = args->rotary_dim;
    p.base = args->base;
    p.delta = args->delta;
    p.T = args->T;
    p.S = args->S;
    cudaError_t e = launch_rope(p, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "re-rotation launch");
    return HYPIC_OK;
}

// ----------------------------------------------------------- conv warm-up --

namespace {

hypic_status check_conv(const hypic_conv_args* a) {
    if (!a) return fail(HYPIC_ERR_INVALID_ARG, "args is NULL");
    if (a->n_layers < 1 || a->C < 1 || a->n_seams < 0)
        return fail(HYPIC_ERR_INVALID_ARG, "n_layers %d C %d n_seams %d", a->n_layers, a->C, a->n_seams);
    if (a->K < 1 || a->K > 16) return fail(HYPIC_ERR_UNSUPPORTED, "K %d (supported: 1..16)", a->K);
    if (a->act != 0 && a->act != 1) return fail(HYPIC_ERR_INVALID_ARG, "act %d", a->act);
    if (a->n_tokens < 0 || a->n_tokens > INT32_MAX)
        return fail(HYPIC_ERR_INVALID_ARG, "n_tokens %lld", (long long)a->n_tokens);
    if (!a->cu_seam || !a->cu_seam_host) return fail(HYPIC_ERR_INVALID_ARG, "cu_seam (device and host) required");
    const int32_t* cu = a->cu_seam_host;
    if (cu[0] != 0) return fail(HYPIC_ERR_INVALID_ARG, "cu_seam[0] = %d (must be 0)", cu[0]);
    for (int r = 0; r < a->n_seams; ++r)
        if (cu[r + 1] < cu[r]) return fail(HYPIC_ERR_INVALID_ARG, "cu_seam decreases at %d", r);
    if ((int64_t)cu[a->n_seams] != a->n_tokens)
        return fail(HYPIC_ERR_INVALID_ARG, "cu_seam[n_seams] = %d != n_tokens %lld", cu[a->n_seams],
                    (long long)a->n_tokens);
    if (a->n_tokens > 0 && (!a->x || !a->w || !a->y)) return fail(HYPIC_ERR_INVALID_ARG, "x, w and y required");
    const void* ptrs[] = {a->x, a->hist, a->w, a->bias, a->y};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return fail(HYPIC_ERR_INVALID_ARG, "pointer %p not 16-byte aligned", p);
    const size_t L = (size_t)a->n_layers, C = (size_t)a->C, K = (size_t)a->K;
    const size_t yb = sizeof(float) * L * a->n_tokens * C;
    if (overlap(a->y, yb, a->x, yb) || overlap(a->y, yb, a->hist, sizeof(float) * a->n_seams * L * (K - 1) * C) ||
        overlap(a->y, yb, a->w, sizeof(float) * L * C * K) || overlap(a->y, yb, a->bias, sizeof(float) * L * C))
        return fail(HYPIC_ERR_INVALID_ARG, "y overlaps an input");
    return HYPIC_OK;
}

}  // namespace

extern "C" hypic_status hypic_conv_warmup(const hypic_conv_args* args, hypic_stream_t stream) {
    hypic_status st = check_conv(args);
    if (st != HYPIC_OK) return st;
    if (args->n_tokens == 0 || args->n_seams == 0) return HYPIC_OK;
    ConvParams p;
    p.n_layers = args->n_layers;
    p.C = args->C;
    p.K = args->K;
    p.n_seams = args->n_seams;
    p.act = args->act;
    p.n_tokens = args->n_tokens;
    p.cu_seam = args->cu_seam;
    p.x = args->x;
    p.hist = args->hist;
    p.w = args->w;
    p.bias = args->bias;
    p.y = args->y;
    cudaError_t e = launch_conv_warmup(p, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "conv warm-up launch");
    return HYPIC_OK;
}

// ------------------------------------------------------------------- misc --

extern "C" const char* hypic_status_string(hypic_status s) {
    switch (s) {
        case HYPIC_OK: return "HYPIC_OK";
        case HYPIC_ERR_INVALID_ARG: return "HYPIC_ERR_INVALID_ARG";
        case HYPIC_ERR_UNSUPPORTED: return "HYPIC_ERR_UNSUPPORTED";
        case HYPIC_ERR_WORKSPACE: return "HYPIC_ERR_WORKSPACE";
        case HYPIC_ERR_CUDA: return "HYPIC_ERR_CUDA";
        case HYPIC_ERR_TIMEOUT: return "HYPIC_ERR_TIMEOUT";
    }
    return "HYPIC_ERR_UNKNOWN";
}

extern "C" const char* hypic_last_error_detail(void) { return t_detail; }

namespace hypic {
void set_detail(const char* msg) { snprintf(t_detail, sizeof(t_detail), "%s", msg); }
}  // namespace hypic

extern "C" int hypic_version(void) { return HYPIC_VERSION; }

extern "C" hypic_status hypic_check_device(hypic_stream_t stream) {
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
    unsigned* w = err_word(&e);
    if (!w) return cuda_fail(e, "device error word");
    unsigned v = 0;
    e = cudaMemcpy(&v, w, sizeof(v), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "read device error word");
    if (v != 0) {
        const unsigned zero = 0;
        e = cudaMemcpy(w, &zero, sizeof(zero), cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return cuda_fail(e, "clear device error word");
        if (v == kErrTimeout) return fail(HYPIC_ERR_TIMEOUT, "a bounded device wait ran out");
        return fail(HYPIC_ERR_INVALID_ARG, "device-side index check failed (code %u)", v);
    }
    return HYPIC_OK;
}
