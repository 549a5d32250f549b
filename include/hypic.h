/*
 * hypic.h -- C ABI of libhypic.so, the GB300 (sm_103a) library for the
 * linear-attention state path of HYPIC (position-independent caching for
 * hybrid-attention LLMs).
 *
 * Sources (web pages on HYPIC):
 *   [README]  "HYPIC: Accelerating Hybrid-Attention LLM Serving with
 *             Position-Independent Caching", repository README: section "Key
 *             techniques" (cached transition, seam window) and section "PIC
 *             modes" (addition / transition modes, PIC_SEAM_SINK width knob).
 *   [AIBASE]  aibase news article on HYPIC (Traditional Chinese): the
 *             paragraph on the linear layers (segment-cumulative transition
 *             operator T_C, zero-start end state S(C|0), composition law
 *             S(C1.C2) = T(C2) S(C1) + S(C2)) and the paragraph on the
 *             full-attention layers (seam window of w tokens at each internal
 *             segment start, default w = 8, not cached; at reuse its own T and S
 *             are computed on the fly while the running state advances and each
 *             seam token's output is emitted).
 *   [ARXIV]   arXiv 2607.01299 abstract: near-exact, constant-time composition
 *             of independently cached segments.
 *
 * Families and per-token recurrences (state S is dk x dv, left-multiplied,
 * latest token leftmost; all six are among the families the [AIBASE]
 * linear-layer paragraph names, which prints none of their recurrences: the
 * forms below are the published ones read as left-multiplied transitions):
 *   HYPIC_GDN      S_t = a_t (I - b_t k_t k_t^T) S_{t-1} + b_t k_t v_t^T
 *                  (gated delta rule); T_C is a dense dk x dk matrix.
 *   HYPIC_RETNET   S_t = g S_{t-1} + k_t v_t^T;  T_C = g^L (a scalar).
 *   HYPIC_GLA      S_t = Diag(g_t) S_{t-1} + k_t v_t^T;  T_C = prod g_t (dk-vector).
 *   HYPIC_VANILLA  S_t = S_{t-1} + k_t v_t^T;  T_C = I (not stored).
 *   HYPIC_KDA      S_t = (I - b_t k_t k_t^T) Diag(a_t) S_{t-1} + b_t k_t v_t^T
 *                  (Kimi delta attention: a per-channel gate a_t, read from g,
 *                  acts before the delta projection); T_C is a dense dk x dk
 *                  matrix stored like GDN's.
 *   HYPIC_MAMBA2   S_t = a_t S_{t-1} + k_t v_t^T with a scalar decay a_t per
 *                  token and head (read from alpha; the input step size is
 *                  taken as folded into k);  T_C = prod a_t (a scalar).
 *   Seam outputs: o_t = S_t^T q_t, with S_t the state after token t's write.
 *
 * Conventions common to every call
 *   - Every tensor pointer is a DEVICE pointer owned by the caller, except the
 *     arguments whose name ends in _host, which are host pointers read during
 *     the call only.  The library allocates no memory; scratch memory comes
 *     from the caller (see hypic_build_workspace_size).
 *   - Layouts are dense row-major, innermost dimension last; every tensor
 *     pointer must be 16-byte aligned.
 *       k, v, q        [n_layers][n_tokens][n_heads][dk | dv]   (f32 or bf16)
 *       alpha, beta    [n_layers][n_tokens][n_heads]             (f32)
 *                      (alpha: GDN's gate, MAMBA2's decay; beta: GDN, KDA)
 *       gamma          [n_layers][n_heads]                       (f32)
 *       g              [n_layers][n_tokens][n_heads][dk]         (f32; GLA, KDA)
 *       per-item state [n_items][n_layers][n_heads][dk][dv]      (f32)
 *   - Calls are asynchronous on the given stream and the library keeps no
 *     state between calls (except the device error word, below); distinct
 *     threads may call concurrently.
 *   - Every argument is checked on the host before anything is launched; a
 *     rejected call returns HYPIC_ERR_INVALID_ARG or HYPIC_ERR_UNSUPPORTED
 *     and touches no output.  hypic_last_error_detail() then says why.
 *   - A launch failure returns HYPIC_ERR_CUDA.  Kernels that wait on
 *     asynchronous copies bound every wait; a wait that runs out sets the
 *     device error word, which hypic_check_device() reports as
 *     HYPIC_ERR_TIMEOUT.
 *   - A zero-length segment (or body) yields the identity pair (T = I, S = 0).
 *   - The library neither normalises k nor scales q.
 */
#ifndef HYPIC_H_
#define HYPIC_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define HYPIC_VERSION 150 /* 1.5.0: hypic_conv_warmup */

#if defined(__GNUC__)
#define HYPIC_API __attribute__((visibility("default")))
#else
#define HYPIC_API
#endif

typedef struct CUstream_st* hypic_stream_t; /* same type as cudaStream_t */

typedef enum {
    HYPIC_OK = 0,
    HYPIC_ERR_INVALID_ARG = 1, /* null / misaligned pointer, bad size, bad offsets */
    HYPIC_ERR_UNSUPPORTED = 2, /* valid but not implemented (family x dtype x dims) */
    HYPIC_ERR_WORKSPACE = 3,   /* workspace missing or smaller than required */
    HYPIC_ERR_CUDA = 4,        /* a CUDA runtime call failed */
    HYPIC_ERR_TIMEOUT = 5      /* a bounded device-side wait ran out */
} hypic_status;

typedef enum {
    HYPIC_GDN = 0,
    HYPIC_RETNET = 1,
    HYPIC_GLA = 2,
    HYPIC_VANILLA = 3,
    HYPIC_KDA = 4,
    HYPIC_MAMBA2 = 5
} hypic_family;
typedef enum { HYPIC_F32 = 0, HYPIC_BF16 = 1 } hypic_dtype;

/* ------------------------------------------------------------------ build --
 * Cached pair (T_C, S(C|0)) of every (segment, layer, head) of a ragged batch
 * ([AIBASE] linear-layer paragraph; [README] "Key techniques", cached
 * transition).  Segment s occupies tokens [cu_seqlens[s], cu_seqlens[s+1]) of
 * the packed token arrays; its cached pair covers the body
 * [cu_seqlens[s] + seam_skip[s], cu_seqlens[s+1]): the leading seam_skip[s]
 * tokens are the seam window that is not cached ([AIBASE] full-attention
 * paragraph).  seam_skip == NULL means 0 for every segment.
 *
 * Inputs by family (unused ones must be NULL):
 *   GDN      k, v (in_dtype), alpha, beta (f32)
 *   RETNET   k, v, gamma                       (beta must be NULL: b = 1)
 *   GLA      k, v, g
 *   VANILLA  k, v
 *   KDA      k, v, g (the per-channel gate a_t), beta
 *   MAMBA2   k, v, alpha (the per-token decay a_t)
 * Outputs, leading dims [n_segments][n_layers][n_heads]:
 *   S_out   [..][dk][dv] f32
 *   T_out   GDN, KDA: [..][dk][dk] f32 mantissa, with T_exp_out [..] int32 such
 *           that T_C = T_out * 2^T_exp_out (the exponent keeps T_C representable
 *           when its entries fall below the f32 range, as they do for long
 *           segments with strong decay); RETNET: [..] f32 scalar g^L;
 *           MAMBA2: [..] f32 scalar prod a_t; GLA: [..][dk] f32 vector;
 *           VANILLA: NULL.
 *   T_exp_out  GDN and KDA only (NULL otherwise).
 * Supported: dk, dv in {16, 32, 64, 128}; GDN and KDA require dk == dv.
 * Work order: segments are processed longest body first (LPT order).
 */
typedef struct {
    int family;                /* hypic_family */
    int in_dtype;              /* hypic_dtype of k and v */
    int n_layers, n_heads, dk, dv;
    int n_segments;
    int64_t n_tokens;          /* rows of the packed token arrays */
    const int32_t* cu_seqlens;       /* device [n_segments+1], non-decreasing, 0 .. n_tokens */
    const int32_t* cu_seqlens_host;  /* host copy of the same (validation, planning) */
    const int32_t* seam_skip;        /* device [n_segments] or NULL */
    const int32_t* seam_skip_host;   /* host copy or NULL (must match seam_skip) */
    const void* k;
    const void* v;
    const float* alpha;
    const float* beta;
    const float* gamma;
    const float* g;
    float* T_out;
    int32_t* T_exp_out;
    float* S_out;
} hypic_build_args;

/* Bytes of device scratch the build needs for these arguments: the plan and
   work counter (a few KB); for KDA at dk = dv = 128 with bf16 k and v also the
   tables of its tensor-core path, 128 KB per 64-token chunk, layer and head,
   for at most 4 GiB of chunks at a time (a longer segment is built in parts,
   each chained after the pair of the parts before it).  Returns 0 when the
   arguments are invalid. */
HYPIC_API size_t hypic_build_workspace_size(const hypic_build_args* args);

/* Launch the build on `stream`.  `workspace` is device memory of at least
   hypic_build_workspace_size(args) bytes, 256-byte aligned, owned by the
   caller and not used by any other call until this one completes on the
   stream.  Returns HYPIC_ERR_WORKSPACE when it is NULL or too small.  KDA at
   d = 128 (bf16) takes its segments in batches whose chunk tables fit the
   workspace. */
HYPIC_API hypic_status hypic_segment_build(const hypic_build_args* args, void* workspace,
                                 size_t workspace_bytes, hypic_stream_t stream);

/* ---------------------------------------------------------------- compose --
 * Chain composition of cached pairs ([AIBASE] linear-layer paragraph:
 * S(C1.C2) = T(C2) S(C1) + S(C2); [ARXIV] constant-time composition).  For
 * chain r and every (layer, head): S <- S0[r] (or 0 when S0 == NULL), then
 * S <- T_p S + S_p for p = seg_idx[cu_chain[r]], ..., seg_idx[cu_chain[r+1]-1]
 * in that order; S_out[r] <- S.  A chain of length 0 copies its start state.
 * T_p S is a dk x dk matrix product (GDN and KDA, with T_p = T_tab *
 * 2^T_exp_tab; T_exp_tab == NULL means exponent 0), a scalar (RETNET,
 * MAMBA2), a row scaling (GLA) or the identity (VANILLA: plain addition,
 * T_tab must be NULL).
 * Pair tables (the build's outputs, or any cache of them):
 *   T_tab [n_pairs][n_layers][n_heads](...) as T_out above; S_tab
 *   [n_pairs][n_layers][n_heads][dk][dv].
 * S_out [n_chains][n_layers][n_heads][dk][dv] must not overlap the tables or S0.
 * T_out (optional, NULL for VANILLA) receives each chain's own transition
 * T_chain = T_{p_n} ... T_{p_1} (the identity for an empty chain), laid out
 * like the build's T_out with leading dims [n_chains][n_layers][n_heads];
 * GDN and KDA also need T_exp_out [n_chains][n_layers][n_heads] int32
 * (T_chain = T_out * 2^T_exp_out).  With S0 == NULL the chain's result is
 * then itself a cached pair (T_out, S_out) of the concatenated segments, so
 * chains of chains compose like pairs ([AIBASE] composition law applied to a
 * tree of segments).  Neither may overlap an input or S_out.  With T_out the
 * dense families run on CUDA cores at every d.
 * Supported: dk, dv in {16, 32, 64, 128}; GDN and KDA require dk == dv.
 */
typedef struct {
    int family;
    int n_layers, n_heads, dk, dv;
    int n_pairs;
    const float* T_tab;
    const int32_t* T_exp_tab;
    const float* S_tab;
    int n_chains;
    const int32_t* cu_chain;        /* device [n_chains+1], non-decreasing from 0 */
    const int32_t* cu_chain_host;   /* host copy */
    const int32_t* seg_idx;         /* device [cu_chain[n_chains]], each in [0, n_pairs) */
    const int32_t* seg_idx_host;    /* host copy (validation) */
    const float* S0;                /* device [n_chains][..] or NULL */
    float* S_out;
    float* T_out;                   /* device, optional: each chain's own transition (above) */
    int32_t* T_exp_out;             /* device [n_chains][n_layers][n_heads]: with T_out, GDN / KDA */
} hypic_compose_args;

HYPIC_API hypic_status hypic_compose(const hypic_compose_args* args, hypic_stream_t stream);

/* ------------------------------------------------------------------- seam --
 * Seam-window advance ([AIBASE] full-attention paragraph; [README] "PIC
 * modes", seam width PIC_SEAM_SINK, default 8).  For seam r and every
 * (layer, head): S <- state_in[r] (or 0 when state_in == NULL), then for each
 * token t in [cu_seam[r], cu_seam[r+1]) of the packed seam-token arrays:
 * advance S by the family's recurrence and write o_out[layer][t][head] =
 * S_t^T q_t; finally state_out[r] <- S.  The fraction-to-count mapping of the
 * width knob is the caller's; the library takes explicit token ranges.
 * Inputs: q, k (in_dtype) [n_layers][n_tokens][n_heads][dk], v [..][dv] and the
 * family's gates as for the build (over the seam tokens).
 * state_in, state_out [n_seams][n_layers][n_heads][dk][dv] f32; they may be
 * the same buffer (in-place advance) but must not otherwise overlap.
 * o_out [n_layers][n_tokens][n_heads][dv] f32.
 * Supported: dk, dv in {16, 32, 64, 128}.
 */
typedef struct {
    int family;
    int in_dtype;
    int n_layers, n_heads, dk, dv;
    int n_seams;
    int64_t n_tokens;
    const int32_t* cu_seam;         /* device [n_seams+1], non-decreasing from 0 to n_tokens */
    const int32_t* cu_seam_host;    /* host copy */
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
} hypic_seam_args;

HYPIC_API hypic_status hypic_seam_advance(const hypic_seam_args* args, hypic_stream_t stream);

/* ------------------------------------------------------------ reuse chain --
 * The reuse path of a request in one call ([AIBASE] linear-layer paragraph:
 * the seam tokens after each cached segment are recomputed live and advance
 * the running state, and the cached pairs are composed onto it).  For chain r
 * and every (layer, head): S <- S0[r] (or 0 when S0 == NULL), then for each
 * step j in [cu_chain[r], cu_chain[r+1]):
 *   (1) advance S over the seam tokens [cu_step[j], cu_step[j+1]) of the
 *       packed seam-token arrays, writing o_out[layer][t][head] = S_t^T q_t
 *       for each, exactly as hypic_seam_advance;
 *   (2) S <- T_p S + S_p with p = seg_idx[j], exactly as hypic_compose.
 * Finally S_out[r] <- S.  A step without seam tokens is a plain compose step.
 * Pair tables, T_exp_tab, seg_idx, S0 and S_out: as for hypic_compose.
 * Seam tokens (n_tokens = cu_step[n_steps], n_steps = cu_chain[n_chains]):
 * q, k, v, the gates and o_out as for hypic_seam_advance.
 * GDN with dk = dv = 128 runs as one fused kernel that keeps every running
 * state on chip from the first step to the last (no workspace).  Every other
 * supported case runs the two calls step by step and needs a workspace of
 * hypic_chain_workspace_size(args) bytes (two states of one chain), 256-byte
 * aligned, owned by the caller until the call completes on the stream;
 * HYPIC_ERR_WORKSPACE when it is needed and NULL or too small.
 * Supported: as hypic_seam_advance and hypic_compose together.
 */
typedef struct {
    int family;
    int in_dtype;                   /* of q, k, v */
    int n_layers, n_heads, dk, dv;
    int n_pairs;
    const float* T_tab;
    const int32_t* T_exp_tab;
    const float* S_tab;
    int n_chains;
    const int32_t* cu_chain;        /* device [n_chains+1], non-decreasing from 0 */
    const int32_t* cu_chain_host;   /* host copy */
    const int32_t* seg_idx;         /* device [n_steps], each in [0, n_pairs) */
    const int32_t* seg_idx_host;    /* host copy (validation) */
    const int32_t* cu_step;         /* device [n_steps+1], non-decreasing from 0 to n_tokens */
    const int32_t* cu_step_host;    /* host copy */
    int64_t n_tokens;               /* seam tokens in all */
    const void* q;
    const void* k;
    const void* v;
    const float* alpha;
    const float* beta;
    const float* gamma;
    const float* g;
    const float* S0;                /* device [n_chains][n_layers][n_heads][dk][dv] or NULL */
    float* S_out;                   /* device [n_chains][n_layers][n_heads][dk][dv] */
    float* o_out;                   /* device [n_layers][n_tokens][n_heads][dv] */
} hypic_chain_args;

/* Workspace bytes hypic_reuse_chain needs for these arguments (0 on the
   fused path); 0 also when the arguments are invalid (the call reports why). */
HYPIC_API size_t hypic_chain_workspace_size(const hypic_chain_args* args);
HYPIC_API hypic_status hypic_reuse_chain(const hypic_chain_args* args, void* workspace, size_t workspace_bytes,
                                         hypic_stream_t stream);

/* -------------------------------------------------------- no-alloc build --
 * No counterpart in the HYPIC pages: this entry point exists for callers of the
 * library that are not allowed to allocate device memory themselves -- for
 * example a plugin that an inference engine hands only its input and output
 * buffers, or a serving loop whose memory is owned by another allocator and
 * must not grow or be synchronised by cudaMalloc in the middle of a request.
 *
 * It computes exactly what hypic_segment_build computes, with the same
 * arguments and errors, but takes no workspace: its scratch (the work order
 * and work counter, about 64 KB) is a fixed array inside this library, and
 * every GPU that loads the library keeps that array until the process exits.
 *   - n_segments is limited to HYPIC_NOALLOC_MAX_SEGMENTS; a larger batch is
 *     rejected with HYPIC_ERR_WORKSPACE before anything is launched (use
 *     hypic_segment_build with a caller workspace instead).
 *   - Every call looks up the array's device address (cudaGetSymbolAddress)
 *     with the calling thread's current device.  The first call on a device
 *     may also make the CUDA runtime load this library's device code there
 *     (lazy module loading); make that first call before any stream capture.
 *   - Every call on a device shares the one array.  Each call rewrites the
 *     whole order and zeroes the counter before using them, but calls whose
 *     work overlaps on the GPU (other streams, other threads) race on it:
 *     serialise them.
 *   - The call itself allocates nothing (no cudaMalloc, no allocating library
 *     routine).
 *   - KDA at d = 128 runs its CUDA-core kernel here: the chunk tables of its
 *     tensor-core path do not fit the fixed array.
 */
#define HYPIC_NOALLOC_MAX_SEGMENTS 16384
HYPIC_API hypic_status hypic_segment_build_noalloc(const hypic_build_args* args, hypic_stream_t stream);

/* ------------------------------------------------------------ re-rotation --
 * State re-rotation for variants whose keys carry rotary position embeddings
 * ([AIBASE] linear-layer paragraph: the "state re-rotation" patch, named but
 * not spelled out there).  A cached segment reused delta positions away sees
 * each of its keys as R k, R = R(delta) the rotary rotation.  For a family
 * whose per-token transition is built from k k^T and scalars (GDN, RETNET,
 * MAMBA2, VANILLA) each transition A becomes R A R^T and each write k v^T
 * becomes R k v^T, so the pair becomes (R T R^T, R S); this call applies that
 * in place.  GLA and KDA return HYPIC_ERR_UNSUPPORTED: their per-channel gates
 * do not commute with R, so no re-rotation of the pair is exact.
 * R turns the first rotary_dim features in rotate-half pairs: for
 * i < h = rotary_dim / 2, (x_i, x_{i+h}) -> (x_i cos a - x_{i+h} sin a,
 * x_{i+h} cos a + x_i sin a) with a = delta * base^(-2i / rotary_dim); the other
 * features are unchanged.  Angles are formed in double.
 *   delta  device int64 [n_pairs]: the position shift of each pair.
 *   T      device [n_pairs][n_layers][n_heads][dk][dk] f32 mantissa (GDN; its
 *          T_exp is unchanged, R being orthogonal), NULL for the other families.
 *   S      device [n_pairs][n_layers][n_heads][dk][dv] f32.
 * Supported: dk, dv in {16, 32, 64, 128}, rotary_dim even in [2, dk], base > 0.
 */
typedef struct {
    int family;
    int n_layers, n_heads, dk, dv;
    int n_pairs;
    int rotary_dim;
    double base;
    const int64_t* delta;
    float* T;
    float* S;
} hypic_rope_args;

HYPIC_API hypic_status hypic_rope_rerotate(const hypic_rope_args* args, hypic_stream_t stream);

/* ------------------------------------------------------- conv warm-up --
 * Conv-state warm-up for variants with a short causal convolution on the
 * linear layers' inputs ([AIBASE] linear-layer paragraph: the "conv-state
 * warm-up" patch, named only there).  At a seam window the K - 1 inputs
 * before the window come from the new prefix, not from the cached segment's
 * past.  A depthwise causal convolution of width K gives token t (of window r)
 * and channel c
 *     y_t = act(bias_c + sum_{j<K} w[c][j] x_{t-K+1+j}),
 * with the inputs before cu_seam[r] taken from hist[r] (oldest first).
 *   x      device [n_layers][n_tokens][C] f32: the windows' raw inputs, packed
 *          by window (window r = tokens [cu_seam[r], cu_seam[r+1])).
 *   hist   device [n_seams][n_layers][K-1][C] f32, or NULL for zeros (a
 *          window at a sequence start).
 *   w      device [n_layers][C][K] f32 (tap K-1 multiplies the current token);
 *   bias   device [n_layers][C] f32 or NULL.
 *   act    0 = identity, 1 = SiLU (x / (1 + e^-x)).
 *   y      device [n_layers][n_tokens][C] f32; must not overlap the inputs.
 * Supported: 1 <= K <= 16.
 */
typedef struct {
    int n_layers, C, K;
    int n_seams;
    int64_t n_tokens;
    const int32_t* cu_seam;       /* device [n_seams+1], from 0 to n_tokens */
    const int32_t* cu_seam_host;  /* host copy (validation) */
    const float* x;
    const float* hist;
    const float* w;
    const float* bias;
    int act;
    float* y;
} hypic_conv_args;

HYPIC_API hypic_status hypic_conv_warmup(const hypic_conv_args* args, hypic_stream_t stream);

/* ------------------------------------------------------------------ misc -- */

/* Static, never NULL. */
HYPIC_API const char* hypic_status_string(hypic_status status);

/* Detail of the last error returned on the calling thread (thread-local,
   overwritten by the next failing call). */
HYPIC_API const char* hypic_last_error_detail(void);

/* HYPIC_VERSION of the loaded library. */
HYPIC_API int hypic_version(void);

/* Synchronise `stream`, then read and clear the current device's error word:
   HYPIC_ERR_TIMEOUT when a bounded device wait ran out since the last check,
   HYPIC_ERR_CUDA when the stream reports an error, else HYPIC_OK. */
HYPIC_API hypic_status hypic_check_device(hypic_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* HYPIC_H_ */
