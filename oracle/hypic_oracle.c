/*
 * hypic_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, fp64 CPU restatement of the linear-attention state path of
 * HYPIC (position-independent caching for hybrid-attention models).  It is the
 * checker that the CUDA library is compared against; it shares no code, header,
 * table or helper with the GPU path and must never be called by the product.
 * Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline leg use it.
 *
 * Sources, by page:
 *  [AB]  aibase news article on HYPIC (Traditional Chinese), paragraph on the
 *        linear layers ("對線性層..."): a segment C is summarised by the
 *        segment-cumulative transition operator T_C (the ordered product of all
 *        per-token transition matrices of C) and the zero-start end state
 *        S(C|0); reuse composes S(C1.C2) = T(C2) S(C1) + S(C2); naive addition
 *        S(C1)+S(C2) is exact only for plain linear attention.
 *  [AB2] same article, paragraph on the full-attention layers ("對全注意力層..."):
 *        the first w tokens of each internal segment form a seam window that is
 *        not cached; at reuse the linear layers compute the window's own T and S
 *        on the fly, advance the running state through it and emit each seam
 *        token's output.
 *  [AX]  arXiv abstract (2607.01299): near-exact, constant-time composition of
 *        independently cached segments.
 *  Per-token recurrences (the families named in [AB]); the state S is dk x dv
 *  and is left-multiplied by the transition, latest token leftmost:
 *    GDN    (gated delta rule, Yang/Kautz/Hatamizadeh, "Gated Delta Networks"):
 *           S_t = a_t (I - b_t k_t k_t^T) S_{t-1} + b_t k_t v_t^T
 *    RetNet (scalar decay):   S_t = g S_{t-1} + k_t v_t^T,      T = g^L
 *    GLA    (diagonal decay): S_t = Diag(g_t) S_{t-1} + k_t v_t^T
 *    vanilla linear attention: S_t = S_{t-1} + k_t v_t^T,       T = I
 *    KDA    (Kimi delta attention, a delta rule with a per-channel gate):
 *           S_t = (I - b_t k_t k_t^T) Diag(a_t) S_{t-1} + b_t k_t v_t^T,
 *           a_t in (0, 1]^dk: the gate acts first, then the delta projection
 *    Mamba2 (scalar decay per token, the SSD scan as linear attention):
 *           S_t = a_t S_{t-1} + k_t v_t^T,                     T = prod a_t
 *    output of a token: o_t = S_t^T q_t (state after the token's own write).
 *  [AB] names RetNet, Mamba2, GLA, DeltaNet, GDN and KDA as the families whose
 *  pair needs T_C; it prints none of their recurrences.  The two above are the
 *  published forms read as left-multiplied transitions on a dk x dv state:
 *  Mamba2's input scaling (dt) is taken as already folded into k, and KDA's
 *  gate vector is read from the same per-channel gate array as GLA's.
 *
 * Everything is a token-by-token loop in double precision, exactly in the
 * order above.  Inputs arrive as float32 arrays (bf16 inputs are upcast exactly
 * by the caller) and are widened to double on read.
 *
 * Packed layouts (row-major, innermost last):
 *   k, v, q   [n_layers][n_tokens][n_heads][d]
 *   alpha, beta [n_layers][n_tokens][n_heads]
 *   gamma     [n_layers][n_heads]
 *   g         [n_layers][n_tokens][n_heads][dk]   (GLA, KDA)
 *   alpha     also the per-token decay of Mamba2; beta also KDA's
 *   T (GDN, KDA)      [n_items][n_layers][n_heads][dk][dk]
 *   T (RetNet, Mamba2)[n_items][n_layers][n_heads]
 *   T (GLA)   [n_items][n_layers][n_heads][dk]
 *   S, state  [n_items][n_layers][n_heads][dk][dv]
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_GDN = 0, OR_RETNET = 1, OR_GLA = 2, OR_VANILLA = 3, OR_KDA = 4, OR_MAMBA2 = 5 };

/* Families whose T_C is a dk x dk matrix, and those whose T_C is a scalar. */
static int dense_T(int family) { return family == OR_GDN || family == OR_KDA; }
static int scalar_T(int family) { return family == OR_RETNET || family == OR_MAMBA2; }

/* ---------------------------------------------------------------- tokens -- */

/* Read one token's inputs for (layer, token, head) into double buffers. */
typedef struct {
    int family, n_layers, n_heads, dk, dv;
    long long n_tokens;
    const float *q, *k, *v, *alpha, *beta, *gamma, *g;
} or_inputs;

static void read_vec(const float* base, long long off, int n, double* out)
{
    for (int i = 0; i < n; ++i) out[i] = (double)base[off + i];
}

/* M <- A_t M for the GDN transition A_t = a (I - b k k^T), M is dk x ncols.
   [AB]: the per-token transition matrix of the gated-delta family. */
static void gdn_apply_transition(int dk, int ncols, double* M, const double* k,
                                 double a, double b, double* tmp)
{
    for (int j = 0; j < ncols; ++j) {
        double s = 0.0;
        for (int i = 0; i < dk; ++i) s += k[i] * M[(size_t)i * ncols + j];
        tmp[j] = s; /* (k^T M)_j */
    }
    for (int i = 0; i < dk; ++i)
        for (int j = 0; j < ncols; ++j)
            M[(size_t)i * ncols + j] = a * (M[(size_t)i * ncols + j] - b * k[i] * tmp[j]);
}

/* M <- (I - b k k^T) Diag(a) M for the KDA transition, M is dk x ncols:
   the per-channel gate scales row i of M by a[i], then the delta projection. */
static void kda_apply_transition(int dk, int ncols, double* M, const double* k,
                                 const double* a, double b, double* tmp)
{
    for (int i = 0; i < dk; ++i)
        for (int j = 0; j < ncols; ++j) M[(size_t)i * ncols + j] *= a[i];
    for (int j = 0; j < ncols; ++j) {
        double s = 0.0;
        for (int i = 0; i < dk; ++i) s += k[i] * M[(size_t)i * ncols + j];
        tmp[j] = s; /* (k^T Diag(a) M)_j */
    }
    for (int i = 0; i < dk; ++i)
        for (int j = 0; j < ncols; ++j) M[(size_t)i * ncols + j] -= b * k[i] * tmp[j];
}

/* S <- S + w k v^T (the write term of every family). */
static void add_write(int dk, int dv, double* S, const double* k, const double* v, double w)
{
    for (int i = 0; i < dk; ++i)
        for (int j = 0; j < dv; ++j) S[(size_t)i * dv + j] += w * k[i] * v[j];
}

/* One token of the recurrence of the chosen family, applied to the state S and,
   when T is non-NULL, to the running transition product T (the same left
   multiply, without the write term). */
static void token_step(const or_inputs* in, int layer, long long tok, int head,
                       double* S, double* T, double* Tvec, double* Tscal,
                       double* kb, double* vb, double* gb, double* tmp)
{
    const int dk = in->dk, dv = in->dv, H = in->n_heads;
    const long long row = ((long long)layer * in->n_tokens + tok) * H + head;
    read_vec(in->k, row * dk, dk, kb);
    read_vec(in->v, row * dv, dv, vb);
    switch (in->family) {
    case OR_GDN: {
        const double a = in->alpha[row];
        const double b = in->beta[row];
        gdn_apply_transition(dk, dv, S, kb, a, b, tmp);
        add_write(dk, dv, S, kb, vb, b);
        if (T) gdn_apply_transition(dk, dk, T, kb, a, b, tmp);
        break;
    }
    case OR_RETNET: {
        const double gm = in->gamma[(size_t)layer * H + head];
        for (size_t i = 0; i < (size_t)dk * dv; ++i) S[i] *= gm;
        add_write(dk, dv, S, kb, vb, 1.0);
        if (Tscal) *Tscal *= gm;
        break;
    }
    case OR_GLA: {
        read_vec(in->g, row * dk, dk, gb);
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dv; ++j) S[(size_t)i * dv + j] *= gb[i];
        add_write(dk, dv, S, kb, vb, 1.0);
        if (Tvec) for (int i = 0; i < dk; ++i) Tvec[i] *= gb[i];
        break;
    }
    case OR_KDA: {
        read_vec(in->g, row * dk, dk, gb);
        const double b = in->beta[row];
        kda_apply_transition(dk, dv, S, kb, gb, b, tmp);
        add_write(dk, dv, S, kb, vb, b);
        if (T) kda_apply_transition(dk, dk, T, kb, gb, b, tmp);
        break;
    }
    case OR_MAMBA2: {
        const double a = in->alpha[row];
        for (size_t i = 0; i < (size_t)dk * dv; ++i) S[i] *= a;
        add_write(dk, dv, S, kb, vb, 1.0);
        if (Tscal) *Tscal *= a;
        break;
    }
    default: /* vanilla */
        add_write(dk, dv, S, kb, vb, 1.0);
        break;
    }
}

static int check_common(int family, int n_layers, int n_heads, int dk, int dv)
{
    if (family < OR_GDN || family > OR_MAMBA2) return 1;
    if (n_layers <= 0 || n_heads <= 0 || dk <= 0 || dv <= 0) return 1;
    return 0;
}

/* ----------------------------------------------------------------- build -- */

/*
 * Build the cached pair (T_C, S(C|0)) of every (segment, layer, head) [AB].
 * Segment s covers tokens [cu_seqlens[s] + skip[s], cu_seqlens[s+1]); skip
 * (nullable) removes the seam window of an internal segment from the cached
 * pair [AB2].  The build starts from T = I, S = 0 and runs the token loop.
 * T_out may be NULL (vanilla: T = I is not stored).
 */
int oracle_build(int family, int n_layers, int n_heads, int dk, int dv,
                 int n_seg, const int* cu_seqlens, const int* skip, long long n_tokens,
                 const float* k, const float* v, const float* alpha, const float* beta,
                 const float* gamma, const float* g,
                 double* T_out, double* S_out, int n_threads)
{
    if (check_common(family, n_layers, n_heads, dk, dv) || n_seg < 0) return 1;
    or_inputs in = {family, n_layers, n_heads, dk, dv, n_tokens, NULL, k, v, alpha, beta, gamma, g};
    const long long n_items = (long long)n_seg * n_layers * n_heads;
    int bad = 0;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
#endif
    for (long long it = 0; it < n_items; ++it) {
        const int head = (int)(it % n_heads);
        const int layer = (int)((it / n_heads) % n_layers);
        const int seg = (int)(it / ((long long)n_heads * n_layers));
        const long long b0 = (long long)cu_seqlens[seg] + (skip ? skip[seg] : 0);
        const long long b1 = cu_seqlens[seg + 1];
        double* S = (double*)calloc((size_t)dk * dv, sizeof(double));
        double* T = dense_T(family) ? (double*)calloc((size_t)dk * dk, sizeof(double)) : NULL;
        double* Tv = (family == OR_GLA) ? (double*)malloc((size_t)dk * sizeof(double)) : NULL;
        double Ts = 1.0;
        double* kb = (double*)malloc(sizeof(double) * (size_t)(dk + dv + dk + (dk > dv ? dk : dv)));
        double *vb = kb + dk, *gb = vb + dv, *tmp = gb + dk;
        if (!S || !kb || (dense_T(family) && !T) || (family == OR_GLA && !Tv)) { bad = 1; }
        else {
            if (T) for (int i = 0; i < dk; ++i) T[(size_t)i * dk + i] = 1.0;
            if (Tv) for (int i = 0; i < dk; ++i) Tv[i] = 1.0;
            for (long long t = b0; t < b1; ++t)
                token_step(&in, layer, t, head, S, T, Tv, &Ts, kb, vb, gb, tmp);
            memcpy(S_out + (size_t)it * dk * dv, S, sizeof(double) * (size_t)dk * dv);
            if (T_out) {
                if (dense_T(family)) memcpy(T_out + (size_t)it * dk * dk, T, sizeof(double) * (size_t)dk * dk);
                else if (family == OR_GLA) memcpy(T_out + (size_t)it * dk, Tv, sizeof(double) * (size_t)dk);
                else if (scalar_T(family)) T_out[it] = Ts;
            }
        }
        free(S); free(T); free(Tv); free(kb);
    }
    return bad;
}

/* --------------------------------------------------------------- compose -- */

/*
 * Compose chains of cached pairs [AB]: for chain r, starting from S0[r] (or
 * zero), apply S <- T_i S + S_i for i = seg_idx[cu_chain[r]], ...,
 * seg_idx[cu_chain[r+1]-1] in that order.  The product T_i S is the family's:
 * a dk x dk matrix (GDN, KDA), a scalar (RetNet, Mamba2), a row scaling (GLA) or the
 * identity (vanilla, plain addition).  T_tab holds T_C in double with any
 * stored scale already applied; `naive` != 0 drops T entirely (the addition
 * strawman of [AB], "--pic-mode addition" in the README's PIC modes table).
 * T_out (nullable, not with `naive` or vanilla) receives each chain's own
 * transition, the ordered product T_{p_n} ... T_{p_1} (identity for an empty
 * chain), in the family's T layout: with it the chain is itself a cached pair
 * (T_out, S_out from a zero start) that composes like any other [AB].
 */
int oracle_compose(int family, int n_layers, int n_heads, int dk, int dv, int n_pairs,
                   const double* T_tab, const double* S_tab,
                   int n_chains, const int* cu_chain, const int* seg_idx,
                   const double* S0, double* S_out, int naive, int n_threads, double* T_out)
{
    if (check_common(family, n_layers, n_heads, dk, dv) || n_chains < 0 || n_pairs < 0) return 1;
    if (T_out && (naive || family == OR_VANILLA)) return 1;
    const long long LH = (long long)n_layers * n_heads;
    const long long n_items = (long long)n_chains * LH;
    const size_t dd = (size_t)dk * dv;
    const size_t tn = dense_T(family) ? (size_t)dk * dk : (family == OR_GLA ? (size_t)dk : 1);
    int bad = 0;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
#endif
    for (long long it = 0; it < n_items; ++it) {
        const long long lh = it % LH;
        const int r = (int)(it / LH);
        double* S = (double*)malloc(sizeof(double) * dd);
        double* N = (double*)malloc(sizeof(double) * dd);
        double* Tc = (double*)malloc(sizeof(double) * tn * 2);  /* chain product, and its update */
        if (!S || !N || !Tc) { bad = 1; free(S); free(N); free(Tc); continue; }
        if (S0) memcpy(S, S0 + (size_t)it * dd, sizeof(double) * dd);
        else memset(S, 0, sizeof(double) * dd);
        if (dense_T(family)) {
            memset(Tc, 0, sizeof(double) * tn);
            for (int i = 0; i < dk; ++i) Tc[(size_t)i * dk + i] = 1.0;
        } else {
            for (size_t e = 0; e < tn; ++e) Tc[e] = 1.0;
        }
        for (int j = cu_chain[r]; j < cu_chain[r + 1]; ++j) {
            const int p = seg_idx[j];
            if (p < 0 || p >= n_pairs) { bad = 1; break; }
            if (T_out) { /* Tc <- T_p Tc */
                const double* Tp = T_tab + ((size_t)p * LH + lh) * tn;
                double* Tn = Tc + tn;
                if (dense_T(family)) {
                    for (int i = 0; i < dk; ++i)
                        for (int c = 0; c < dk; ++c) {
                            double acc = 0.0;
                            for (int m = 0; m < dk; ++m) acc += Tp[(size_t)i * dk + m] * Tc[(size_t)m * dk + c];
                            Tn[(size_t)i * dk + c] = acc;
                        }
                } else {
                    for (size_t e = 0; e < tn; ++e) Tn[e] = Tp[e] * Tc[e];
                }
                memcpy(Tc, Tn, sizeof(double) * tn);
            }
            const double* Si = S_tab + ((size_t)p * LH + lh) * dd;
            if (naive || family == OR_VANILLA) {
                for (size_t e = 0; e < dd; ++e) N[e] = S[e];
            } else if (dense_T(family)) {
                const double* Ti = T_tab + ((size_t)p * LH + lh) * (size_t)dk * dk;
                for (int i = 0; i < dk; ++i)
                    for (int c = 0; c < dv; ++c) {
                        double s = 0.0;
                        for (int m = 0; m < dk; ++m) s += Ti[(size_t)i * dk + m] * S[(size_t)m * dv + c];
                        N[(size_t)i * dv + c] = s;
                    }
            } else if (scalar_T(family)) {
                const double ts = T_tab[(size_t)p * LH + lh];
                for (size_t e = 0; e < dd; ++e) N[e] = ts * S[e];
            } else { /* GLA */
                const double* tv = T_tab + ((size_t)p * LH + lh) * (size_t)dk;
                for (int i = 0; i < dk; ++i)
                    for (int c = 0; c < dv; ++c) N[(size_t)i * dv + c] = tv[i] * S[(size_t)i * dv + c];
            }
            for (size_t e = 0; e < dd; ++e) S[e] = N[e] + Si[e];
        }
        memcpy(S_out + (size_t)it * dd, S, sizeof(double) * dd);
        if (T_out) memcpy(T_out + (size_t)it * tn, Tc, sizeof(double) * tn);
        free(S); free(N); free(Tc);
    }
    return bad;
}

/* ------------------------------------------------------------------ seam -- */

/*
 * Seam-window advance [AB2]: for seam r, start from state_in[r] (or zero when
 * state_in is NULL), run the family's token loop over the seam tokens
 * [cu_seam[r], cu_seam[r+1]) of the packed seam-token arrays and emit, after
 * each token's own write, o_t = S_t^T q_t into row t of o_out
 * ([n_layers][n_tokens][n_heads][dv]).  The end state goes to state_out.
 * With one seam covering a whole request from zero this is the full
 * sequential recurrence.
 */
int oracle_seam(int family, int n_layers, int n_heads, int dk, int dv,
                int n_seams, const int* cu_seam, long long n_tokens,
                const float* q, const float* k, const float* v,
                const float* alpha, const float* beta, const float* gamma, const float* g,
                const double* state_in, double* state_out, double* o_out, int n_threads)
{
    if (check_common(family, n_layers, n_heads, dk, dv) || n_seams < 0) return 1;
    or_inputs in = {family, n_layers, n_heads, dk, dv, n_tokens, q, k, v, alpha, beta, gamma, g};
    const long long LH = (long long)n_layers * n_heads;
    const long long n_items = (long long)n_seams * LH;
    const size_t dd = (size_t)dk * dv;
    int bad = 0;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
#endif
    for (long long it = 0; it < n_items; ++it) {
        const int head = (int)(it % n_heads);
        const int layer = (int)((it / n_heads) % n_layers);
        const int r = (int)(it / LH);
        double* S = (double*)malloc(sizeof(double) * dd);
        double* kb = (double*)malloc(sizeof(double) * (size_t)(dk + dv + dk + dk + (dk > dv ? dk : dv)));
        if (!S || !kb) { bad = 1; free(S); free(kb); continue; }
        double *vb = kb + dk, *gb = vb + dv, *qb = gb + dk, *tmp = qb + dk;
        if (state_in) memcpy(S, state_in + (size_t)it * dd, sizeof(double) * dd);
        else memset(S, 0, sizeof(double) * dd);
        for (long long t = cu_seam[r]; t < cu_seam[r + 1]; ++t) {
            token_step(&in, layer, t, head, S, NULL, NULL, NULL, kb, vb, gb, tmp);
            const long long row = ((long long)layer * n_tokens + t) * n_heads + head;
            read_vec(q, row * dk, dk, qb);
            for (int c = 0; c < dv; ++c) {
                double s = 0.0;
                for (int i = 0; i < dk; ++i) s += S[(size_t)i * dv + c] * qb[i];
                o_out[row * dv + c] = s;
            }
        }
        memcpy(state_out + (size_t)it * dd, S, sizeof(double) * dd);
        free(S); free(kb);
    }
    return bad;
}

/* ------------------------------------------------------------ re-rotation -- */

/*
 * State re-rotation for variants whose keys carry RoPE ([AB]: the "state
 * re-rotation" patch).  The page names the patch only; this restates it from
 * the recurrences.  A segment moved by delta positions sees every key as
 * R k, R = R(delta) the rotary rotation; for a family whose per-token
 * transition is built from k k^T and scalars (GDN, RetNet, Mamba2, vanilla)
 * that maps each transition A to R A R^T and each write k v^T to R k v^T, so
 * the cached pair becomes (R T R^T, R S).  R acts on the first rotary_dim
 * features in rotate-half pairs: for i < h = rotary_dim / 2 the pair
 * (x_i, x_{i+h}) turns by the angle delta * base^(-2i / rotary_dim).
 * R is formed here as an explicit dk x dk matrix and applied by plain matrix
 * products.  T (dense families only, else NULL) and S are rewritten in place:
 *   T [n_pairs][n_layers][n_heads][dk][dk], S [...][dk][dv], delta [n_pairs].
 */
int oracle_rope(int family, int n_layers, int n_heads, int dk, int dv, int n_pairs,
                int rotary_dim, double base, const long long* delta, double* T, double* S)
{
    if (check_common(family, n_layers, n_heads, dk, dv) || n_pairs < 0) return 1;
    if (family == OR_GLA || family == OR_KDA) return 1; /* per-channel gates do not commute with R */
    if (rotary_dim < 2 || rotary_dim > dk || (rotary_dim & 1)) return 1;
    if (dense_T(family) != (T != NULL)) return 1;
    const long long LH = (long long)n_layers * n_heads;
    const int h = rotary_dim / 2;
    int bad = 0;
    for (int p = 0; p < n_pairs && !bad; ++p) {
        double* R = (double*)calloc((size_t)dk * dk, sizeof(double));
        double* tmp = (double*)malloc(sizeof(double) * (size_t)dk * (dk > dv ? dk : dv));
        if (!R || !tmp) { bad = 1; free(R); free(tmp); break; }
        for (int i = 0; i < dk; ++i) R[(size_t)i * dk + i] = 1.0;
        for (int i = 0; i < h; ++i) {
            const double a = (double)delta[p] * pow(base, -2.0 * i / rotary_dim);
            const double c = cos(a), sn = sin(a);
            R[(size_t)i * dk + i] = c;
            R[(size_t)i * dk + i + h] = -sn;
            R[(size_t)(i + h) * dk + i] = sn;
            R[(size_t)(i + h) * dk + i + h] = c;
        }
        for (long long lh = 0; lh < LH; ++lh) {
            double* Sp = S + ((size_t)p * LH + lh) * (size_t)dk * dv;
            for (int i = 0; i < dk; ++i) /* tmp = R S */
                for (int j = 0; j < dv; ++j) {
                    double acc = 0.0;
                    for (int m = 0; m < dk; ++m) acc += R[(size_t)i * dk + m] * Sp[(size_t)m * dv + j];
                    tmp[(size_t)i * dv + j] = acc;
                }
            memcpy(Sp, tmp, sizeof(double) * (size_t)dk * dv);
            if (T) {
                double* Tp = T + ((size_t)p * LH + lh) * (size_t)dk * dk;
                for (int i = 0; i < dk; ++i) /* tmp = R T */
                    for (int j = 0; j < dk; ++j) {
                        double acc = 0.0;
                        for (int m = 0; m < dk; ++m) acc += R[(size_t)i * dk + m] * Tp[(size_t)m * dk + j];
                        tmp[(size_t)i * dk + j] = acc;
                    }
                for (int i = 0; i < dk; ++i) /* T = tmp R^T */
                    for (int j = 0; j < dk; ++j) {
                        double acc = 0.0;
                        for (int m = 0; m < dk; ++m) acc += tmp[(size_t)i * dk + m] * R[(size_t)j * dk + m];
                        Tp[(size_t)i * dk + j] = acc;
                    }
            }
        }
        free(R); free(tmp);
    }
    return bad;
}

/* ------------------------------------------------------ conv-state warm-up -- */

/*
 * Conv-state warm-up for variants with a short causal convolution on the
 * inputs of the linear layers ([AB]: the "conv-state warm-up" patch, named
 * only).  A depthwise causal convolution of width K gives token t of channel
 * c the value y_t = act(bias_c + sum_{j<K} w[c][j] x_{t-K+1+j}); at a seam
 * window the K-1 inputs before the window come from the NEW prefix (hist),
 * not from the cached segment's own past.  Inputs, fp32 widened to double:
 *   x     [n_layers][n_tokens][C]  the windows' raw inputs, packed by window
 *   hist  [n_seams][n_layers][K-1][C]  the K-1 raw inputs before each window
 *         (oldest first), NULL for zeros (a sequence start)
 *   w     [n_layers][C][K] (tap K-1 multiplies the current token), bias
 *         [n_layers][C] or NULL; act 0 = identity, 1 = SiLU x / (1 + e^-x).
 * Output y [n_layers][n_tokens][C].
 */
int oracle_conv(int n_layers, int C, int K, int n_seams, const int* cu_seam, long long n_tokens,
                const float* x, const float* hist, const float* w, const float* bias, int act, double* y)
{
    if (n_layers <= 0 || C <= 0 || K < 1 || n_seams < 0) return 1;
    for (int r = 0; r < n_seams; ++r)
        for (int l = 0; l < n_layers; ++l)
            for (long long t = cu_seam[r]; t < cu_seam[r + 1]; ++t)
                for (int c = 0; c < C; ++c) {
                    double acc = bias ? (double)bias[(size_t)l * C + c] : 0.0;
                    for (int j = 0; j < K; ++j) {
                        const long long src = t - (K - 1) + j; /* token index in the window's frame */
                        double xv;
                        if (src >= cu_seam[r]) {
                            xv = (double)x[((size_t)l * n_tokens + src) * C + c];
                        } else {
                            const long long hi = (K - 1) - (cu_seam[r] - src); /* 0 = oldest */
                            xv = hist ? (double)hist[(((size_t)r * n_layers + l) * (K - 1) + hi) * C + c] : 0.0;
                        }
                        acc += (double)w[((size_t)l * C + c) * K + j] * xv;
                    }
                    y[((size_t)l * n_tokens + t) * C + c] = act ? acc / (1.0 + exp(-acc)) : acc;
                }
    return 0;
}

int oracle_version(void) { return 5; }
