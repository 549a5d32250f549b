"""Pins of the fp64 oracle against what the pages and the mathematics fix.

None of these re-types the oracle's token loop: each compares it with a
closed form, an invariant, a library routine on a special case, a value the
pages print, or a brute-force product of explicit matrices.  Each is chosen so
that a plausible slip (dropped decay, wrong sign of the erase term, S vs S^T,
wrong multiplication order of T, write term scaled by alpha) fails at least one.
"""
import json
import os

import numpy as np
import pytest

from oracle import oracle as orc

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def unit_rows(rng, shape):
    x = rng.standard_normal(shape)
    return (x / np.linalg.norm(x, axis=-1, keepdims=True)).astype(np.float32)


def hadamard_keys(rng, n, d=16):
    """n exactly orthonormal keys: rows of a d x d Hadamard matrix / sqrt(d)
    with random signs (entries +-1/4 at d=16, exact in binary)."""
    from scipy.linalg import hadamard
    H = hadamard(d).astype(np.float64) / np.sqrt(d)
    rows = rng.permutation(d)[:n]
    return (H[rows] * rng.choice([-1.0, 1.0], size=(n, 1))).astype(np.float32)


def one_head(x):
    """[n_tok][d] -> [1][n_tok][1][d]"""
    return np.asarray(x, np.float32)[None, :, None, :]


def gates(x):
    return np.asarray(x, np.float32)[None, :, None]


# ---------------------------------------------------------------- GDN ----

def test_gdn_single_token_is_projector_and_retrieves():
    """alpha=1, beta=1, |k|=1: T = I - k k^T is a rank-(d-1) orthogonal
    projector with T k = 0; S = k v^T so that k^T S = v^T (delta-rule write)."""
    rng = np.random.default_rng(1)
    d = 16
    k = hadamard_keys(rng, 1)
    v = rng.standard_normal((1, d)).astype(np.float32)
    T, S = orc.build_pairs("gdn", one_head(k), one_head(v), [0, 1],
                           alpha=gates([1.0]), beta=gates([1.0]))
    T, S = T[0, 0, 0], S[0, 0, 0]
    kk = k[0].astype(np.float64)
    np.testing.assert_allclose(T @ T, T, atol=1e-12)
    np.testing.assert_allclose(T @ kk, 0.0, atol=1e-12)
    assert abs(np.trace(T) - (d - 1)) < 1e-12
    np.testing.assert_allclose(kk @ S, v[0], atol=1e-12)


def test_gdn_overwrite_same_key():
    """Delta rule with alpha=1, beta=1: writing (k, v1) then (k, v2) leaves
    S = k v2^T -- the second write erases the first."""
    rng = np.random.default_rng(2)
    d = 16
    k = hadamard_keys(rng, 1)
    v = rng.standard_normal((2, d)).astype(np.float32)
    _, S = orc.build_pairs("gdn", one_head(np.repeat(k, 2, 0)), one_head(v), [0, 2],
                           alpha=gates([1, 1]), beta=gates([1, 1]))
    np.testing.assert_allclose(S[0, 0, 0], np.outer(k[0], v[1]), atol=1e-12)


def test_gdn_determinant_closed_form():
    """det(alpha (I - beta k k^T)) = alpha^d (1 - beta) for |k| = 1, so
    det T_C = prod_t alpha_t^d (1 - beta_t) (numpy slogdet on the result)."""
    rng = np.random.default_rng(3)
    d, L = 16, 40
    k = unit_rows(rng, (L, d)).astype(np.float64)
    k32 = k.astype(np.float32)
    a = rng.uniform(0.9, 1.0, L).astype(np.float32)
    b = rng.uniform(0.0, 0.9, L).astype(np.float32)
    T, _ = orc.build_pairs("gdn", one_head(k32), one_head(rng.standard_normal((L, d))), [0, L],
                           alpha=gates(a), beta=gates(b))
    kn = np.linalg.norm(k32.astype(np.float64), axis=1) ** 2  # float32 keys are unit up to rounding
    want = np.sum(d * np.log(a.astype(np.float64)) + np.log1p(-b.astype(np.float64) * kn))
    sign, got = np.linalg.slogdet(T[0, 0, 0])
    assert sign > 0
    assert abs(got - want) < 1e-9


def test_gdn_orthonormal_keys_closed_form():
    """Orthonormal keys make the transitions commute:
    T = (prod alpha)(I - sum beta_t k_t k_t^T) and
    S = sum_t (prod_{s>t} alpha_s) beta_t k_t v_t^T  (the write term is not
    decayed by its own alpha_t)."""
    rng = np.random.default_rng(4)
    d, L = 16, 12
    K = hadamard_keys(rng, L)
    V = rng.standard_normal((L, d)).astype(np.float32)
    a = rng.uniform(0.5, 1.0, L).astype(np.float32)
    b = rng.uniform(0.0, 1.0, L).astype(np.float32)
    T, S = orc.build_pairs("gdn", one_head(K), one_head(V), [0, L], alpha=gates(a), beta=gates(b))
    Kd, Vd, ad, bd = (x.astype(np.float64) for x in (K, V, a, b))
    T_want = np.prod(ad) * (np.eye(d) - Kd.T @ np.diag(bd) @ Kd)
    later = np.array([np.prod(ad[t + 1:]) for t in range(L)])
    S_want = Kd.T @ np.diag(later * bd) @ Vd
    np.testing.assert_allclose(T[0, 0, 0], T_want, atol=1e-14)
    np.testing.assert_allclose(S[0, 0, 0], S_want, atol=1e-13)


def test_gdn_gate_special_cases():
    """alpha=1, beta=0: T = I, S = 0.  beta=0: T = (prod alpha) I, S = 0."""
    rng = np.random.default_rng(5)
    d, L = 16, 30
    k = unit_rows(rng, (L, d))
    v = rng.standard_normal((L, d)).astype(np.float32)
    a = rng.uniform(0.8, 1.0, L).astype(np.float32)
    T, S = orc.build_pairs("gdn", one_head(k), one_head(v), [0, L],
                           alpha=gates(np.ones(L)), beta=gates(np.zeros(L)))
    np.testing.assert_array_equal(T[0, 0, 0], np.eye(d))
    np.testing.assert_array_equal(S[0, 0, 0], 0.0)
    T, S = orc.build_pairs("gdn", one_head(k), one_head(v), [0, L],
                           alpha=gates(a), beta=gates(np.zeros(L)))
    np.testing.assert_allclose(T[0, 0, 0], np.prod(a.astype(np.float64)) * np.eye(d), rtol=1e-13)
    np.testing.assert_array_equal(S[0, 0, 0], 0.0)


def test_gdn_brute_force_explicit_matrices():
    """T_C is the ordered product A_L ... A_1 of explicit per-token matrices and
    S(C|0) = sum_t (A_L ... A_{t+1}) beta_t k_t v_t^T (latest token leftmost)."""
    rng = np.random.default_rng(6)
    d, L = 8, 24
    k = unit_rows(rng, (L, d))
    v = rng.standard_normal((L, d)).astype(np.float32)
    a = rng.uniform(0.7, 1.0, L).astype(np.float32)
    b = rng.uniform(0.0, 1.0, L).astype(np.float32)
    T, S = orc.build_pairs("gdn", one_head(k), one_head(v), [0, L], alpha=gates(a), beta=gates(b))
    kd, vd = k.astype(np.float64), v.astype(np.float64)
    A = [float(a[t]) * (np.eye(d) - float(b[t]) * np.outer(kd[t], kd[t])) for t in range(L)]
    def ordered_product(mats):  # mats in token order; latest ends up leftmost
        P = np.eye(d)
        for M in mats:
            P = M @ P
        return P

    T_bf = ordered_product(A)
    S_bf = np.zeros((d, d))
    for t in range(L):
        S_bf += ordered_product(A[t + 1:]) @ (float(b[t]) * np.outer(kd[t], vd[t]))
    np.testing.assert_allclose(T[0, 0, 0], T_bf, atol=1e-13)
    np.testing.assert_allclose(S[0, 0, 0], S_bf, atol=1e-12)


# ------------------------------------------------- composition (all families) --

def _family_inputs(fam, rng, n, d, H=2):
    k = unit_rows(rng, (1, n, H, d))
    v = rng.standard_normal((1, n, H, d)).astype(np.float32)
    kw = {}
    if fam == "gdn":
        kw["alpha"] = rng.uniform(0.95, 1.0, (1, n, H)).astype(np.float32)
        kw["beta"] = rng.uniform(0.0, 0.5, (1, n, H)).astype(np.float32)
    elif fam == "retnet":
        kw["gamma"] = np.array([[0.97, 0.995]], np.float32)[:, :H]
    elif fam == "gla":
        kw["g"] = rng.uniform(0.9, 1.0, (1, n, H, d)).astype(np.float32)
    elif fam == "kda":
        kw["g"] = rng.uniform(0.9, 1.0, (1, n, H, d)).astype(np.float32)
        kw["beta"] = rng.uniform(0.0, 0.5, (1, n, H)).astype(np.float32)
    elif fam == "mamba2":
        kw["alpha"] = rng.uniform(0.9, 1.0, (1, n, H)).astype(np.float32)
    return k, v, kw


def _T_apply(fam, T2, T1):
    """T(C1.C2) from T(C2), T(C1) by the family's product (T2 applied last)."""
    if fam in ("gdn", "kda"):
        return T2 @ T1
    return T2 * T1


@pytest.mark.parametrize("fam", ["gdn", "retnet", "gla", "vanilla", "kda", "mamba2"])
def test_associativity_build_equals_compose(fam):
    """The composition law of the aibase article: building C1.C2 in one pass
    equals composing the separately built pairs, S(C1.C2) = T(C2) S(C1) + S(C2),
    and the transition products chain as T(C1.C2) = T(C2) T(C1)."""
    rng = np.random.default_rng(7)
    d, n1, n2 = 16, 37, 53
    k, v, kw = _family_inputs(fam, rng, n1 + n2, d)
    T12, S12 = orc.build_pairs(fam, k, v, [0, n1 + n2], **kw)
    T, S = orc.build_pairs(fam, k, v, [0, n1, n1 + n2], **kw)
    S_c = orc.compose(fam, T, S, [0, 2], [0, 1])
    np.testing.assert_allclose(S_c[0], S12[0], atol=1e-12)
    if T is not None:
        np.testing.assert_allclose(_T_apply(fam, T[1], T[0]), T12[0], atol=1e-13)


def test_compose_from_start_state_equals_seam_from_that_state():
    """Running the token loop from a non-zero state S0 (the seam path) ends at
    T_C S0 + S(C|0) (compose with a start state)."""
    rng = np.random.default_rng(8)
    d, n = 16, 45
    k, v, kw = _family_inputs("gdn", rng, n, d)
    q = unit_rows(rng, (1, n, 2, d))
    S0 = rng.standard_normal((1, 1, 2, d, d))
    T, S = orc.build_pairs("gdn", k, v, [0, n], **kw)
    end_c = orc.compose("gdn", T, S, [0, 1], [0], S0=S0)
    end_s, _ = orc.seam("gdn", q, k, v, [0, n], state_in=S0, **kw)
    np.testing.assert_allclose(end_s, end_c, atol=1e-12)


def test_full_sequence_equals_chain_of_pairs_with_seams():
    """PIC reuse with seam windows: first segment cached whole, each internal
    segment's first w tokens advanced on the fly and its body composed; the
    end state and the seam-token outputs equal the full sequential run."""
    rng = np.random.default_rng(9)
    d, w = 16, 4
    lengths = [20, 33, 18]
    cu = np.cumsum([0] + lengths)
    n = int(cu[-1])
    k, v, kw = _family_inputs("gdn", rng, n, d, H=1)
    q = unit_rows(rng, (1, n, 1, d))
    S_full, o_full = orc.seam("gdn", q, k, v, [0, n], **kw)
    skip = [0, w, w]
    T, S = orc.build_pairs("gdn", k, v, cu, skip=skip, **kw)
    state = orc.compose("gdn", T, S, [0, 1], [0])
    for i in (1, 2):
        state, o = orc.seam("gdn", q, k, v, [int(cu[i]), int(cu[i]) + w], state_in=state, **kw)
        np.testing.assert_allclose(o[:, cu[i]:cu[i] + w], o_full[:, cu[i]:cu[i] + w], atol=1e-12)
        state = orc.compose("gdn", T, S, [0, 1], [i], S0=state)
    np.testing.assert_allclose(state, S_full, atol=1e-12)


def test_seam_output_uses_state_transpose_after_write():
    """o_t = S_t^T q_t with the token's own write included: with alpha=1,
    beta=1, orthonormal keys and q_t = k_t the output is v_t exactly."""
    rng = np.random.default_rng(10)
    d, L = 16, 10
    K = hadamard_keys(rng, L)
    V = rng.standard_normal((L, d)).astype(np.float32)
    _, o = orc.seam("gdn", one_head(K), one_head(K), one_head(V), [0, L],
                    alpha=gates(np.ones(L)), beta=gates(np.ones(L)))
    np.testing.assert_allclose(o[0, :, 0], V, atol=1e-13)


# ------------------------------------------------------ decay families ----

def test_retnet_closed_forms():
    """T = gamma^L exactly; S = K^T diag(gamma^(L-1-t)) V."""
    rng = np.random.default_rng(11)
    d, L, gm = 16, 64, np.float32(0.97)
    k = unit_rows(rng, (L, d))
    v = rng.standard_normal((L, d)).astype(np.float32)
    T, S = orc.build_pairs("retnet", one_head(k), one_head(v), [0, L], gamma=np.array([[gm]]))
    g64 = np.float64(gm)
    assert abs(T[0, 0, 0] - g64 ** L) <= 1e-15 * g64 ** L
    w = g64 ** (L - 1 - np.arange(L))
    np.testing.assert_allclose(S[0, 0, 0], k.astype(np.float64).T @ (w[:, None] * v.astype(np.float64)), atol=1e-12)


def test_retnet_naive_addition_reproduces_printed_22_percent():
    """The aibase article prints 22% for the naive-addition error on a RetNet
    slow-decay head at 256 tokens.  Composing through the oracle with and
    without T reproduces it, and equals 1 - gamma^256 for any prefix."""
    fx = json.load(open(os.path.join(GOLD, "retnet_naive_addition_22pct.json")))
    L2 = fx["segment_tokens"]
    gm = np.float32(1.0 - 2.0 ** fx["gamma_exponent"])
    rng = np.random.default_rng(12)
    d, L1 = 32, 300
    k = unit_rows(rng, (L1 + L2, d))
    v = rng.standard_normal((L1 + L2, d)).astype(np.float32)
    T, S = orc.build_pairs("retnet", one_head(k), one_head(v), [0, L1, L1 + L2], gamma=np.array([[gm]]))
    true = orc.compose("retnet", T, S, [0, 2], [0, 1])
    naive = orc.compose("retnet", T, S, [0, 2], [0, 1], naive=True)
    ratio = np.linalg.norm(naive - true) / np.linalg.norm(S[0])
    assert abs(ratio - (1.0 - np.float64(gm) ** L2)) < 1e-12
    assert abs(100.0 * ratio - fx["printed_percent"]) <= fx["rounding_half_width_percent"]


def test_gla_closed_forms_and_retnet_special_case():
    """GLA: T = prod_t g_t elementwise, row i of S is a scalar-decay sum with
    decay g[.,i]; with g constant per head GLA equals RetNet."""
    rng = np.random.default_rng(13)
    d, L = 16, 50
    k = unit_rows(rng, (L, d))
    v = rng.standard_normal((L, d)).astype(np.float32)
    g = rng.uniform(0.8, 1.0, (L, d)).astype(np.float32)
    T, S = orc.build_pairs("gla", one_head(k), one_head(v), [0, L], g=one_head(g))
    gd = g.astype(np.float64)
    np.testing.assert_allclose(T[0, 0, 0], np.prod(gd, axis=0), rtol=1e-13)
    later = np.concatenate([np.cumprod(gd[::-1], axis=0)[::-1][1:], np.ones((1, d))])  # prod_{s>t} g_s
    S_want = (later * k.astype(np.float64)).T @ v.astype(np.float64)
    np.testing.assert_allclose(S[0, 0, 0], S_want, atol=1e-12)
    gm = np.float32(0.93)
    _, S_gla = orc.build_pairs("gla", one_head(k), one_head(v), [0, L], g=one_head(np.full((L, d), gm, np.float32)))
    _, S_ret = orc.build_pairs("retnet", one_head(k), one_head(v), [0, L], gamma=np.array([[gm]]))
    np.testing.assert_allclose(S_gla, S_ret, atol=1e-13)


def test_vanilla_addition_is_exact():
    """Plain linear attention: S = K^T V, and naive addition equals the true
    composition (the aibase article: addition is exact there)."""
    rng = np.random.default_rng(14)
    d, n1, n2 = 16, 30, 40
    k = unit_rows(rng, (n1 + n2, d))
    v = rng.standard_normal((n1 + n2, d)).astype(np.float32)
    _, S = orc.build_pairs("vanilla", one_head(k), one_head(v), [0, n1, n1 + n2])
    np.testing.assert_allclose(S[0, 0, 0], k[:n1].astype(np.float64).T @ v[:n1].astype(np.float64), atol=1e-12)
    a = orc.compose("vanilla", None, S, [0, 2], [0, 1])
    b = orc.compose("vanilla", None, S, [0, 2], [0, 1], naive=True)
    np.testing.assert_array_equal(a, b)


def test_gdn_naive_addition_is_not_exact():
    """For GDN, dropping T(C2) leaves a structural error (the strawman)."""
    rng = np.random.default_rng(15)
    d, n1, n2 = 16, 30, 40
    k, v, kw = _family_inputs("gdn", rng, n1 + n2, d)
    T, S = orc.build_pairs("gdn", k, v, [0, n1, n1 + n2], **kw)
    true = orc.compose("gdn", T, S, [0, 2], [0, 1])
    naive = orc.compose("gdn", T, S, [0, 2], [0, 1], naive=True)
    assert np.linalg.norm(naive - true) > 0.05 * np.linalg.norm(true)


# --------------------------------------------------------------- misc -----

def test_zero_length_segment_is_identity_pair():
    rng = np.random.default_rng(16)
    d = 16
    k, v, kw = _family_inputs("gdn", rng, 5, d)
    T, S = orc.build_pairs("gdn", k, v, [0, 0, 5], **kw)
    np.testing.assert_array_equal(T[0, 0, 0], np.eye(d))
    np.testing.assert_array_equal(S[0], 0.0)


def test_scaled_storage_roundtrip():
    rng = np.random.default_rng(17)
    T = rng.standard_normal((3, 4, 4)) * np.array([1e-60, 1.0, 1e30])[:, None, None]
    T[1] = 0.0
    m, e = orc.f64_to_scaled(T)
    back = orc.scaled_to_f64(m, e)
    np.testing.assert_allclose(back, T, rtol=1e-7, atol=0)
    assert np.all(np.abs(m[[0, 2]]).max(axis=(-2, -1)) < 1.0)
    assert np.all(np.abs(m[[0, 2]]).max(axis=(-2, -1)) >= 0.5)


def test_rel_fro():
    ref = np.ones((2, 3, 3))
    x = ref.copy()
    x[1] *= 1.01
    r = orc.rel_fro(x, ref, (-2, -1))
    np.testing.assert_allclose(r, [0.0, 0.01], atol=1e-15)


# ------------------------------------------------------------ KDA, Mamba2 ----

def test_kda_brute_force_explicit_matrices():
    """KDA: T_C = A_L ... A_1 with explicit per-token matrices
    A_t = (I - b_t k_t k_t^T) Diag(a_t) (the gate first, then the delta
    projection), S(C|0) = sum_t (A_L ... A_{t+1}) b_t k_t v_t^T."""
    rng = np.random.default_rng(21)
    d, L = 8, 24
    k = unit_rows(rng, (L, d))
    v = rng.standard_normal((L, d)).astype(np.float32)
    a = rng.uniform(0.5, 1.0, (L, d)).astype(np.float32)
    b = rng.uniform(0.0, 1.0, L).astype(np.float32)
    T, S = orc.build_pairs("kda", one_head(k), one_head(v), [0, L], g=one_head(a), beta=gates(b))
    kd, vd, ad = k.astype(np.float64), v.astype(np.float64), a.astype(np.float64)
    A = [(np.eye(d) - float(b[t]) * np.outer(kd[t], kd[t])) @ np.diag(ad[t]) for t in range(L)]
    def ordered_product(mats):
        P = np.eye(d)
        for M in mats:
            P = M @ P
        return P

    S_bf = np.zeros((d, d))
    for t in range(L):
        S_bf += ordered_product(A[t + 1:]) @ (float(b[t]) * np.outer(kd[t], vd[t]))
    np.testing.assert_allclose(T[0, 0, 0], ordered_product(A), atol=1e-13)
    np.testing.assert_allclose(S[0, 0, 0], S_bf, atol=1e-12)
    # the gate does not commute with the projection: the other order differs
    A_swapped = [np.diag(ad[t]) @ (np.eye(d) - float(b[t]) * np.outer(kd[t], kd[t])) for t in range(L)]
    Tsw = ordered_product(A_swapped)
    assert np.linalg.norm(Tsw - T[0, 0, 0]) > 1e-2 * np.linalg.norm(T[0, 0, 0])


def test_kda_with_a_uniform_gate_is_gdn():
    """A per-channel gate equal in every channel is GDN's scalar gate:
    (I - b k k^T) (a I) = a (I - b k k^T); pair and seam outputs agree."""
    rng = np.random.default_rng(22)
    d, L = 16, 70
    k = unit_rows(rng, (1, L, 2, d))
    v = rng.standard_normal((1, L, 2, d)).astype(np.float32)
    q = unit_rows(rng, (1, L, 2, d))
    a = rng.uniform(0.8, 1.0, (1, L, 2)).astype(np.float32)
    b = rng.uniform(0.0, 1.0, (1, L, 2)).astype(np.float32)
    g = np.repeat(a[..., None], d, axis=-1)
    Tk, Sk = orc.build_pairs("kda", k, v, [0, 30, L], g=g, beta=b)
    Tg, Sg = orc.build_pairs("gdn", k, v, [0, 30, L], alpha=a, beta=b)
    np.testing.assert_allclose(Tk, Tg, atol=1e-13)
    np.testing.assert_allclose(Sk, Sg, atol=1e-12)
    _, ok = orc.seam("kda", q, k, v, [0, L], g=g, beta=b)
    _, og = orc.seam("gdn", q, k, v, [0, L], alpha=a, beta=b)
    np.testing.assert_allclose(ok, og, atol=1e-12)


def test_kda_without_writes_is_the_gate_product():
    """b = 0: no erase and no write, so T = Diag(prod_t a_t) and S = 0."""
    rng = np.random.default_rng(23)
    d, L = 16, 40
    k = unit_rows(rng, (L, d))
    v = rng.standard_normal((L, d)).astype(np.float32)
    a = rng.uniform(0.8, 1.0, (L, d)).astype(np.float32)
    T, S = orc.build_pairs("kda", one_head(k), one_head(v), [0, L], g=one_head(a),
                           beta=gates(np.zeros(L)))
    np.testing.assert_allclose(T[0, 0, 0], np.diag(np.prod(a.astype(np.float64), axis=0)), rtol=1e-13, atol=0)
    assert np.all(S == 0)


def test_mamba2_closed_forms_and_retnet_special_case():
    """Mamba2: T = prod_t a_t, S = sum_t (prod_{s>t} a_s) k_t v_t^T; with a
    constant gate it is RetNet."""
    rng = np.random.default_rng(24)
    d, L = 16, 60
    k = unit_rows(rng, (L, d))
    v = rng.standard_normal((L, d)).astype(np.float32)
    a = rng.uniform(0.7, 1.0, L).astype(np.float32)
    T, S = orc.build_pairs("mamba2", one_head(k), one_head(v), [0, L], alpha=gates(a))
    ad = a.astype(np.float64)
    np.testing.assert_allclose(T[0, 0, 0], np.prod(ad), rtol=1e-13)
    later = np.concatenate([np.cumprod(ad[::-1])[::-1][1:], [1.0]])  # prod_{s>t} a_s
    S_want = (later[:, None] * k.astype(np.float64)).T @ v.astype(np.float64)
    np.testing.assert_allclose(S[0, 0, 0], S_want, atol=1e-12)
    gm = np.float32(0.95)
    Tm, Sm = orc.build_pairs("mamba2", one_head(k), one_head(v), [0, L], alpha=gates(np.full(L, gm)))
    Tr, Sr = orc.build_pairs("retnet", one_head(k), one_head(v), [0, L], gamma=np.array([[gm]]))
    np.testing.assert_allclose(Tm, Tr, rtol=1e-13)
    np.testing.assert_allclose(Sm, Sr, atol=1e-13)


# ------------------------------------------------- chain transition (T out) ----

@pytest.mark.parametrize("fam", ["gdn", "retnet", "gla", "kda", "mamba2"])
def test_chain_transition_is_the_pair_of_the_concatenation(fam):
    """A chain's own transition product is the T_C of the concatenated
    segments (one-pass build), its zero-start S is their S(C|0), so the chain
    is itself a cached pair: from a start S0 it gives T_chain S0 + S_chain, and
    pairs of chains compose like pairs (tree reduction).  An empty chain is
    the identity pair."""
    rng = np.random.default_rng(41)
    d, lens = 8, [20, 7, 33, 15]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    k, v, kw = _family_inputs(fam, rng, int(cu[-1]), d)
    T_all, S_all = orc.build_pairs(fam, k, v, [0, int(cu[-1])], **kw)
    T, S = orc.build_pairs(fam, k, v, cu, **kw)
    S_c, T_c = orc.compose(fam, T, S, [0, 4, 4], [0, 1, 2, 3], want_T=True)
    np.testing.assert_allclose(T_c[0], T_all[0], atol=1e-13)
    np.testing.assert_allclose(S_c[0], S_all[0], atol=1e-12)
    eye = np.broadcast_to(np.eye(d), T_c[1].shape) if fam in ("gdn", "kda") else np.ones_like(T_c[1])
    np.testing.assert_array_equal(T_c[1], eye)
    assert np.all(S_c[1] == 0)
    S0 = rng.standard_normal((1,) + S.shape[1:])
    S_from = orc.compose(fam, T, S, [0, 4], [0, 1, 2, 3], S0=S0)
    TS0 = np.einsum("lhij,lhjc->lhic", T_c[0], S0[0]) if fam in ("gdn", "kda") else (
        T_c[0][..., None] * S0[0] if fam == "gla" else T_c[0][..., None, None] * S0[0])
    np.testing.assert_allclose(S_from[0], TS0 + S_c[0], atol=1e-12)
    # pair of pairs: (p0 p1) and (p2 p3) as two chains, then their two pairs
    S_h, T_h = orc.compose(fam, T, S, [0, 2, 4], [0, 1, 2, 3], want_T=True)
    S_t, T_t = orc.compose(fam, T_h, S_h, [0, 2], [0, 1], want_T=True)
    np.testing.assert_allclose(T_t[0], T_all[0], atol=1e-13)
    np.testing.assert_allclose(S_t[0], S_all[0], atol=1e-12)


# ------------------------------------------------------- RoPE re-rotation ----

def rope_matrix(d, rdim, delta, base=10000.0):
    """The rotary rotation as an explicit matrix, built from its definition
    x -> x cos(a) + rotate_half(x) sin(a) on the first rdim features."""
    h = rdim // 2
    ang = delta * base ** (-2.0 * np.arange(h) / rdim)
    R = np.eye(d)
    for i in range(h):
        x = np.zeros(d); x[i] = 1.0
        y = np.zeros(d); y[i + h] = 1.0
        # images of the basis vectors e_i and e_{i+h}
        R[:, i] = x * np.cos(ang[i]) + y * np.sin(ang[i])
        R[:, i + h] = y * np.cos(ang[i]) - x * np.sin(ang[i])
    return R


@pytest.mark.parametrize("fam", ["gdn", "retnet", "mamba2", "vanilla"])
@pytest.mark.parametrize("rdim", [16, 8])
def test_rope_rerotation_equals_building_with_rotated_keys(fam, rdim):
    """Moving a segment by delta positions rotates every key by R(delta);
    building the pair from the rotated keys gives the re-rotated pair
    (R T R^T, R S), whatever the segment's content.  (The rotated keys are
    rounded to float32 when the oracle reads them: the two sides then differ
    by that rounding, ~1e-7 relative.)"""
    rng = np.random.default_rng(51)
    d, n = 16, 40
    k, v, kw = _family_inputs(fam, rng, n, d)
    cu = [0, 25, n]
    deltas = [1000, -37]
    T, S = orc.build_pairs(fam, k, v, cu, **kw)
    dense = fam == "gdn"
    Tr, Sr = orc.rope(fam, T if dense else None, S, deltas, rotary_dim=rdim)
    for p, (a, b) in enumerate(zip(cu[:-1], cu[1:])):
        R = rope_matrix(d, rdim, deltas[p])
        k_rot = np.einsum("ij,lthj->lthi", R, k[:, a:b].astype(np.float64)).astype(np.float32)
        sl = {key: (val[:, a:b] if val.ndim >= 3 else val) for key, val in kw.items()}
        T2, S2 = orc.build_pairs(fam, k_rot, v[:, a:b], [0, b - a], **sl)
        np.testing.assert_allclose(Sr[p], S2[0], rtol=0, atol=2e-6 * np.abs(S2[0]).max())
        if dense:
            np.testing.assert_allclose(Tr[p], T2[0], rtol=0, atol=2e-6)
        elif T is not None:
            np.testing.assert_array_equal(T2[0], T[p])  # a scalar transition does not see R


def test_rope_rotation_properties():
    """R is orthogonal, R(0) = I, R(d1) R(d2) = R(d1 + d2), and re-rotating
    twice equals re-rotating once by the summed shift."""
    rng = np.random.default_rng(52)
    d = 16
    for rdim in (16, 10):
        R1, R2 = rope_matrix(d, rdim, 123), rope_matrix(d, rdim, -40)
        np.testing.assert_allclose(R1 @ R1.T, np.eye(d), atol=1e-12)
        np.testing.assert_allclose(R1 @ R2, rope_matrix(d, rdim, 83), atol=1e-9)
        np.testing.assert_allclose(rope_matrix(d, rdim, 0), np.eye(d), atol=0)
    T = rng.standard_normal((1, 1, 2, d, d))
    S = rng.standard_normal((1, 1, 2, d, d))
    Ta, Sa = orc.rope("gdn", T, S, [123], rotary_dim=10)
    Tb, Sb = orc.rope("gdn", Ta, Sa, [-40], rotary_dim=10)
    Tc, Sc = orc.rope("gdn", T, S, [83], rotary_dim=10)
    np.testing.assert_allclose(Tb, Tc, atol=1e-9)
    np.testing.assert_allclose(Sb, Sc, atol=1e-9)
    R = rope_matrix(d, 10, 123)
    np.testing.assert_allclose(Sa[0, 0, 1], R @ S[0, 0, 1], atol=1e-12)
    np.testing.assert_allclose(Ta[0, 0, 1], R @ T[0, 0, 1] @ R.T, atol=1e-12)


# ------------------------------------------------------ conv-state warm-up ----

def test_conv_warmup_equals_convolution_of_the_whole_sequence():
    """A window whose history is the true K-1 inputs before it gets the same
    outputs as the causal convolution of the whole sequence (np.convolve per
    channel, zero padding at the start); with SiLU, y = z / (1 + e^-z)."""
    rng = np.random.default_rng(61)
    L, C, K, n = 2, 6, 4, 50
    xs = rng.standard_normal((L, n, C)).astype(np.float32)
    w = rng.standard_normal((L, C, K)).astype(np.float32)
    b = rng.standard_normal((L, C)).astype(np.float32)
    # the whole sequence as windows: [0, 20) from a sequence start, [20, 28), [28, 50)
    starts = [0, 20, 28, 50]
    hist = np.zeros((3, L, K - 1, C), np.float32)
    for r, s0 in enumerate(starts[:-1]):
        for j in range(K - 1):
            src = s0 - (K - 1) + j
            if src >= 0:
                hist[r, :, j] = xs[:, src]
    for act in (0, 1):
        y = orc.conv(xs, starts, w, hist=hist, bias=b, act=act)
        for l in range(L):
            for c in range(C):
                z = np.convolve(xs[l, :, c].astype(np.float64), w[l, c, ::-1].astype(np.float64))[:n] + b[l, c]
                want = z / (1.0 + np.exp(-z)) if act else z
                np.testing.assert_allclose(y[l, :, c], want, atol=1e-12)
    # without the true history the first K-1 outputs of a window differ, the rest do not
    y0 = orc.conv(xs, starts, w, hist=None, bias=b, act=0)
    y1 = orc.conv(xs, starts, w, hist=hist, bias=b, act=0)
    assert np.abs(y0[:, 20:23] - y1[:, 20:23]).max() > 1e-3
    np.testing.assert_array_equal(y0[:, 23:28], y1[:, 23:28])
