"""GPU parity of hypic_compose's chain transition output (T_out) against the
fp64 oracle: each chain's own transition T_{p_n} ... T_{p_1} for every family
with a transition, with and without a start state, an empty chain, strong
decay (the product far below the float32 range, kept by its exponent), and a
two-level tree: chains of pairs, then a chain of those chains' pairs."""
import numpy as np
import pytest

from linear_attn_state_hypic_gb300 import synth
from oracle import oracle as orc
from tests.helpers import TOL_F32, assert_rel, dev, gdn_T64, host

pytestmark = pytest.mark.gpu

DENSE = ("gdn", "kda")


@pytest.fixture(scope="module")
def B():
    from linear_attn_state_hypic_gb300 import binding
    return binding


def family_gates(fam, rng, L, n, H, dk, lo):
    if fam == "gdn":
        return {"alpha": rng.uniform(lo, 1.0, (L, n, H)).astype(np.float32),
                "beta": rng.uniform(0.0, 0.3, (L, n, H)).astype(np.float32)}
    if fam == "kda":
        return {"g": rng.uniform(lo, 1.0, (L, n, H, dk)).astype(np.float32),
                "beta": rng.uniform(0.0, 0.3, (L, n, H)).astype(np.float32)}
    if fam == "mamba2":
        return {"alpha": rng.uniform(lo, 1.0, (L, n, H)).astype(np.float32)}
    if fam == "gla":
        return {"g": rng.uniform(lo, 1.0, (L, n, H, dk)).astype(np.float32)}
    return {"gamma": rng.uniform(lo, 1.0, (L, H)).astype(np.float32)}


def pair_table(fam, seed, n_pairs, L, H, dk, dv, seg_len, lo):
    """Oracle-built pairs, stored as the GPU stores them: (T as stored, T_exp
    or None, S float32, T as float64 with the exponent applied)."""
    rng = np.random.default_rng(seed)
    cu = synth.cu_from_lengths([seg_len] * n_pairs)
    n = int(cu[-1])
    k = synth._unit_rows(rng, (L, n, H, dk))
    v = rng.standard_normal((L, n, H, dv)).astype(np.float32)
    T, S = orc.build_pairs(fam, k, v, cu, **family_gates(fam, rng, L, n, H, dk, lo))
    if fam in DENSE:
        Tm, Te = orc.f64_to_scaled(T)
        return Tm, Te, S.astype(np.float32), orc.scaled_to_f64(Tm, Te)
    T32 = T.astype(np.float32)
    return T32, None, S.astype(np.float32), T32.astype(np.float64)


def T_of(fam, T, T_exp):
    return gdn_T64(T, T_exp) if fam in DENSE else host(T)


def check_T(fam, got, ref, what):
    if fam in DENSE:
        assert_rel(got, ref, TOL_F32, what=what)
    elif fam == "gla":
        assert_rel(got, ref, TOL_F32, axes=(-1,), what=what)
    else:
        assert_rel(got[..., None], ref[..., None], TOL_F32, axes=(-1,), what=what)


@pytest.mark.parametrize("fam,dk,dv", [("gdn", 128, 128), ("gdn", 32, 32), ("kda", 64, 64), ("kda", 128, 128),
                                       ("retnet", 32, 32), ("mamba2", 64, 16), ("gla", 64, 16), ("gla", 16, 32)])
@pytest.mark.parametrize("with_s0", [False, True])
def test_chain_transition(B, fam, dk, dv, with_s0):
    L, H, P = 2, 2, 5
    Tt, Te, S32, T64 = pair_table(fam, 90 + dk + dv, P, L, H, dk, dv, 40, lo=0.99)
    chains = [[0, 1, 2, 3, 4], [4, 2], [], [1, 1, 1]]
    cu = np.array([0] + list(np.cumsum([len(c) for c in chains])), np.int32)
    idx = np.array([i for c in chains for i in c], np.int32)
    rng = np.random.default_rng(dk)
    S0 = (rng.standard_normal((len(chains), L, H, dk, dv)) / np.sqrt(dk)).astype(np.float32) if with_s0 else None
    out, T, T_exp = B.compose(fam, dev(S32), cu, idx, T_tab=dev(Tt), T_exp_tab=None if Te is None else dev(Te),
                              S0=dev(S0), want_T=True)
    B.check_device()
    S_ref, T_ref = orc.compose(fam, T64, S32.astype(np.float64), cu, idx, S0=S0, want_T=True)
    assert_rel(host(out), S_ref, TOL_F32, what=f"{fam} chain end state")
    got = T_of(fam, T, T_exp)
    check_T(fam, got, T_ref, f"{fam} chain transition")
    np.testing.assert_array_equal(got[2], T_ref[2])  # the empty chain: the identity


@pytest.mark.parametrize("fam,d", [("gdn", 32), ("kda", 32), ("gdn", 128)])
def test_chain_transition_strong_decay(B, fam, d):
    """Pairs of 256-token segments with strong decay: a chain of 8 multiplies
    their transitions far below the float32 range; the exponent keeps it (at
    d = 128 on the tensor-core compose's transition mode)."""
    L, H = 1, 2
    Tt, Te, S32, T64 = pair_table(fam, 7, 4, L, H, d, d, 256, lo=0.8)
    cu, idx = np.array([0, 8], np.int32), np.array([0, 1, 2, 3, 3, 2, 1, 0], np.int32)
    out, T, T_exp = B.compose(fam, dev(S32), cu, idx, T_tab=dev(Tt), T_exp_tab=dev(Te), want_T=True)
    B.check_device()
    S_ref, T_ref = orc.compose(fam, T64, S32.astype(np.float64), cu, idx, want_T=True)
    assert int(host(T_exp).min()) < -126
    assert_rel(host(out), S_ref, TOL_F32, what=f"{fam} end state (strong decay)")
    assert_rel(gdn_T64(T, T_exp), T_ref, TOL_F32, what=f"{fam} chain transition (strong decay)")


@pytest.mark.parametrize("fam,d", [("gdn", 64), ("kda", 32), ("mamba2", 32), ("gla", 32), ("gdn", 128)])
def test_tree_of_chains(B, fam, d):
    """Level 1: chains (p0 p1), (p2 p3), (p4 p5) with T_out, from zero; level 2:
    one chain over the three resulting pairs.  It equals the flat chain
    p0 .. p5 (the chain of pairs is itself a pair)."""
    L, H, P = 1, 2, 6
    Tt, Te, S32, T64 = pair_table(fam, 11, P, L, H, d, d, 48, lo=0.98)
    cu1, idx1 = np.array([0, 2, 4, 6], np.int32), np.arange(6, dtype=np.int32)
    S1, T1, E1 = B.compose(fam, dev(S32), cu1, idx1, T_tab=dev(Tt), T_exp_tab=None if Te is None else dev(Te),
                           want_T=True)
    S2, T2, E2 = B.compose(fam, S1, [0, 3], [0, 1, 2], T_tab=T1, T_exp_tab=E1, want_T=True)
    B.check_device()
    S_ref, T_ref = orc.compose(fam, T64, S32.astype(np.float64), [0, 6], np.arange(6), want_T=True)
    assert_rel(host(S2), S_ref, TOL_F32, what=f"{fam} tree end state")
    check_T(fam, T_of(fam, T2, E2), T_ref, f"{fam} tree transition")
