"""GPU parity of hypic_rope_rerotate (the state re-rotation of cached pairs
for RoPE variants) against the fp64 oracle, and the property it exists for: a
pair re-rotated by delta equals the pair built from the keys rotated by
R(delta), so a segment cached at one position can be reused at another."""
import numpy as np
import pytest

from linear_attn_state_hypic_gb300 import synth
from oracle import oracle as orc
from tests.helpers import TOL_F32, assert_rel, dev, gdn_T64, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from linear_attn_state_hypic_gb300 import binding
    return binding


def gates(fam, rng, L, n, H):
    if fam == "gdn":
        return {"alpha": rng.uniform(0.97, 1.0, (L, n, H)).astype(np.float32),
                "beta": rng.uniform(0.0, 0.5, (L, n, H)).astype(np.float32)}
    if fam == "retnet":
        return {"gamma": rng.uniform(0.97, 1.0, (L, H)).astype(np.float32)}
    if fam == "mamba2":
        return {"alpha": rng.uniform(0.97, 1.0, (L, n, H)).astype(np.float32)}
    return {}


def rope_matrix(d, rdim, delta, base=10000.0):
    h = rdim // 2
    ang = delta * base ** (-2.0 * np.arange(h) / rdim)
    R = np.eye(d)
    for i in range(h):
        R[i, i], R[i, i + h], R[i + h, i], R[i + h, i + h] = np.cos(ang[i]), -np.sin(ang[i]), np.sin(ang[i]), np.cos(ang[i])
    return R


@pytest.mark.parametrize("fam,d,rdim", [("gdn", 128, 128), ("gdn", 64, 32), ("retnet", 32, 32),
                                        ("mamba2", 128, 64), ("vanilla", 16, 16)])
def test_rerotation_matches_oracle(B, fam, d, rdim):
    rng = np.random.default_rng(d + rdim)
    L, H = 2, 3
    lengths = [50, 0, 90, 17]
    cu = synth.cu_from_lengths(lengths)
    n = int(cu[-1])
    k = synth._unit_rows(rng, (L, n, H, d))
    v = rng.standard_normal((L, n, H, d)).astype(np.float32)
    gw = gates(fam, rng, L, n, H)
    T, T_exp, S = B.segment_build(fam, dev(k), dev(v), cu, **{key: dev(val) for key, val in gw.items()})
    deltas = [1_000_003, -4096, 0, 77]
    T0 = gdn_T64(T, T_exp) if fam == "gdn" else None
    S0 = host(S)
    B.rope_rerotate(fam, S, deltas, T=T if fam == "gdn" else None, rotary_dim=rdim)
    B.check_device()
    Tr, Sr = orc.rope(fam, T0, S0, deltas, rotary_dim=rdim)
    assert_rel(host(S), Sr, TOL_F32, what=f"{fam} re-rotated S")
    if fam == "gdn":
        assert_rel(gdn_T64(T, T_exp), Tr, TOL_F32, what="gdn re-rotated T")
    np.testing.assert_array_equal(host(S)[1], 0.0)  # the empty segment stays the identity pair


@pytest.mark.parametrize("fam", ["gdn", "retnet"])
def test_rerotated_pair_equals_build_from_rotated_keys(B, fam):
    """Build a segment's pair, re-rotate it by delta; build the same segment
    from the rotated keys R(delta) k: the two pairs agree (up to the float32
    rounding of the rotated keys), and so do chains composed from them."""
    rng = np.random.default_rng(5)
    L, H, d, rdim = 1, 2, 64, 64
    lengths = [120, 80]
    cu = synth.cu_from_lengths(lengths)
    n = int(cu[-1])
    k = synth._unit_rows(rng, (L, n, H, d))
    v = rng.standard_normal((L, n, H, d)).astype(np.float32)
    gw = gates(fam, rng, L, n, H)
    gdev = {key: dev(val) for key, val in gw.items()}
    delta = 12345
    T, T_exp, S = B.segment_build(fam, dev(k), dev(v), cu, **gdev)
    B.rope_rerotate(fam, S, [delta] * len(lengths), T=T if fam == "gdn" else None, rotary_dim=rdim)
    R = rope_matrix(d, rdim, delta)
    k_rot = np.einsum("ij,lthj->lthi", R, k.astype(np.float64)).astype(np.float32)
    T2, T2_exp, S2 = B.segment_build(fam, dev(k_rot), dev(v), cu, **gdev)
    B.check_device()
    assert_rel(host(S), host(S2), 1e-5, what=f"{fam} re-rotated S vs build from rotated keys")
    if fam == "gdn":
        assert_rel(gdn_T64(T, T_exp), gdn_T64(T2, T2_exp), 1e-5, what="gdn re-rotated T vs rotated-key build")
    a = B.compose(fam, S, [0, 2], [0, 1], T_tab=T, T_exp_tab=T_exp)
    b = B.compose(fam, S2, [0, 2], [0, 1], T_tab=T2, T_exp_tab=T2_exp)
    assert_rel(host(a), host(b), 1e-5, what=f"{fam} chain of re-rotated pairs")
