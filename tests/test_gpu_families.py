"""GPU parity of the KDA and Mamba2 families against the fp64 oracle, through
the C ABI: build (ragged, every supported d, fp32 and bf16 inputs, seam skips,
strong decay), compose (the tensor-core path for KDA at d = 128 and the
CUDA-core paths), seam advance, the reuse chain (step-by-step path) and the
whole reuse path against the full sequential recurrence.

KDA: S_t = (I - b_t k_t k_t^T) Diag(a_t) S_{t-1} + b_t k_t v_t^T with the
per-channel gate a_t in ``g``; Mamba2: S_t = a_t S_{t-1} + k_t v_t^T with the
per-token decay a_t in ``alpha``."""
import numpy as np
import pytest

from linear_attn_state_hypic_gb300 import synth
from oracle import oracle as orc
from tests.helpers import TOL_BF16, TOL_F32, assert_rel, dev, gdn_T64, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from linear_attn_state_hypic_gb300 import binding
    return binding


def tokens(rng, L, n, H, d, dtype):
    k = synth._unit_rows(rng, (L, n, H, d))
    v = rng.standard_normal((L, n, H, d)).astype(np.float32)
    q = synth._unit_rows(rng, (L, n, H, d))
    if dtype == "bf16":
        k, v, q = (synth.round_bf16(x) for x in (k, v, q))
    return q, k, v


def gates(fam, rng, L, n, H, d, lo=0.85):
    if fam == "kda":
        return {"g": rng.uniform(lo, 1.0, (L, n, H, d)).astype(np.float32),
                "beta": rng.uniform(0.0, 1.0, (L, n, H)).astype(np.float32)}
    return {"alpha": rng.uniform(lo, 1.0, (L, n, H)).astype(np.float32)}


def check_pairs(fam, T, T_exp, S, To, So, tol):
    assert_rel(host(S), So, tol, what=f"{fam} S")
    if fam == "kda":
        assert_rel(gdn_T64(T, T_exp), To, tol, what="kda T")
    else:
        assert_rel(host(T)[..., None], To[..., None], tol, axes=(-1,), what="mamba2 T")


@pytest.mark.parametrize("fam", ["kda", "mamba2"])
@pytest.mark.parametrize("d,dtype", [(16, "f32"), (32, "f32"), (64, "f32"), (128, "f32"), (128, "bf16")])
def test_build(B, fam, d, dtype):
    rng = np.random.default_rng(d + (7 if fam == "kda" else 0))
    lengths = [1, 63, 64, 65, 0, 130, 257]
    cu = synth.cu_from_lengths(lengths)
    n, L, H = int(cu[-1]), 2, 3
    _, k, v = tokens(rng, L, n, H, d, dtype)
    gw = gates(fam, rng, L, n, H, d)
    skip = np.array([0, 8, 8, 3, 0, 1, 8], np.int32)
    T, T_exp, S = B.segment_build(fam, dev(k, dtype), dev(v, dtype), cu, seam_skip=skip,
                                  **{key: dev(val) for key, val in gw.items()})
    B.check_device()
    To, So = orc.build_pairs(fam, k, v, cu, skip=skip, **gw)
    check_pairs(fam, T, T_exp, S, To, So, TOL_BF16 if dtype == "bf16" else TOL_F32)
    # the empty segment 4 is the identity pair
    if fam == "kda":
        np.testing.assert_array_equal(gdn_T64(T, T_exp)[4], np.broadcast_to(np.eye(d), (L, H, d, d)))
    else:
        np.testing.assert_array_equal(host(T)[4], 1.0)
    assert np.all(host(S)[4] == 0)


@pytest.mark.parametrize("fam", ["kda", "mamba2"])
def test_build_strong_decay_long_segment(B, fam):
    """Gates in [0.5, 1) over 1,500 tokens: T_C falls far below the float32
    range (KDA keeps it as mantissa and exponent; the scalar Mamba2 T_C is
    allowed to underflow to 0 like the oracle's value rounded to float32)."""
    rng = np.random.default_rng(31)
    d, L, H = 64, 1, 2
    cu = synth.cu_from_lengths([1500, 700])
    n = int(cu[-1])
    _, k, v = tokens(rng, L, n, H, d, "f32")
    gw = gates(fam, rng, L, n, H, d, lo=0.5)
    T, T_exp, S = B.segment_build(fam, dev(k), dev(v), cu, **{key: dev(val) for key, val in gw.items()})
    B.check_device()
    To, So = orc.build_pairs(fam, k, v, cu, **gw)
    assert_rel(host(S), So, TOL_F32, what=f"{fam} S (strong decay)")
    if fam == "kda":
        assert int(host(T_exp).min()) < -126  # would underflow float32 without the exponent
        assert_rel(gdn_T64(T, T_exp), To, TOL_F32, what="kda T (strong decay)")
    else:
        np.testing.assert_allclose(host(T), To.astype(np.float32).astype(np.float64), rtol=1e-4, atol=0)


def pair_table(fam, seed, n_pairs, L, H, d, seg_len):
    """Pairs built by the oracle, stored as the GPU stores them (KDA: float32
    mantissa and int32 exponent)."""
    rng = np.random.default_rng(seed)
    cu = synth.cu_from_lengths([seg_len] * n_pairs)
    n = int(cu[-1])
    _, k, v = tokens(rng, L, n, H, d, "f32")
    gw = gates(fam, rng, L, n, H, d, lo=0.995)  # slow decay: ||T|| ~ 1, so T S matters
    if fam == "kda":
        gw["beta"] *= 0.2
    T, S = orc.build_pairs(fam, k, v, cu, **gw)
    S32 = S.astype(np.float32)
    if fam == "kda":
        Tm, Te = orc.f64_to_scaled(T)
        return Tm, Te, S32, orc.scaled_to_f64(Tm, Te)
    T32 = T.astype(np.float32)
    return T32, None, S32, T32.astype(np.float64)


@pytest.mark.parametrize("fam,d", [("kda", 128), ("kda", 32), ("mamba2", 64), ("mamba2", 128)])
def test_compose(B, fam, d):
    L, H, P = 2, 2, 5
    Tm, Te, S32, T64 = pair_table(fam, 40 + d, P, L, H, d, 48)
    chains = [[0, 1, 2, 3, 4], [4, 2], [], [1, 1, 1]]
    cu = np.array([0] + list(np.cumsum([len(c) for c in chains])), np.int32)
    idx = np.array([i for c in chains for i in c], np.int32)
    rng = np.random.default_rng(d)
    S0 = (rng.standard_normal((len(chains), L, H, d, d)) / np.sqrt(d)).astype(np.float32)
    out = B.compose(fam, dev(S32), cu, idx, T_tab=dev(Tm), T_exp_tab=None if Te is None else dev(Te), S0=dev(S0))
    B.check_device()
    ref = orc.compose(fam, T64, S32.astype(np.float64), cu, idx, S0=S0)
    assert_rel(host(out), ref, TOL_F32, what=f"{fam} compose")


@pytest.mark.parametrize("fam,dtype,d", [("kda", "f32", 16), ("kda", "bf16", 128), ("mamba2", "f32", 64),
                                         ("mamba2", "bf16", 128)])
@pytest.mark.parametrize("inplace", [False, True])
def test_seam_advance(B, fam, dtype, d, inplace):
    rng = np.random.default_rng(d + 5)
    lens = [8, 0, 1, 40, 8]
    cu = synth.cu_from_lengths(lens)
    n, L, H = int(cu[-1]), 2, 3
    q, k, v = tokens(rng, L, n, H, d, dtype)
    gw = gates(fam, rng, L, n, H, d)
    st = (rng.standard_normal((len(lens), L, H, d, d)) / np.sqrt(d)).astype(np.float32)
    st_in = dev(st)
    s_out, o = B.seam_advance(fam, dev(q, dtype), dev(k, dtype), dev(v, dtype), cu, state_in=st_in,
                              state_out=st_in if inplace else None, **{key: dev(val) for key, val in gw.items()})
    B.check_device()
    ref_s, ref_o = orc.seam(fam, q, k, v, cu, state_in=st, **gw)
    tol = TOL_BF16 if dtype == "bf16" else TOL_F32
    assert_rel(host(s_out), ref_s, tol, what=f"{fam} seam state")
    assert_rel(host(o), ref_o, tol, axes=(-1,), what=f"{fam} seam outputs")


@pytest.mark.parametrize("fam,d,dtype", [("kda", 128, "bf16"), ("kda", 64, "f32"), ("mamba2", 128, "bf16")])
def test_reuse_path_equals_full_sequential(B, fam, d, dtype):
    """Build every body of a ragged request (an 8-token seam at each internal
    segment start), then one hypic_reuse_chain call over all segments: the end
    state and every seam output equal the full sequential recurrence."""
    rng = np.random.default_rng(71 + d)
    lengths = rng.integers(60, 260, size=5)
    L, H = 2, 2
    cu = synth.cu_from_lengths(lengths)
    n = int(cu[-1])
    q, k, v = tokens(rng, L, n, H, d, dtype)
    gw = gates(fam, rng, L, n, H, d, lo=0.97)
    skip = np.full(len(lengths), 8, np.int32)
    skip[0] = 0
    gdev = {key: dev(val) for key, val in gw.items()}
    T, T_exp, S = B.segment_build(fam, dev(k, dtype), dev(v, dtype), cu, seam_skip=skip, **gdev)
    n_seg = len(lengths)
    seam_tok = np.concatenate([np.arange(cu[i], cu[i] + skip[i]) for i in range(n_seg)])
    cu_step = np.concatenate([[0], np.cumsum(skip)]).astype(np.int32)
    pick = lambda x: np.ascontiguousarray(x[:, seam_tok])
    sg = {key: dev(pick(val)) for key, val in gw.items()}
    out, o = B.reuse_chain(fam, S, np.array([0, n_seg], np.int32), np.arange(n_seg, dtype=np.int32), cu_step,
                           dev(pick(q), dtype), dev(pick(k), dtype), dev(pick(v), dtype), T_tab=T, T_exp_tab=T_exp,
                           **sg)
    B.check_device()
    full_s, full_o = orc.seam(fam, q, k, v, [0, n], **gw)
    tol = TOL_BF16 if dtype == "bf16" else TOL_F32
    assert_rel(host(out), full_s, tol, what=f"{fam} reuse-path end state")
    assert_rel(host(o), full_o[:, seam_tok], tol, axes=(-1,), what=f"{fam} seam outputs")
