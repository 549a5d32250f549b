"""GPU parity of hypic_segment_build against the fp64 oracle, element by
element per object (relative Frobenius), through the C ABI."""
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


def gpu_build(B, fam, inp, dtype, skip=None):
    k, v = dev(inp["k"], dtype), dev(inp["v"], dtype)
    kw = {}
    for key in ("alpha", "beta", "gamma", "g"):
        if inp.get(key) is not None:
            kw[key] = dev(inp[key])
    T, T_exp, S = B.segment_build(fam, k, v, inp["cu_seqlens"], seam_skip=skip, **kw)
    B.check_device()
    return T, T_exp, S


def oracle_build(fam, inp, skip=None):
    kw = {key: inp[key] for key in ("alpha", "beta", "gamma", "g") if inp.get(key) is not None}
    return orc.build_pairs(fam, inp["k"], inp["v"], inp["cu_seqlens"], skip=skip, **kw)


def check_build(B, fam, inp, dtype, tol, skip=None):
    T, T_exp, S = gpu_build(B, fam, inp, dtype, skip)
    To, So = oracle_build(fam, inp, skip)
    assert_rel(host(S), So, tol, what=f"{fam} S")
    if fam == "gdn":
        assert_rel(gdn_T64(T, T_exp), To, tol, what="gdn T")
    elif fam == "gla":
        assert_rel(host(T), To, tol, axes=(-1,), what="gla T")
    elif fam == "retnet":
        assert_rel(host(T)[..., None], To[..., None], tol, axes=(-1,), what="retnet T")
    return T, T_exp, S


def test_gdn_tiny_build(B):
    """Two 64-token segments, d=16, fp32."""
    check_build(B, "gdn", synth.gdn_tiny(0), "f32", TOL_F32)


@pytest.mark.parametrize("d", [16, 32, 64, 128])
def test_gdn_fp32_dims_ragged(B, d):
    lengths = [1, 63, 64, 65, 0, 130, 257]
    inp = synth.gdn_ragged(seed=d, H=3, d=d, lengths=lengths, dtype="f32")
    check_build(B, "gdn", inp, "f32", TOL_F32)


@pytest.mark.parametrize("variant", ["faithful", "highret", "middecay", "fastdecay"])
def test_gdn_bf16_d128_ragged(B, variant):
    lengths = [700, 1, 64, 129, 0, 2048, 513]
    inp = synth.gdn_ragged(seed=3, H=4, d=128, lengths=lengths, variant=variant)
    check_build(B, "gdn", inp, "bf16", TOL_BF16)


def test_gdn_multi_layer_and_seam_skip(B):
    lengths = [300, 129, 8, 77]
    inp = synth.gdn_ragged(seed=4, H=2, d=128, lengths=lengths, n_layers=3, variant="highret")
    skip = np.array([0, 8, 8, 3], np.int32)   # one body is empty (8 of 8 skipped)
    T, T_exp, S = check_build(B, "gdn", inp, "bf16", TOL_BF16, skip=skip)
    # the empty body is the identity pair
    np.testing.assert_array_equal(gdn_T64(T, T_exp)[2], np.broadcast_to(np.eye(128), (3, 2, 128, 128)))
    assert np.all(host(S)[2] == 0)


def test_gdn_tc_long_segments(B):
    """Tensor-core path over 4096- and 3000-token bodies (64 and 47 chunks):
    many renormalisations of the stored state, T_C far below float32 range
    (kept through the stored exponent)."""
    inp = synth.gdn_ragged(seed=6, H=2, d=128, lengths=[4096, 3000])
    T, T_exp, S = check_build(B, "gdn", inp, "bf16", TOL_BF16)
    assert int(T_exp.cpu().numpy().min()) < -300


def test_gdn_long_segment_T_exponent(B):
    """T_C of a 4096-token segment with alpha ~ U(0.85, 1) is ~1e-140: far
    below float32, so it only survives through the stored exponent."""
    inp = synth.gdn_ragged(seed=5, H=1, d=64, lengths=[4096], dtype="f32")
    T, T_exp, S = check_build(B, "gdn", inp, "f32", TOL_F32)
    assert int(T_exp.cpu().numpy().min()) < -300


@pytest.mark.parametrize("fam", ["retnet", "gla", "vanilla"])
def test_decay_families_build(B, fam):
    inp = synth.decay_small(0)
    use = {"k": inp["k"], "v": inp["v"], "cu_seqlens": inp["cu_seqlens"]}
    if fam == "retnet":
        use["gamma"] = inp["gamma"]
    if fam == "gla":
        use["g"] = inp["g"]
    check_build(B, fam, use, "f32", TOL_F32)


@pytest.mark.parametrize("fam,d", [("retnet", 16), ("gla", 32), ("vanilla", 128), ("gla", 128)])
def test_decay_families_dims_ragged(B, fam, d):
    rng = np.random.default_rng(d)
    lengths = [1, 0, 65, 200]
    cu = synth.cu_from_lengths(lengths)
    n = int(cu[-1])
    use = {"k": synth.round_bf16(rng.standard_normal((2, n, 2, d)).astype(np.float32) / np.sqrt(d)),
           "v": synth.round_bf16(rng.standard_normal((2, n, 2, d)).astype(np.float32)), "cu_seqlens": cu}
    if fam == "retnet":
        use["gamma"] = rng.uniform(0.9, 1.0, (2, 2)).astype(np.float32)
    if fam == "gla":
        use["g"] = rng.uniform(0.9, 1.0, (2, n, 2, d)).astype(np.float32)
    check_build(B, fam, use, "bf16", TOL_F32)


def test_gdn_full_size_ragged_sampled(B):
    """The full ragged batch (32 segments of 512-2048 tokens, 32 heads, d=128,
    bf16) in one call; the oracle checks sampled (segment, head) objects."""
    inp = synth.gdn_ragged(seed=0)
    T, T_exp, S = gpu_build(B, "gdn", inp, "bf16")
    Tg, Sg = gdn_T64(T, T_exp), host(S)
    cu = inp["cu_seqlens"]
    lens = np.diff(cu)
    samples = [(int(np.argmax(lens)), 0), (int(np.argmin(lens)), 31), (5, 17), (20, 3)]
    for seg, h in samples:
        sl = slice(int(cu[seg]), int(cu[seg + 1]))
        one = {key: np.ascontiguousarray(inp[key][:, sl, h:h + 1]) for key in ("k", "v", "alpha", "beta")}
        one["cu_seqlens"] = [0, int(lens[seg])]
        To, So = oracle_build("gdn", one)
        assert_rel(Sg[seg, :, h:h + 1], So[0], TOL_BF16, what=f"S seg {seg} head {h}")
        assert_rel(Tg[seg, :, h:h + 1], To[0], TOL_BF16, what=f"T seg {seg} head {h}")
