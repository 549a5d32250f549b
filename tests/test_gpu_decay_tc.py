"""GPU parity of the decay families' tensor-core build (RetNet, Mamba2, GLA,
vanilla; d=128, bf16 keys and values) against the fp64 oracle, through the C
ABI.  The oracle reads the same bf16 values exactly, and the kernel carries
the weighted keys as bf16 pairs (about 16 significant bits), so the fp32 bar
applies.  Ragged bodies up to 2048 tokens (32 chunks, taken from the end
backwards), empty bodies, seam windows left out of the pair, and strong
decays whose early tokens weigh nothing."""
import numpy as np
import pytest

from linear_attn_state_hypic_gb300 import synth
from oracle import oracle as orc
from tests.helpers import TOL_F32, assert_rel, dev, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from linear_attn_state_hypic_gb300 import binding
    return binding


def inputs(fam, seed, lengths, n_layers=2, H=3, d=128, decay=(0.9, 1.0)):
    rng = np.random.default_rng(seed)
    cu = synth.cu_from_lengths(lengths)
    n = int(cu[-1])
    k = rng.standard_normal((n_layers, n, H, d)).astype(np.float32)
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    use = {"k": synth.round_bf16(k), "v": synth.round_bf16(rng.standard_normal((n_layers, n, H, d)).astype(np.float32)),
           "cu_seqlens": cu}
    lo, hi = decay
    if fam == "retnet":
        use["gamma"] = rng.uniform(lo, hi, (n_layers, H)).astype(np.float32)
    elif fam == "mamba2":
        use["alpha"] = rng.uniform(lo, hi, (n_layers, n, H)).astype(np.float32)
    elif fam == "gla":
        use["g"] = rng.uniform(lo, hi, (n_layers, n, H, d)).astype(np.float32)
    return use


def check(B, fam, use, skip=None):
    kw = {key: dev(use[key]) for key in ("gamma", "alpha", "g") if key in use}
    T, _, S = B.segment_build(fam, dev(use["k"], "bf16"), dev(use["v"], "bf16"), use["cu_seqlens"], seam_skip=skip,
                              **kw)
    B.check_device()
    To, So = orc.build_pairs(fam, use["k"], use["v"], use["cu_seqlens"], skip=skip,
                             **{key: use[key] for key in ("gamma", "alpha", "g") if key in use})
    assert_rel(host(S), So, TOL_F32, what=f"{fam} S")
    if To is not None:
        # T is stored in fp32: a decay product below ~1e-38 (0.9^2048 is 1e-94) cannot be represented.
        # Compared entry by entry where it can; where it cannot, it must be negligible.
        Tg = host(T)
        small = np.abs(To) < 1e-30
        assert np.all(np.abs(Tg[small]) < 1e-29), f"{fam} T: an unrepresentable product came out large"
        if np.any(~small):
            rel = np.abs(Tg[~small] - To[~small]) / np.abs(To[~small])
            assert rel.max() <= TOL_F32, f"{fam} T: max relative error {rel.max():.3e}"
    return S


@pytest.mark.parametrize("fam", ["retnet", "mamba2", "gla", "vanilla"])
def test_decay_tc_ragged(B, fam):
    lengths = [1, 0, 63, 64, 65, 700, 2048, 129]
    use = inputs(fam, 11, lengths)
    skip = np.array([0, 0, 8, 0, 8, 8, 3, 64], np.int32)   # the last body is 65 tokens; one more is empty
    check(B, fam, use)
    check(B, fam, use, skip=skip)


@pytest.mark.parametrize("fam", ["retnet", "mamba2", "gla"])
def test_decay_tc_strong_decay(B, fam):
    """Decays down to 0.5 per token: the weights of early tokens underflow to
    zero on both sides long before a 1,500-token body ends."""
    use = inputs(fam, 12, [1500, 300, 5], decay=(0.5, 0.95))
    check(B, fam, use)


def test_decay_tc_many_segments_one_call(B):
    """64 segments x 4 heads x 3 layers in one call: items spread over every
    SM and through the item ring, in longest-body-first order."""
    rng = np.random.default_rng(13)
    lengths = rng.integers(0, 600, 64)
    use = inputs("gla", 13, lengths, n_layers=3, H=4)
    check(B, "gla", use)
