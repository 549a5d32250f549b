"""GPU parity of the KDA build on the tensor cores (d = 128, bf16 keys and
values: every 64-token chunk's own pair, then the chunk pairs chained by the
tensor-core compose) against the fp64 oracle and against the CUDA-core build
(hypic_segment_build_noalloc runs KDA on CUDA cores), through the C ABI.

KDA: S_t = (I - b_t k_t k_t^T) Diag(a_t) S_{t-1} + b_t k_t v_t^T, the
per-channel gate a_t in ``g`` (aibase article on HYPIC, linear-layer
paragraph: the cached pair (T_C, S(C|0)) of a segment)."""
import numpy as np
import pytest

from linear_attn_state_hypic_gb300 import synth
from oracle import oracle as orc
from tests.helpers import TOL_BF16, assert_rel, dev, gdn_T64, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from linear_attn_state_hypic_gb300 import binding
    return binding


def kda_inputs(rng, lengths, L, H, glo=0.85, ghi=1.0, d=128):
    cu = synth.cu_from_lengths(lengths)
    n = int(cu[-1])
    k = synth.round_bf16(synth._unit_rows(rng, (L, n, H, d)))
    v = synth.round_bf16(rng.standard_normal((L, n, H, d)).astype(np.float32))
    g = rng.uniform(glo, ghi, (L, n, H, d)).astype(np.float32)
    beta = rng.uniform(0.0, 1.0, (L, n, H)).astype(np.float32)
    return cu, k, v, g, beta


def build(B, k, v, g, beta, cu, skip=None, noalloc=False):
    if not noalloc:
        out = B.segment_build("kda", dev(k, "bf16"), dev(v, "bf16"), cu, g=dev(g), beta=dev(beta), seam_skip=skip)
        B.check_device()
        return out
    import torch
    kd, vd, gd, bd = dev(k, "bf16"), dev(v, "bf16"), dev(g), dev(beta)
    n_seg = len(cu) - 1
    out = B.alloc_build_outputs("kda", n_seg, k.shape[0], k.shape[2], 128, 128, kd.device)
    a, keep = B.build_args("kda", kd, vd, cu, g=gd, beta=bd, seam_skip=skip, T_out=out[0], T_exp_out=out[1],
                           S_out=out[2])
    B._check(B.hypic_segment_build_noalloc(a, B._stream(None)))
    torch.cuda.synchronize()
    B.check_device()
    del keep
    return out


def test_kda_tc_ragged_with_seam_skips(B):
    """Ragged bodies around the chunk length (1, 63, 64, 65, 128, 129 tokens),
    empty ones, seam skips, two layers of three heads."""
    rng = np.random.default_rng(401)
    lengths = [1, 63, 64, 65, 0, 136, 129, 300, 9]
    skip = np.array([0, 0, 0, 1, 0, 8, 0, 5, 9], np.int32)
    cu, k, v, g, beta = kda_inputs(rng, lengths, 2, 3)
    T, T_exp, S = build(B, k, v, g, beta, cu, skip)
    To, So = orc.build_pairs("kda", k, v, cu, skip=skip, g=g, beta=beta)
    assert_rel(host(S), So, TOL_BF16, what="kda S")
    assert_rel(gdn_T64(T, T_exp), To, TOL_BF16, what="kda T")
    for s in (4, 8):  # empty bodies: the identity pair
        np.testing.assert_array_equal(gdn_T64(T, T_exp)[s], np.broadcast_to(np.eye(128), (2, 3, 128, 128)))
        assert np.all(host(S)[s] == 0)


def test_kda_tc_extreme_gates(B):
    """Gates from U(0, 1) with some exactly 0 and exactly 1: within a chunk
    the gate products fall far below the fp32 range (a ratio of prefix
    products would overflow), and T_C needs its exponent."""
    rng = np.random.default_rng(402)
    cu, k, v, g, beta = kda_inputs(rng, [200, 333, 64], 1, 2, glo=0.0, ghi=1.0)
    g[0, 10:20, :, :7] = 0.0
    g[0, 250:300, :, 100:] = 1.0
    T, T_exp, S = build(B, k, v, g, beta, cu)
    To, So = orc.build_pairs("kda", k, v, cu, g=g, beta=beta)
    assert_rel(host(S), So, TOL_BF16, what="kda S (extreme gates)")
    assert_rel(gdn_T64(T, T_exp), To, TOL_BF16, what="kda T (extreme gates)")


def test_kda_tc_strong_decay_long_segment(B):
    """Gates in [0.5, 1) over 1,500 tokens: T_C leaves the fp32 range and is
    kept as mantissa and exponent by the compose that chains the chunks."""
    rng = np.random.default_rng(403)
    cu, k, v, g, beta = kda_inputs(rng, [1500, 700], 1, 2, glo=0.5)
    T, T_exp, S = build(B, k, v, g, beta, cu)
    To, So = orc.build_pairs("kda", k, v, cu, g=g, beta=beta)
    assert int(host(T_exp).min()) < -126
    assert_rel(host(S), So, TOL_BF16, what="kda S (strong decay)")
    assert_rel(gdn_T64(T, T_exp), To, TOL_BF16, what="kda T (strong decay)")


def test_kda_tc_matches_cuda_core_build_over_batches(B):
    """More than 4 GiB of chunk tables (300 segments x 64 heads), so the
    tensor-core path takes its segments in two batches: every pair agrees with
    the CUDA-core build of the same inputs, and a sample with the oracle."""
    rng = np.random.default_rng(404)
    lengths = rng.integers(100, 190, 300)
    cu, k, v, g, beta = kda_inputs(rng, lengths, 1, 64)
    n_chunks = int(np.sum((lengths + 63) // 64))
    assert n_chunks * 64 * 128 * 1024 > 4 << 30
    T, T_exp, S = build(B, k, v, g, beta, cu)
    Tn, Tn_exp, Sn = build(B, k, v, g, beta, cu, noalloc=True)
    assert_rel(host(S), host(Sn).astype(np.float64), 1e-3, what="S, tensor cores vs CUDA cores")
    assert_rel(gdn_T64(T, T_exp), gdn_T64(Tn, Tn_exp), 1e-3, what="T, tensor cores vs CUDA cores")
    for s in (0, 150, 299):  # one segment of each batch, and the first
        sl = slice(int(cu[s]), int(cu[s + 1]))
        kk, vv, gg, bb = (x[:, sl, :4] for x in (k, v, g, beta))
        To, So = orc.build_pairs("kda", np.ascontiguousarray(kk), np.ascontiguousarray(vv),
                                 np.array([0, sl.stop - sl.start], np.int32), g=np.ascontiguousarray(gg),
                                 beta=np.ascontiguousarray(bb))
        assert_rel(host(S)[s:s + 1, :, :4], So, TOL_BF16, what=f"S of segment {s}")
        assert_rel(gdn_T64(T, T_exp)[s:s + 1, :, :4], To, TOL_BF16, what=f"T of segment {s}")


def test_kda_tc_segment_longer_than_a_batch(B):
    """A segment whose chunk tables alone exceed the 4 GiB the workspace holds
    (36,000 tokens x 64 heads: 563 chunks of 64 x 64 heads x 128 KB), between
    two short ones: the tensor-core path builds it in parts, each chained after
    the pair of the parts before it (composition law).  Gates near 1 keep T_C
    of the long segment inside the fp64 range of the oracle.  Every pair agrees
    with the CUDA-core build; two heads of the long segment with the oracle."""
    rng = np.random.default_rng(405)
    lengths = [300, 36000, 200]
    cu, k, v, g, beta = kda_inputs(rng, lengths, 1, 64, glo=0.999)
    assert ((36000 + 63) // 64) * 64 * 128 * 1024 > 4 << 30
    T, T_exp, S = build(B, k, v, g, beta, cu)
    Tn, Tn_exp, Sn = build(B, k, v, g, beta, cu, noalloc=True)
    assert_rel(host(S), host(Sn), 1e-3, what="S, tensor cores vs CUDA cores")
    assert_rel(gdn_T64(T, T_exp), gdn_T64(Tn, Tn_exp), 1e-3, what="T, tensor cores vs CUDA cores")
    sl = slice(int(cu[1]), int(cu[2]))
    kk, vv, gg, bb = (np.ascontiguousarray(x[:, sl, :2]) for x in (k, v, g, beta))
    To, So = orc.build_pairs("kda", kk, vv, np.array([0, sl.stop - sl.start], np.int32), g=gg, beta=bb)
    assert_rel(host(S)[1:2, :, :2], So, TOL_BF16, what="S of the long segment")
    assert_rel(gdn_T64(T, T_exp)[1:2, :, :2], To, TOL_BF16, what="T of the long segment")


def test_kda_tc_safe_and_guarded_chunks_in_one_call(B):
    """Most chunks have gates in [0.85, 1) and take the tensor-core gram; in a
    few, some channels' gates are ~1e-3, so the chunk's decay leaves the range
    of k / g_t and it forms its gram from running products on CUDA cores.  Both
    kinds of chunk in one launch, against the oracle."""
    rng = np.random.default_rng(406)
    lengths = [640, 300, 129]
    cu, k, v, g, beta = kda_inputs(rng, lengths, 1, 4)
    g[0, 64:128, :, :5] = 1e-3       # chunk 1 of segment 0: g_C of those channels ~1e-192
    g[0, 700:710, 1, 60:64] = 1e-4   # inside segment 1, one head
    T, T_exp, S = build(B, k, v, g, beta, cu)
    To, So = orc.build_pairs("kda", k, v, cu, g=g, beta=beta)
    assert_rel(host(S), So, TOL_BF16, what="kda S (mixed chunks)")
    assert_rel(gdn_T64(T, T_exp), To, TOL_BF16, what="kda T (mixed chunks)")


def test_kda_tc_zero_beta_is_the_gate_product(B):
    """b = 0: every delta step is the identity, so T_C = Diag(prod_t a_t) and
    S = 0 (a closed form, no oracle)."""
    rng = np.random.default_rng(407)
    lengths = [200, 64, 1]
    cu, k, v, g, beta = kda_inputs(rng, lengths, 1, 3, glo=0.9)
    beta[:] = 0.0
    T, T_exp, S = build(B, k, v, g, beta, cu)
    assert np.all(host(S) == 0)
    Tg = gdn_T64(T, T_exp)
    for s in range(len(lengths)):
        prod = np.prod(g[0, int(cu[s]):int(cu[s + 1])].astype(np.float64), axis=0)  # [H][d]
        want = np.stack([np.diag(prod[h]) for h in range(3)])[None]
        np.testing.assert_allclose(Tg[s], want, rtol=1e-5, atol=0)
