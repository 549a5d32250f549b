"""GPU parity of hypic_compose and hypic_seam_advance against the fp64 oracle,
and of the whole reuse path (build bodies, seam advance, compose) against the
full sequential recurrence."""
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


def gdn_pair_table(seed, n_pairs, n_layers, H, d, L, variant="highret"):
    """Pairs built by the oracle from synthetic tokens; T stored as the GPU
    stores it (float32 mantissa, int32 exponent) and S rounded to float32."""
    inp = synth.gdn_ragged(seed=seed, H=H, d=d, lengths=[L] * n_pairs, n_layers=n_layers,
                           variant=variant, dtype="f32")
    T, S = orc.build_pairs("gdn", inp["k"], inp["v"], inp["cu_seqlens"], alpha=inp["alpha"], beta=inp["beta"])
    Tm, Te = orc.f64_to_scaled(T)
    S32 = S.astype(np.float32)
    return Tm, Te, S32, orc.scaled_to_f64(Tm, Te), S32.astype(np.float64)


def test_gdn_compose_chains(B):
    """Chains over oracle-built high-retention pairs (||T|| ~ 1, so errors in
    T S stay visible), zero and random starts, an empty chain, a repeated
    pair."""
    d, L, H, P = 128, 96, 2, 6
    Tm, Te, S32, T64, S64 = gdn_pair_table(1, P, 2, H, d, L)
    chains = [[0, 1, 2, 3, 4, 5], [5, 4, 3], [], [2, 2, 2, 2]]
    cu = np.array([0] + list(np.cumsum([len(c) for c in chains])), np.int32)
    idx = np.array([i for c in chains for i in c], np.int32)
    rng = np.random.default_rng(2)
    S0 = (rng.standard_normal((len(chains), 2, H, d, d)) / np.sqrt(d)).astype(np.float32)
    S0[0] = 0
    out = B.compose("gdn", dev(S32), cu, idx, T_tab=dev(Tm), T_exp_tab=dev(Te), S0=dev(S0))
    B.check_device()
    ref = orc.compose("gdn", T64, S64, cu, idx, S0=S0)
    assert_rel(host(out), ref, TOL_F32, what="gdn compose")


def test_gdn_compose_without_start_or_exponents(B):
    d, H, P = 64, 3, 4
    Tm, Te, S32, T64, S64 = gdn_pair_table(3, P, 1, H, d, 80)
    cu, idx = np.array([0, 4], np.int32), np.array([3, 1, 0, 2], np.int32)
    out = B.compose("gdn", dev(S32), cu, idx, T_tab=dev(Tm))
    ref = orc.compose("gdn", Tm.astype(np.float64), S64, cu, idx)
    assert_rel(host(out), ref, TOL_F32, what="gdn compose, exponent table NULL")


@pytest.mark.parametrize("fam", ["retnet", "gla", "vanilla"])
def test_decay_compose_matches_sequential_and_reports_naive_error(B, fam):
    """Decay workload: build 8 x 256-token segments, compose them in order
    and compare with the 2048-token sequential run; the naive addition
    (the same S tables composed as plain linear attention) is reported per
    head and must match the oracle's naive error."""
    inp = synth.decay_small(0)
    k, v = dev(inp["k"]), dev(inp["v"])
    kw, okw = {}, {}
    if fam == "retnet":
        kw["gamma"], okw["gamma"] = dev(inp["gamma"]), inp["gamma"]
    if fam == "gla":
        kw["g"], okw["g"] = dev(inp["g"]), inp["g"]
    T, _, S = B.segment_build(fam, k, v, inp["cu_seqlens"], **kw)
    n_seg = len(inp["cu_seqlens"]) - 1
    cu, idx = np.array([0, n_seg], np.int32), np.arange(n_seg, dtype=np.int32)
    out = B.compose(fam, S, cu, idx, T_tab=T)
    naive = B.compose("vanilla", S, cu, idx)
    B.check_device()
    n = int(inp["cu_seqlens"][-1])
    full, _ = orc.seam(fam, inp["q"], inp["k"], inp["v"], [0, n], **okw)
    assert_rel(host(out), full, TOL_F32, what=f"{fam} composed vs sequential")
    To, So = orc.build_pairs(fam, inp["k"], inp["v"], inp["cu_seqlens"], **okw)
    naive_ref = orc.compose(fam, To, So, cu, idx, naive=True)
    err_gpu = np.linalg.norm(host(naive) - host(out), axis=(-2, -1)) / np.linalg.norm(full, axis=(-2, -1))
    err_ref = np.linalg.norm(naive_ref - full, axis=(-2, -1)) / np.linalg.norm(full, axis=(-2, -1))
    np.testing.assert_allclose(err_gpu, err_ref, rtol=1e-3, atol=1e-6)
    if fam == "vanilla":
        assert np.max(err_ref) < 1e-12
    print(f"\n{fam} naive-addition error per head (/||S_true||):", np.round(err_gpu.ravel(), 4))


@pytest.mark.parametrize("fam,dtype,d", [("gdn", "bf16", 128), ("gdn", "f32", 16), ("retnet", "f32", 64),
                                         ("gla", "bf16", 128), ("vanilla", "f32", 32)])
@pytest.mark.parametrize("inplace", [False, True])
def test_seam_advance(B, fam, dtype, d, inplace):
    rng = np.random.default_rng(d)
    lens = [8, 0, 1, 40, 8]
    cu = synth.cu_from_lengths(lens)
    n, Lyr, H = int(cu[-1]), 2, 3
    rb = synth.round_bf16 if dtype == "bf16" else (lambda x: x)
    unit = lambda s: (lambda x: x / np.linalg.norm(x, axis=-1, keepdims=True))(rng.standard_normal(s)).astype(np.float32)
    q, k = rb(unit((Lyr, n, H, d))), rb(unit((Lyr, n, H, d)))
    v = rb(rng.standard_normal((Lyr, n, H, d)).astype(np.float32))
    okw = {}
    if fam == "gdn":
        okw["alpha"], okw["beta"] = synth.gdn_gates(rng, (Lyr, n, H), "faithful")
    if fam == "retnet":
        okw["gamma"] = rng.uniform(0.9, 1, (Lyr, H)).astype(np.float32)
    if fam == "gla":
        okw["g"] = rng.uniform(0.8, 1, (Lyr, n, H, d)).astype(np.float32)
    st = (rng.standard_normal((len(lens), Lyr, H, d, d)) / np.sqrt(d)).astype(np.float32)
    st_in = dev(st)
    kw = {key: dev(val) for key, val in okw.items()}
    out_state = st_in if inplace else None
    s_out, o = B.seam_advance(fam, dev(q, dtype), dev(k, dtype), dev(v, dtype), cu, state_in=st_in,
                              state_out=out_state, **kw)
    B.check_device()
    ref_s, ref_o = orc.seam(fam, q, k, v, cu, state_in=st, **okw)
    tol = TOL_BF16 if dtype == "bf16" else TOL_F32
    assert_rel(host(s_out), ref_s, tol, what=f"{fam} seam state")
    assert_rel(host(o), ref_o, tol, axes=(-1,), what=f"{fam} seam outputs")


@pytest.mark.parametrize("fam,dtype,d", [("kda", "bf16", 128), ("mamba2", "f32", 64), ("gdn", "f32", 32)])
def test_seam_advance_from_zero_long_windows(B, fam, dtype, d):
    """No start state (zeros, nothing copied in), windows longer than the tokens
    a seam-head takes ahead (8), and many seam-heads per CTA.  The outputs are
    checked per (layer, head) over all tokens: from a zero state some outputs are
    small differences of decayed terms, and a per-row relative error would
    divide the fp32 rounding of the state by their tiny norms."""
    rng = np.random.default_rng(100 + d)
    lens = [17, 9, 0, 33, 8, 1, 24, 16] * 6
    cu = synth.cu_from_lengths(lens)
    n, Lyr, H = int(cu[-1]), 2, 5
    rb = synth.round_bf16 if dtype == "bf16" else (lambda x: x)
    unit = lambda s: (lambda x: x / np.linalg.norm(x, axis=-1, keepdims=True))(rng.standard_normal(s)).astype(np.float32)
    q, k = rb(unit((Lyr, n, H, d))), rb(unit((Lyr, n, H, d)))
    v = rb(rng.standard_normal((Lyr, n, H, d)).astype(np.float32))
    okw = {}
    if fam == "gdn":
        okw["alpha"], okw["beta"] = synth.gdn_gates(rng, (Lyr, n, H), "middecay")
    if fam == "kda":
        okw["g"] = rng.uniform(0.85, 1, (Lyr, n, H, d)).astype(np.float32)
        okw["beta"] = rng.uniform(0, 1, (Lyr, n, H)).astype(np.float32)
    if fam == "mamba2":
        okw["alpha"] = rng.uniform(0.85, 1, (Lyr, n, H)).astype(np.float32)
    kw = {key: dev(val) for key, val in okw.items()}
    s_out, o = B.seam_advance(fam, dev(q, dtype), dev(k, dtype), dev(v, dtype), cu, **kw)
    B.check_device()
    ref_s, ref_o = orc.seam(fam, q, k, v, cu, state_in=None, **okw)
    tol = TOL_BF16 if dtype == "bf16" else TOL_F32
    assert_rel(host(s_out), ref_s, tol, what=f"{fam} seam state from zero")
    assert_rel(host(o), ref_o, tol, axes=(1, 3), what=f"{fam} seam outputs from zero")


def reuse_path(B, inp_dev, cu, skip, seam_tok, n_layers, H, d, q_seam, alpha=None, beta=None):
    """Build every body, then advance a running state through the chain:
    state = pair(seg 0); for each internal segment: seam advance over its
    first tokens (outputs for the full-attention layers), then compose the
    body pair.  Returns (final state, seam outputs)."""
    torch = __import__("torch")
    T, T_exp, S = B.segment_build("gdn", inp_dev["k"], inp_dev["v"], cu, seam_skip=skip,
                                  alpha=inp_dev["alpha"], beta=inp_dev["beta"])
    n_seg = len(cu) - 1
    state = B.compose("gdn", S, [0, 1], [0], T_tab=T, T_exp_tab=T_exp)
    ks, vs = inp_dev["k"][:, seam_tok], inp_dev["v"][:, seam_tok]
    a_s, b_s = inp_dev["alpha"][:, seam_tok], inp_dev["beta"][:, seam_tok]
    outs = []
    pos = 0
    nxt = torch.empty_like(state)
    for i in range(1, n_seg):
        w = int(skip[i])
        sl = slice(pos, pos + w)
        _, o = B.seam_advance("gdn", q_seam[:, sl].contiguous(), ks[:, sl].contiguous(), vs[:, sl].contiguous(),
                              [0, w], alpha=a_s[:, sl].contiguous(), beta=b_s[:, sl].contiguous(), state_in=state,
                              state_out=state)
        outs.append(o)
        B.compose("gdn", S, [0, 1], [i], T_tab=T, T_exp_tab=T_exp, S0=state, out=nxt)
        state, nxt = nxt, state
        pos += w
    B.check_device()
    return state, torch.cat(outs, dim=1)


def test_reuse_path_equals_full_sequential(B):
    """Small long-request replica: ragged segments with an 8-token seam at
    every internal segment start; the final state and every seam output
    equal the full sequential recurrence over the whole request."""
    torch = __import__("torch")
    rng = np.random.default_rng(7)
    lengths = rng.integers(60, 300, size=6)
    n_layers, H, d = 2, 2, 128
    inp = synth.gdn_ragged(seed=7, H=H, d=d, lengths=lengths, n_layers=n_layers, with_q=True, variant="highret")
    cu = inp["cu_seqlens"]
    skip = np.full(len(lengths), 8, np.int32)
    skip[0] = 0
    seam_tok = np.concatenate([np.arange(cu[i], cu[i] + 8) for i in range(1, len(lengths))])
    inp_dev = {"k": dev(inp["k"], "bf16"), "v": dev(inp["v"], "bf16"), "alpha": dev(inp["alpha"]),
               "beta": dev(inp["beta"])}
    q_seam = dev(np.ascontiguousarray(inp["q"][:, seam_tok]), "bf16")
    state, o = reuse_path(B, inp_dev, cu, skip, torch.from_numpy(seam_tok).cuda(), n_layers, H, d, q_seam)
    n = int(cu[-1])
    full_s, full_o = orc.seam("gdn", inp["q"], inp["k"], inp["v"], [0, n], alpha=inp["alpha"], beta=inp["beta"])
    assert_rel(host(state), full_s, TOL_BF16, what="reuse-path end state")
    assert_rel(host(o), full_o[:, seam_tok], TOL_BF16, axes=(-1,), what="seam outputs")


def test_gdn_compose_faithful_pairs_long_chains(B):
    """Pairs of 512-token segments with strong decay (T_C ~ 1e-18, stored as
    mantissa x 2^exp with exp near -60) composed along 40-step chains with
    repeats: the stored exponent must be applied exactly, and the slice ring
    of the tensor-core path wraps many times."""
    d, H, P = 128, 2, 6
    Tm, Te, S32, T64, S64 = gdn_pair_table(5, P, 1, H, d, 512, variant="faithful")
    assert Te.min() < -40
    rng = np.random.default_rng(6)
    chains = [list(rng.integers(0, P, 40)), list(rng.integers(0, P, 17)), [3]]
    cu = np.array([0] + list(np.cumsum([len(c) for c in chains])), np.int32)
    idx = np.array([i for c in chains for i in c], np.int32)
    S0 = (rng.standard_normal((len(chains), 1, H, d, d)) / np.sqrt(d)).astype(np.float32)
    out = B.compose("gdn", dev(S32), cu, idx, T_tab=dev(Tm), T_exp_tab=dev(Te), S0=dev(S0))
    B.check_device()
    ref = orc.compose("gdn", T64, S64, cu, idx, S0=S0)
    assert_rel(host(out), ref, TOL_F32, what="gdn compose, faithful pairs")
