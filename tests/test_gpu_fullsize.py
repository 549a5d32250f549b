"""Parity at full size, in the launch configuration the benchmark times.

* The long cold request (30 GDN layers x 32 heads, d=128, bf16, 100,000
  tokens, 8-token seams): one build call over every body, then the reuse
  chain as one hypic_reuse_chain call (the fused kernel) and, as a cross
  check, as separate seam-advance and one-step compose calls.  Sampled (layer, head)
  objects are checked against the fp64 sequential recurrence over the whole
  request (end state and every seam output) and against the oracle's pairs
  for sampled segments.
* The compose table (30 x 32 heads, 128 pairs, 16 chains of 64 steps):
  sampled (chain, layer, head) end states against the oracle's chain.

Inputs are drawn on the device by the seeded generator; only the sampled
slices are copied to the host for the oracle."""
import numpy as np
import pytest

from linear_attn_state_hypic_gb300 import synth
from oracle import oracle as orc
from tests.helpers import TOL_BF16, TOL_F32, assert_rel, gdn_T64, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from linear_attn_state_hypic_gb300 import binding
    return binding


def test_long_request_full_size_sampled(B):
    import torch
    r = synth.long_request_device(seed=0)
    cu, skip, seam_tok = r["cu_seqlens"], r["seam_skip"], r["seam_tok"]
    n_seg, L, N, H, d = len(cu) - 1, 30, int(cu[-1]), 32, 128
    T, T_exp, S = B.segment_build("gdn", r["k"], r["v"], cu, alpha=r["alpha"], beta=r["beta"], seam_skip=skip)
    st = torch.as_tensor(seam_tok, device="cuda")
    ks, vs, a_s, b_s = (x[:, st].contiguous() for x in (r["k"], r["v"], r["alpha"], r["beta"]))
    # the product path: one reuse chain (compose segment 0, then seam i + compose i)
    cu_step = np.concatenate([[0, 0], np.cumsum(skip[1:])]).astype(np.int32)
    state, o_all = B.reuse_chain("gdn", S, [0, n_seg], np.arange(n_seg, dtype=np.int32), cu_step, r["q_seam"], ks, vs,
                                 T_tab=T, T_exp_tab=T_exp, alpha=a_s, beta=b_s)
    # the same chain as separate seam-advance and compose calls
    st1 = B.compose("gdn", S, [0, 1], [0], T_tab=T, T_exp_tab=T_exp)
    nxt = torch.empty_like(st1)
    outs, pos = [], 0
    for i in range(1, n_seg):
        w = int(skip[i])
        sl = slice(pos, pos + w)
        _, o = B.seam_advance("gdn", r["q_seam"][:, sl].contiguous(), ks[:, sl].contiguous(), vs[:, sl].contiguous(),
                              [0, w], alpha=a_s[:, sl].contiguous(), beta=b_s[:, sl].contiguous(),
                              state_in=st1, state_out=st1)
        outs.append(o)
        B.compose("gdn", S, [0, 1], [i], T_tab=T, T_exp_tab=T_exp, S0=st1, out=nxt)
        st1, nxt = nxt, st1
        pos += w
    B.check_device()
    o_steps = torch.cat(outs, dim=1)
    assert_rel(host(state), host(st1), TOL_F32, what="fused chain vs step-by-step calls: end states")
    assert_rel(host(o_all), host(o_steps), TOL_F32, axes=(-1,), what="fused chain vs step-by-step calls: outputs")
    samples = [(0, 0), (29, 31), (13, 7), (29, 2)]
    # The sampled (layer, head) pairs become the heads of one 1-layer problem,
    # so the oracle runs them in parallel.
    pick = lambda x: np.stack([x[layer, :, head].float().cpu().numpy() for layer, head in samples], axis=1)[None]
    one = {key: np.ascontiguousarray(pick(r[key])) for key in ("k", "v", "alpha", "beta")}
    q_full = np.zeros_like(one["k"])
    q_full[0, seam_tok] = pick(r["q_seam"])[0]
    ref_s, ref_o = orc.seam("gdn", q_full, one["k"], one["v"], [0, N], alpha=one["alpha"], beta=one["beta"])
    segs = [int(np.argmax(np.diff(cu))), n_seg - 1]   # the longest and the last (shortest) segment
    for j, (layer, head) in enumerate(samples):
        assert_rel(host(state[:, layer, head]), ref_s[:, 0, j], TOL_BF16, what=f"end state layer {layer} head {head}")
        assert_rel(host(o_all[layer, :, head]), ref_o[0, seam_tok, j], TOL_BF16, axes=(-1,),
                   what=f"seam outputs layer {layer} head {head}")
    for seg in segs:
        b0, b1 = int(cu[seg]) + int(skip[seg]), int(cu[seg + 1])
        sub = {key: np.ascontiguousarray(one[key][:, b0:b1]) for key in one}
        To, So = orc.build_pairs("gdn", sub["k"], sub["v"], [0, b1 - b0], alpha=sub["alpha"], beta=sub["beta"])
        for j, (layer, head) in enumerate(samples):
            assert_rel(host(S[seg, layer, head]), So[0, 0, j], TOL_BF16, what=f"S seg {seg} layer {layer} head {head}")
            assert_rel(gdn_T64(T[seg:seg + 1, layer, head], T_exp[seg:seg + 1, layer, head])[0], To[0, 0, j],
                       TOL_BF16, what=f"T seg {seg} layer {layer} head {head}")


def test_compose_table_full_size_sampled(B):
    """30 layers x 32 heads, 128 pairs, 16 chains of 64 distinct pairs; chains
    0-7 start from zero, 8-15 from a random state.  T tables are random with
    spectral norm ~0.7 (so T S matters at every step) and small exponents."""
    import torch
    L, H, d, P = 30, 32, 128, 128
    ch = synth.compose_chains(seed=0, with_tables=False)
    g = torch.Generator(device="cuda")
    g.manual_seed(1)
    T_tab = torch.randn((P, L, H, d, d), generator=g, device="cuda") * (0.35 / np.sqrt(d))
    S_tab = torch.randn((P, L, H, d, d), generator=g, device="cuda") * (1.0 / np.sqrt(d))
    T_exp = torch.randint(-2, 2, (P, L, H), generator=g, device="cuda", dtype=torch.int32)
    S0 = torch.from_numpy(ch["S0"]).cuda()
    out = B.compose("gdn", S_tab, ch["cu_chain"], ch["seg_idx"], T_tab=T_tab, T_exp_tab=T_exp, S0=S0)
    B.check_device()
    idx = ch["seg_idx"].reshape(16, 64)
    for chain, layer, head in [(0, 0, 0), (15, 29, 31), (8, 11, 5), (3, 20, 17)]:
        pairs = torch.as_tensor(idx[chain], device="cuda")
        Tm = T_tab[pairs, layer, head].cpu().numpy()
        Te = T_exp[pairs, layer, head].cpu().numpy()
        Sp = S_tab[pairs, layer, head].cpu().numpy().astype(np.float64)
        T64 = orc.scaled_to_f64(Tm, Te)
        ref = orc.compose("gdn", T64[:, None, None], Sp[:, None, None], [0, 64], np.arange(64),
                          S0=ch["S0"][chain:chain + 1, layer:layer + 1, head:head + 1])
        assert_rel(host(out[chain, layer, head]), ref[0, 0, 0], TOL_F32, what=f"chain {chain} layer {layer} head {head}")
