"""hypic_reuse_chain against the oracle: per step, the seam window's token
recurrence (with its outputs) and then the step's cached pair, for every
chain and (layer, head).

* GDN, d = 128: the fused tensor-core kernel (state on chip for the whole
  chain), with bf16 and fp32 seam inputs, seam widths 0, 1, 3, 8, 9 and 17
  (empty, padded, exactly one unit, several units), an empty chain and a
  random start state.
* GDN, d = 64, and the decay families: the step-by-step path (seam advance and
  compose kernels with a workspace).

The pair tables are random (GDN: T with spectral norm ~0.7 and small
exponents, so T S matters at every step); the oracle composes the same
tables in fp64 and runs the seam recurrence on the same (bf16-rounded)
inputs."""
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


def make_case(seed, fam, L, H, d, n_pairs, chain_lens, widths, dtype, with_s0, variant="faithful"):
    rng = np.random.default_rng(seed)
    n_chains = len(chain_lens)
    cu_chain = np.concatenate([[0], np.cumsum(chain_lens)]).astype(np.int32)
    n_steps = int(cu_chain[-1])
    assert len(widths) == n_steps
    seg_idx = rng.integers(0, n_pairs, n_steps).astype(np.int32)
    cu_step = np.concatenate([[0], np.cumsum(widths)]).astype(np.int32)
    N = int(cu_step[-1])
    S_tab = (rng.standard_normal((n_pairs, L, H, d, d)) / np.sqrt(d)).astype(np.float32)
    T_tab = T_exp = None
    if fam == "gdn":
        T_tab = (rng.standard_normal((n_pairs, L, H, d, d)) * (0.35 / np.sqrt(d))).astype(np.float32)
        T_exp = rng.integers(-2, 2, (n_pairs, L, H)).astype(np.int32)
    elif fam == "retnet":
        T_tab = rng.uniform(0.3, 0.99, (n_pairs, L, H)).astype(np.float32)
    elif fam == "gla":
        T_tab = rng.uniform(0.3, 0.99, (n_pairs, L, H, d)).astype(np.float32)
    k = synth._unit_rows(rng, (L, N, H, d))
    q = synth._unit_rows(rng, (L, N, H, d))
    v = rng.standard_normal((L, N, H, d)).astype(np.float32)
    if dtype == "bf16":
        q, k, v = (synth.round_bf16(x) for x in (q, k, v))
    gates = {}
    if fam == "gdn":
        gates["alpha"], gates["beta"] = synth.gdn_gates(rng, (L, N, H), variant)
    elif fam == "retnet":
        gates["gamma"] = rng.uniform(0.8, 0.99, (L, H)).astype(np.float32)
    elif fam == "gla":
        gates["g"] = rng.uniform(0.8, 1.0, (L, N, H, d)).astype(np.float32)
    S0 = (rng.standard_normal((n_chains, L, H, d, d)) / np.sqrt(d)).astype(np.float32) if with_s0 else None
    return dict(cu_chain=cu_chain, seg_idx=seg_idx, cu_step=cu_step, S_tab=S_tab, T_tab=T_tab, T_exp=T_exp,
                q=q, k=k, v=v, gates=gates, S0=S0)


def oracle_chain(fam, c):
    """Step by step in fp64: seam window (outputs kept), then the one-step compose."""
    T64 = None
    if fam == "gdn":
        T64 = orc.scaled_to_f64(c["T_tab"], c["T_exp"])
    elif fam in ("retnet", "gla"):
        T64 = c["T_tab"].astype(np.float64)
    n_chains = len(c["cu_chain"]) - 1
    L, N, H, d = c["k"].shape
    ends = np.zeros((n_chains, L, H, d, d))
    o_all = np.zeros((L, N, H, d))
    for r in range(n_chains):
        S = None if c["S0"] is None else c["S0"][r:r + 1].astype(np.float64)
        for j in range(c["cu_chain"][r], c["cu_chain"][r + 1]):
            t0, t1 = int(c["cu_step"][j]), int(c["cu_step"][j + 1])
            if t1 > t0:
                sl = slice(t0, t1)
                g = {key: (val[:, sl] if val.ndim >= 3 else val) for key, val in c["gates"].items()}
                S, o = orc.seam(fam, c["q"][:, sl], c["k"][:, sl], c["v"][:, sl], [0, t1 - t0], state_in=S, **g)
                o_all[:, sl] = o
            S = orc.compose(fam, T64, c["S_tab"], [0, 1], [int(c["seg_idx"][j])], S0=S)
        ends[r] = 0.0 if S is None else S[0]
    return ends, o_all


def run_gpu(B, fam, c, dtype):
    g = {key: dev(val) for key, val in c["gates"].items()}
    out, o = B.reuse_chain(fam, dev(c["S_tab"]), c["cu_chain"], c["seg_idx"], c["cu_step"],
                           dev(c["q"], dtype), dev(c["k"], dtype), dev(c["v"], dtype),
                           T_tab=dev(c["T_tab"]), T_exp_tab=None if c["T_exp"] is None else dev(c["T_exp"]),
                           S0=dev(c["S0"]), **g)
    B.check_device()
    return host(out), host(o)


def check(B, fam, c, dtype, tol):
    out, o = run_gpu(B, fam, c, dtype)
    ref, ref_o = oracle_chain(fam, c)
    assert_rel(out, ref, tol, what=f"{fam} chain end states")
    t = np.concatenate([np.arange(c["cu_step"][j], c["cu_step"][j + 1]) for j in range(len(c["cu_step"]) - 1)])
    if len(t):
        assert_rel(o[:, t], ref_o[:, t], tol, axes=(-1,), what=f"{fam} seam outputs")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("with_s0", [False, True])
def test_chain_fused_gdn_d128(B, dtype, with_s0):
    c = make_case(11, "gdn", L=2, H=3, d=128, n_pairs=5, chain_lens=[4, 0, 3, 1],
                  widths=[0, 8, 3, 17, 8, 1, 9, 0], dtype=dtype, with_s0=with_s0)
    check(B, "gdn", c, dtype, TOL_F32)


@pytest.mark.parametrize("variant", ["faithful", "fastdecay"])
def test_chain_fused_gdn_d128_gaps_and_full_units(B, variant):
    """Steps without a seam inside a chain (the next compose takes the composed
    column as it is), consecutive ones, windows of exactly one, two and three full
    units, a chain that starts without a seam, and fast decay (alpha in
    [0.05, 0.6]: a unit's decay down to ~1e-11)."""
    c = make_case(14, "gdn", L=1, H=2, d=128, n_pairs=4, chain_lens=[6, 2],
                  widths=[8, 0, 16, 0, 0, 24, 0, 5], dtype="f32", with_s0=True, variant=variant)
    check(B, "gdn", c, "f32", TOL_F32)


def test_chain_fused_matches_step_by_step_calls(B):
    """The fused call equals the same chain run as hypic_seam_advance +
    hypic_compose calls (the library's own kernels, step by step)."""
    import torch
    c = make_case(12, "gdn", L=1, H=2, d=128, n_pairs=3, chain_lens=[3], widths=[8, 8, 8], dtype="bf16",
                  with_s0=False)
    out, o = run_gpu(B, "gdn", c, "bf16")
    S_tab, T_tab, T_exp = dev(c["S_tab"]), dev(c["T_tab"]), dev(c["T_exp"])
    q, k, v = (dev(c[x], "bf16") for x in ("q", "k", "v"))
    al, be = dev(c["gates"]["alpha"]), dev(c["gates"]["beta"])
    state = None
    o2 = torch.zeros((1, 24, 2, 128), dtype=torch.float32, device="cuda")
    for j in range(3):
        sl = slice(8 * j, 8 * j + 8)
        state, oj = B.seam_advance("gdn", q[:, sl].contiguous(), k[:, sl].contiguous(), v[:, sl].contiguous(), [0, 8],
                                   alpha=al[:, sl].contiguous(), beta=be[:, sl].contiguous(), state_in=state)
        o2[:, sl] = oj
        state = B.compose("gdn", S_tab, [0, 1], [int(c["seg_idx"][j])], T_tab=T_tab, T_exp_tab=T_exp, S0=state)
    B.check_device()
    assert_rel(out, host(state), TOL_F32, what="fused vs step-by-step end state")
    assert_rel(o, host(o2), TOL_F32, axes=(-1,), what="fused vs step-by-step seam outputs")


@pytest.mark.parametrize("fam,d", [("gdn", 64), ("retnet", 32), ("gla", 64), ("vanilla", 16)])
def test_chain_step_by_step_path(B, fam, d):
    c = make_case(13, fam, L=2, H=2, d=d, n_pairs=4, chain_lens=[3, 2, 0], widths=[5, 0, 8, 2, 1],
                  dtype="f32", with_s0=True)
    check(B, fam, c, "f32", TOL_F32)
