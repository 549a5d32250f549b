"""Segment parallelism on one GPU: the request's segments split by the LPT
partition into disjoint sub-batches, each built by its own
hypic_segment_build call (as each rank would), the pairs placed into one
table by segment (what the pair gather produces), then the reuse chain run
on that table -- all equal to the single build call and the same chain,
bit for bit: a pair depends only on its own segment and every kernel reduces
in a fixed order.  The chain itself is checked against the fp64 token loop
over the whole request."""
import numpy as np
import pytest
import torch

from linear_attn_state_hypic_gb300 import shard, synth
from oracle import oracle as orc
from tests.helpers import TOL_BF16, TOL_F32, assert_rel, dev, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from linear_attn_state_hypic_gb300 import binding
    return binding


@pytest.mark.parametrize("d,dtype,world", [(128, "bf16", 2), (128, "bf16", 3), (64, "f32", 2)])
def test_disjoint_builds_then_chain_equal_one_call(B, d, dtype, world):
    lengths = [700, 1, 64, 129, 0, 513, 2048, 90, 300]
    inp = synth.gdn_ragged(seed=31, H=3, d=d, lengths=lengths, n_layers=2, with_q=True, dtype=dtype)
    cu = inp["cu_seqlens"]
    skip = np.minimum(np.array([8, 0, 8, 5, 0, 8, 8, 3, 8], np.int32), np.diff(cu)).astype(np.int32)
    n_seg = len(cu) - 1
    k, v = dev(inp["k"], dtype), dev(inp["v"], dtype)
    al, be = dev(inp["alpha"]), dev(inp["beta"])

    T1, E1, S1 = B.segment_build("gdn", k, v, cu, alpha=al, beta=be, seam_skip=skip)

    T2, E2, S2 = torch.zeros_like(T1), torch.zeros_like(E1), torch.zeros_like(S1)
    parts = shard.lpt_partition(np.diff(cu) - skip, world)
    assert sorted(s for p in parts for s in p) == list(range(n_seg))
    for segs in parts:
        if not segs:
            continue
        sub_cu, sub_skip, tok = shard.local_inputs(cu, skip, segs)
        t = torch.as_tensor(tok, device="cuda")
        pick = lambda x: x.index_select(1, t).contiguous()
        Tr, Er, Sr = B.segment_build("gdn", pick(k), pick(v), sub_cu, alpha=pick(al), beta=pick(be),
                                     seam_skip=sub_skip)
        rows = torch.as_tensor(segs, device="cuda")
        T2[rows], E2[rows], S2[rows] = Tr, Er, Sr
    B.check_device()
    np.testing.assert_array_equal(host(T2), host(T1))
    np.testing.assert_array_equal(host(E2), host(E1))
    np.testing.assert_array_equal(host(S2), host(S1))

    # one chain over every segment in order, as the reuse path runs it: step s
    # advances the state through segment s's seam window (its first skip[s]
    # tokens, left out of the cached pair) and then composes the body pair
    seg_idx = np.arange(n_seg, dtype=np.int32)
    cu_chain = np.array([0, n_seg], np.int32)
    heads = np.concatenate([np.arange(cu[s], cu[s] + skip[s]) for s in range(n_seg)])
    cu_step = np.concatenate([[0], np.cumsum(skip)]).astype(np.int32)
    tt = torch.as_tensor(heads, device="cuda")
    q = dev(inp["q"], dtype)
    sq, sk, sv, sa, sb = (x.index_select(1, tt).contiguous() for x in (q, k, v, al, be))
    outs = []
    for T, E, S in ((T1, E1, S1), (T2, E2, S2)):
        out, o = B.reuse_chain("gdn", S, cu_chain, seg_idx, cu_step, sq, sk, sv, T_tab=T, T_exp_tab=E,
                               alpha=sa, beta=sb)
        outs.append((host(out), host(o)))
    B.check_device()
    np.testing.assert_array_equal(outs[1][0], outs[0][0])
    np.testing.assert_array_equal(outs[1][1], outs[0][1])
    # and the chain is the request's own recurrence: its end state and seam
    # outputs are those of the fp64 token loop over all tokens
    n = int(cu[-1])
    ref_s, ref_o = orc.seam("gdn", inp["q"], inp["k"], inp["v"], [0, n], alpha=inp["alpha"], beta=inp["beta"])
    tol = TOL_BF16 if dtype == "bf16" else TOL_F32
    assert_rel(outs[0][0][0], ref_s[0], tol, what="chain end state vs the full-sequence oracle")
    assert_rel(outs[0][1], ref_o[:, heads], tol, axes=(-1,), what="seam outputs vs the full-sequence oracle")
