"""Segment parallelism, host side (CPU only): the LPT partition of a
request's segments across ranks, the token gather of a rank's sub-batch, and
the pair gather itself over two real torch.distributed ranks (gloo).

In the two-rank test each rank builds the pairs of its own segments (with the
oracle: there is no GPU here), the ranks exchange them with gather_pairs, and
the gathered tables -- and the reuse chain composed from them -- must equal
the single-process build of the whole batch exactly: every pair depends only
on its own segment."""
import os
import socket
import sys

import numpy as np
import pytest

from linear_attn_state_hypic_gb300 import shard, synth
from oracle import oracle as orc

REPO = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_lpt_partition_assigns_every_segment_once_and_balances():
    rng = np.random.default_rng(0)
    lengths = rng.integers(0, 2049, 77)
    for world in (1, 2, 3, 8):
        parts = shard.lpt_partition(lengths, world)
        assert len(parts) == world
        flat = sorted(s for p in parts for s in p)
        assert flat == list(range(77))
        assert all(p == sorted(p) for p in parts)
        loads = [int(lengths[p].sum()) if p else 0 for p in parts]
        # greedy longest-first: the spread never exceeds the longest body
        assert max(loads) - min(loads) <= int(lengths.max())
    assert shard.lpt_partition([5, 5, 5], 2) == [[0, 2], [1]]


def test_local_inputs_gathers_the_rank_tokens():
    cu = np.array([0, 4, 4, 10, 13], np.int32)
    skip = np.array([0, 0, 2, 1], np.int32)
    sub_cu, sub_skip, tok = shard.local_inputs(cu, skip, [0, 3])
    assert sub_cu.tolist() == [0, 4, 7]
    assert sub_skip.tolist() == [0, 1]
    assert tok.tolist() == [0, 1, 2, 3, 10, 11, 12]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _case():
    inp = synth.gdn_ragged(seed=21, H=2, d=16, lengths=[40, 7, 64, 0, 23, 90, 33], dtype="f32")
    inp["seam_skip"] = np.array([0, 3, 8, 0, 5, 8, 2], np.int32)
    return inp


def _rank_main(rank, world, port, out_dir):
    sys.path.insert(0, REPO)
    import torch
    import torch.distributed as dist
    from linear_attn_state_hypic_gb300 import shard as sh
    from oracle import oracle as o
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    inp = _case()
    cu, skip = inp["cu_seqlens"], inp["seam_skip"]
    n_seg = len(cu) - 1
    parts = sh.lpt_partition(np.diff(cu) - skip, world)
    segs = parts[rank]
    sub_cu, sub_skip, tok = sh.local_inputs(cu, skip, segs)
    pick = lambda x: np.ascontiguousarray(x[:, tok])
    T, S = o.build_pairs("gdn", pick(inp["k"]), pick(inp["v"]), sub_cu, alpha=pick(inp["alpha"]),
                         beta=pick(inp["beta"]), skip=sub_skip, n_threads=1)
    T_full, S_full = sh.gather_pairs([torch.from_numpy(T), torch.from_numpy(S)], segs, n_seg)
    np.save(os.path.join(out_dir, f"T{rank}.npy"), T_full.numpy())
    np.save(os.path.join(out_dir, f"S{rank}.npy"), S_full.numpy())
    dist.destroy_process_group()


def test_two_gloo_ranks_gather_equals_one_build(tmp_path):
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
    world = 2
    ctx = mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=False,
                             start_method="spawn")
    while not ctx.join(timeout=120):
        pass
    inp = _case()
    cu, skip = inp["cu_seqlens"], inp["seam_skip"]
    T1, S1 = orc.build_pairs("gdn", inp["k"], inp["v"], cu, alpha=inp["alpha"], beta=inp["beta"], skip=skip,
                             n_threads=1)
    for r in range(world):
        Tg, Sg = np.load(tmp_path / f"T{r}.npy"), np.load(tmp_path / f"S{r}.npy")
        np.testing.assert_array_equal(Tg, T1)
        np.testing.assert_array_equal(Sg, S1)
    # the chain composed from the gathered tables is the single-process one
    n_seg = len(cu) - 1
    Tg, Sg = np.load(tmp_path / "T0.npy"), np.load(tmp_path / "S0.npy")
    ref = orc.compose("gdn", T1, S1, [0, n_seg], np.arange(n_seg))
    got = orc.compose("gdn", Tg, Sg, [0, n_seg], np.arange(n_seg))
    np.testing.assert_array_equal(got, ref)
