"""Segment parallelism, host side (CPU only): the LPT partition of a
request's segments across ranks, the token gather of a rank's sub-batch, the
combine rank's table layout, and the pair stream itself over real
torch.distributed ranks (gloo).

In the multi-rank test each rank builds the pairs of its own segments batch by
batch (with the oracle: there is no GPU here) and streams each finished batch
to the combine rank, which builds its own share in place.  The combine rank's
table -- read through its segment index -- and the chain composed from it must
equal the single-process build of the whole batch exactly: every pair depends
only on its own segment.  The other ranks receive nothing."""
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


def _rank_main(rank, world, port, out_dir, n_batches):
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
    k, v, al, be = (pick(inp[key]) for key in ("k", "v", "alpha", "beta"))
    d = k.shape[-1]

    def build_batch(lo, hi, views):  # the pairs of segs[lo:hi], from their own tokens only
        a, b = int(sub_cu[lo]), int(sub_cu[hi])
        T, S = o.build_pairs("gdn", k[:, a:b], v[:, a:b], sub_cu[lo:hi + 1] - a, alpha=al[:, a:b], beta=be[:, a:b],
                             skip=sub_skip[lo:hi], n_threads=1)
        views[0].copy_(torch.from_numpy(T))
        views[1].copy_(torch.from_numpy(S))

    rows = n_seg if rank == 0 else len(segs)
    tables = [torch.full((rows, 1, 2, d, d), float("nan"), dtype=torch.float64) for _ in range(2)]
    sh.stream_pairs(build_batch, tables, parts, rank, dst=0, n_batches=n_batches)
    if rank == 0:
        np.save(os.path.join(out_dir, "T.npy"), tables[0].numpy())
        np.save(os.path.join(out_dir, "S.npy"), tables[1].numpy())
    dist.destroy_process_group()


@pytest.mark.parametrize("world,n_batches", [(2, 1), (2, 3), (3, 2)])
def test_gloo_ranks_stream_pairs_equal_one_build(tmp_path, world, n_batches):
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
    ctx = mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path), n_batches), nprocs=world,
                             join=False, start_method="spawn")
    while not ctx.join(timeout=120):
        pass
    inp = _case()
    cu, skip = inp["cu_seqlens"], inp["seam_skip"]
    n_seg = len(cu) - 1
    T1, S1 = orc.build_pairs("gdn", inp["k"], inp["v"], cu, alpha=inp["alpha"], beta=inp["beta"], skip=skip,
                             n_threads=1)
    parts = shard.lpt_partition(np.diff(cu) - skip, world)
    _, row_of = shard.combine_rows(parts)
    Tg, Sg = np.load(tmp_path / "T.npy"), np.load(tmp_path / "S.npy")
    np.testing.assert_array_equal(Tg[row_of], T1)
    np.testing.assert_array_equal(Sg[row_of], S1)
    # the chain composed on the combine rank, through its segment index, is the single-process one
    ref = orc.compose("gdn", T1, S1, [0, n_seg], np.arange(n_seg))
    got = orc.compose("gdn", Tg, Sg, [0, n_seg], row_of)
    np.testing.assert_array_equal(got, ref)


def test_combine_rows_and_batches():
    offsets, row_of = shard.combine_rows([[0, 3], [1], [2, 4, 5]])
    assert offsets.tolist() == [0, 2, 3, 6]
    assert row_of.tolist() == [0, 2, 3, 1, 4, 5]
    with pytest.raises(ValueError):
        shard.combine_rows([[0], [0]])
    assert shard.batch_bounds(7, 3) == [(0, 2), (2, 5), (5, 7)]
    assert shard.batch_bounds(2, 4) == [(0, 1), (1, 2)]
    assert shard.batch_bounds(0, 4) == []
