"""Segment parallelism across GPUs: the host side.

Every cached pair (T_C, S(C|0)) depends only on its own segment (the aibase
article on HYPIC, paragraph on the linear layers), so a request's segments can
be built on different GPUs with no exchange during the build.  The article's
segment parallelism has scatter workers that build and one combine worker that
composes, with the workers' results streamed to it segment by segment rather
than in one burst.  This module holds that plan:

* ``lpt_partition``: segments to ranks, longest body first onto the least
  loaded rank (the build's own work order, applied across GPUs);
* ``local_inputs``: a rank's sub-batch in the request's packed token array;
* ``combine_rows``: where each rank's pairs land in the combine rank's table
  (rank after rank, each in its own segment order), so that the compose reads
  them through its segment index with no placement copy;
* ``stream_pairs``: the one exchange.  Each rank builds its share in batches
  and sends every finished batch straight into the combine rank's table
  (point-to-point: NCCL for CUDA tensors, gloo for CPU tensors); the combine
  rank posts its receives up front and builds its own share in place.  No
  rank receives pairs it does not compose.

The build and compose calls themselves are the library's; nothing here does
arithmetic on the pairs."""
from __future__ import annotations

import numpy as np


def lpt_partition(body_lengths, world: int) -> list[list[int]]:
    """Segment indices per rank: each segment, longest first (ties: lower
    index first), goes to the rank with the fewest tokens so far (ties: lower
    rank).  Every rank's list is in increasing segment order."""
    lengths = np.asarray(body_lengths, dtype=np.int64)
    if world < 1:
        raise ValueError(f"world = {world}")
    order = sorted(range(len(lengths)), key=lambda s: (-int(lengths[s]), s))
    load = [0] * world
    parts: list[list[int]] = [[] for _ in range(world)]
    for s in order:
        r = min(range(world), key=lambda i: (load[i], i))
        parts[r].append(s)
        load[r] += int(lengths[s])
    return [sorted(p) for p in parts]


def local_inputs(cu_seqlens, seam_skip, segs):
    """Token ranges of a rank's segments in the request's packed token array:
    (cu_seqlens, seam_skip) of the sub-batch and the token index array that
    gathers its tokens (segments concatenated in the given order)."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    skip = np.zeros(len(cu) - 1, np.int64) if seam_skip is None else np.asarray(seam_skip, np.int64)
    idx = [np.arange(cu[s], cu[s + 1]) for s in segs]
    lens = [int(cu[s + 1] - cu[s]) for s in segs]
    sub_cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    sub_skip = np.array([skip[s] for s in segs], np.int32)
    tok = np.concatenate(idx) if idx else np.zeros(0, np.int64)
    return sub_cu, sub_skip, tok


def combine_rows(parts):
    """(offsets, row_of): rank r's pairs occupy rows [offsets[r], offsets[r] +
    len(parts[r])) of the combine rank's table, in the rank's own segment
    order; row_of[s] is the row of segment s (the compose's segment index)."""
    n_seg = sum(len(p) for p in parts)
    offsets = np.concatenate([[0], np.cumsum([len(p) for p in parts])]).astype(np.int64)
    row_of = np.full(n_seg, -1, np.int64)
    for r, p in enumerate(parts):
        for i, s in enumerate(p):
            row_of[s] = offsets[r] + i
    if n_seg and row_of.min() < 0:
        raise ValueError("the parts do not cover every segment exactly once")
    return offsets, row_of


def batch_bounds(n: int, n_batches: int):
    """Split n consecutive items into at most n_batches non-empty runs:
    a list of (start, stop)."""
    n_batches = max(1, min(int(n_batches), n)) if n else 0
    edges = [round(i * n / n_batches) for i in range(n_batches + 1)] if n_batches else [0]
    return [(edges[i], edges[i + 1]) for i in range(n_batches) if edges[i + 1] > edges[i]]


def stream_pairs(build_batch, tables, parts, rank: int, *, dst: int = 0, n_batches: int = 4, group=None):
    """Build this rank's share of the pairs in batches and stream them to the
    combine rank ``dst``.

    build_batch(lo, hi, views): fills ``views`` (one tensor per pair table,
    leading dimension hi - lo) with the pairs of this rank's segments
    parts[rank][lo:hi].  tables: on ``dst``, the full tables (leading
    dimension = every segment, laid out by ``combine_rows``); on every other
    rank, tables with len(parts[rank]) rows for its own share.  Returns the
    list of outstanding communication handles' results (all waited)."""
    import torch.distributed as dist
    world = len(parts)
    offsets, _ = combine_rows(parts)
    handles = []
    if rank == dst:
        for r in range(world):  # every receive posted before any build: the senders never wait on them
            if r == dst:
                continue
            for lo, hi in batch_bounds(len(parts[r]), n_batches):
                a, b = offsets[r] + lo, offsets[r] + hi
                for t in tables:
                    handles.append(dist.irecv(t[a:b], src=r, group=group))
        base = offsets[dst]
        for lo, hi in batch_bounds(len(parts[dst]), n_batches):
            build_batch(lo, hi, [t[base + lo:base + hi] for t in tables])
    else:
        for lo, hi in batch_bounds(len(parts[rank]), n_batches):
            views = [t[lo:hi] for t in tables]
            build_batch(lo, hi, views)
            for v in views:  # (a batch is sent as soon as it is built; the next one builds meanwhile)
                handles.append(dist.isend(v, dst=dst, group=group))
    for h in handles:
        h.wait()
    return len(handles)
