"""Segment parallelism across GPUs: the host side.

Every cached pair (T_C, S(C|0)) depends only on its own segment (the aibase
article on HYPIC, paragraph on the linear layers), so a request's segments can
be built on different GPUs with no exchange during the build; the only
exchange is one gather of the finished pairs to the GPU that composes them
(the article's scatter / combine workers).  This module holds that plan:

* ``lpt_partition``: segments to ranks, longest body first onto the least
  loaded rank (the build's own work order, applied across GPUs);
* ``gather_pairs``: every rank's pair tables into full tables indexed by
  segment, on every rank (``torch.distributed.all_gather`` of fixed-size
  padded blocks: NCCL for CUDA tensors, gloo for CPU tensors).

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


def gather_pairs(tables, segs, n_seg: int, group=None):
    """Full pair tables from every rank's share.

    tables: tensors of this rank's pairs, each with the segment as its leading
    dimension (len(segs) rows, e.g. T mantissa, T exponent, S); segs: this
    rank's segment indices (the rows' order).  Returns, on every rank, the
    same tensors with n_seg rows, row s holding segment s's pair."""
    import torch
    import torch.distributed as dist
    world = dist.get_world_size(group)
    counts = [None] * world
    dist.all_gather_object(counts, list(int(s) for s in segs), group=group)
    width = max(len(c) for c in counts)
    out = []
    for t in tables:
        pad = torch.zeros((width,) + tuple(t.shape[1:]), dtype=t.dtype, device=t.device)
        pad[: t.shape[0]] = t
        parts = [torch.empty_like(pad) for _ in range(world)]
        dist.all_gather(parts, pad, group=group)
        full = torch.empty((n_seg,) + tuple(t.shape[1:]), dtype=t.dtype, device=t.device)
        for r, seg_list in enumerate(counts):
            if seg_list:
                full[torch.as_tensor(seg_list, device=t.device)] = parts[r][: len(seg_list)]
        out.append(full)
    return out
