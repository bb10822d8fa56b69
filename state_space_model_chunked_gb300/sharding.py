"""Splitting the SSD path across GPUs.

Every (batch row, head) recurrence is independent, so the scan and the
decode step shard over batch rows and heads with no exchange in the data
path: each GPU runs ssd_scan_fwd / ssd_state_update on its own slice.  Heads
are split on group boundaries so each GPU keeps whole groups (heads of one
group share B and C, and the tensor-core kernel pairs them).  A packed batch
of sequences splits into contiguous runs of whole sequences with even token
shares (ssd_scan_fwd_varlen on each run).

Timing across ranks takes the maximum over ranks (the slowest GPU finishes
the job).
"""
from __future__ import annotations


def head_range(nheads: int, ngroups: int, world: int, rank: int):
    """Contiguous [start, stop) head range for `rank` of `world`, cut on group
    boundaries and as even as whole groups allow.  With more ranks than
    groups, the trailing ranks get empty ranges."""
    if nheads % ngroups:
        raise ValueError("nheads must be a multiple of ngroups")
    if not 0 <= rank < world:
        raise ValueError("rank out of range")
    per_group = nheads // ngroups
    g0 = (ngroups * rank) // world
    g1 = (ngroups * (rank + 1)) // world
    return g0 * per_group, g1 * per_group


def head_shard(nheads: int, ngroups: int, world: int, rank: int, pair: int = 2):
    """Heads [h0, h1) and groups [g0, g1) of `rank`.  With at least as many
    groups as ranks this is head_range (whole groups).  With fewer groups --
    the 2.7B layer has one group of 80 heads -- each group is split evenly
    among world / ngroups ranks on `pair`-head boundaries (the tensor-core
    kernel pairs the heads of a group); every rank of a group then reads that
    group's B and C, which are inputs, so nothing is exchanged.  Shapes that
    do not split that way fall back to head_range."""
    if nheads % ngroups:
        raise ValueError("nheads must be a multiple of ngroups")
    if not 0 <= rank < world:
        raise ValueError("rank out of range")
    per_group = nheads // ngroups
    parts = world // ngroups if world > ngroups and world % ngroups == 0 else 0
    if parts and per_group % (pair * parts) == 0:
        g = rank // parts
        share = per_group // parts
        h0 = g * per_group + (rank % parts) * share
        return h0, h0 + share, g, g + 1
    h0, h1 = head_range(nheads, ngroups, world, rank)
    return h0, h1, h0 // per_group, h1 // per_group


def batch_range(batch: int, world: int, rank: int):
    """Contiguous [start, stop) batch-row range for `rank` of `world`."""
    if not 0 <= rank < world:
        raise ValueError("rank out of range")
    return (batch * rank) // world, (batch * (rank + 1)) // world


def sequence_range(cu_seqlens, world: int, rank: int):
    """Contiguous [start, stop) range of packed sequences for `rank` of
    `world`, cut at the sequence boundaries nearest to even shares of the
    tokens (a sequence is never split: its recurrence is sequential).  Every
    rank's token count is within the longest sequence of total / world.
    Returns (s0, s1, offsets): the rank's cu_seqlens rebased to 0."""
    import numpy as np
    if not 0 <= rank < world:
        raise ValueError("rank out of range")
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    if cu.ndim != 1 or cu.size < 1 or cu[0] != 0 or np.any(np.diff(cu) < 0):
        raise ValueError("cu_seqlens must start at 0 and not decrease")
    nseq, total = cu.size - 1, int(cu[-1])

    def cut(r):
        if r <= 0:
            return 0
        if r >= world:
            return nseq
        target = total * r / world
        i = int(np.searchsorted(cu, target))        # first boundary >= target
        if i > 0 and target - cu[i - 1] < (cu[i] - target if i <= nseq else np.inf):
            i -= 1
        return min(max(i, 0), nseq)

    s0, s1 = cut(rank), cut(rank + 1)
    s1 = max(s1, s0)
    return s0, s1, (cu[s0:s1 + 1] - cu[s0]).astype(np.int32)


def max_over_ranks(value: float, dist=None, device=None) -> float:
    """Maximum of a per-rank float over the process group (identity without one)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())
