"""Splitting the SSD path across GPUs.

Every (batch row, head) recurrence is independent, so the scan and the
decode step shard over batch rows and heads with no exchange in the data
path: each GPU runs ssd_scan_fwd / ssd_state_update on its own slice.  Heads
are split on group boundaries so each GPU keeps whole groups (heads of one
group share B and C, and the tensor-core kernel pairs them).  A packed batch
of sequences splits into contiguous runs of whole sequences with even token
shares (ssd_scan_fwd_varlen on each run).

One long sequence can also split over GPUs by tokens (token_range,
scan_sequence_sharded), at the cost of one exchange: each GPU scans its range
from a zero state, the ranges' (log-decay, state) pairs are all-gathered,
each GPU chains them to the state entering its range, and scans the range
again from it.

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


def token_range(seqlen: int, world: int, rank: int, align: int = 128):
    """Contiguous [t0, t1) token range of one sequence for `rank` of `world`:
    even shares of whole `align`-token tiles (the tensor-core kernels' tile),
    the ragged tail with the last rank.  With more ranks than tiles the
    trailing ranks get empty ranges."""
    if not 0 <= rank < world:
        raise ValueError("rank out of range")
    if seqlen < 0 or align <= 0:
        raise ValueError("seqlen must be >= 0 and align > 0")
    tiles = -(-seqlen // align)
    t0 = min(seqlen, (tiles * rank // world) * align)
    t1 = min(seqlen, (tiles * (rank + 1) // world) * align)
    return t0, t1


def scan_sequence_sharded(x, dt, A, B, C, D=None, init=None, chunk=256, *, group=None,
                          ops=None, **dt_kw):
    """This rank's token range of one long sequence, scanned as part of the
    whole (x [b, Lr, H, P], dt [b, Lr, H], B, C [b, Lr, G, N]: the rank's
    tokens; A, D, init [b, H, P, N] or None: the same on every rank).

    Step-3 of the recurrence at the granularity of one rank's range: the
    range's state from a zero start F_r and log-decay a_r = A * sum(dt) are
    all-gathered, H_in[0] = init and H_in[r+1] = exp(a_r) H_in[r] + F_r give
    the state entering this range, and the range is scanned again from it.
    Returns (y, final): y of the rank's tokens and the state at the end of
    its range (the sequence's final state on the last rank).

    ``ops`` = (scan, range_log_decay, chain_states) with the signatures of the
    package's functions; the default is the package's own (the library's
    kernels), and the tests pass CPU stand-ins.  dt transform keywords go to
    both the scans and the log-decay."""
    import torch
    import torch.distributed as dist
    if ops is None:
        from . import _binding as ssd
        ops = (lambda *a, **k: ssd.scan_fwd(*a, **k), ssd.range_log_decay, ssd.chain_states)
    scan, log_decay_of, chain = ops
    world = dist.get_world_size(group) if dist.is_initialized() else 1
    rank = dist.get_rank(group) if dist.is_initialized() else 0
    b, L, H, P = x.shape
    N = B.shape[3]
    if L > 0:
        _, contrib = scan(x, dt, A, B, C, D, chunk, None, **dt_kw)
        a = log_decay_of(dt, A, **dt_kw)
    else:       # an empty range passes the state through unchanged (states in A's dtype)
        contrib = torch.zeros((b, H, P, N), dtype=A.dtype, device=x.device)
        a = torch.zeros((b, H), dtype=A.dtype, device=x.device)
    if world > 1:
        contribs = [torch.empty_like(contrib) for _ in range(world)]
        decays = [torch.empty_like(a) for _ in range(world)]
        dist.all_gather(contribs, contrib.contiguous(), group=group)
        dist.all_gather(decays, a.contiguous(), group=group)
    else:
        contribs, decays = [contrib], [a]
    entering = chain(torch.stack(contribs), torch.stack(decays), init)[rank].contiguous()
    if L == 0:
        return x.new_empty((b, 0, H, P)), entering
    return scan(x, dt, A, B, C, D, chunk, entering, **dt_kw)
