"""Prefill of one sequence split over the ranks of a process group.

The states are additive across segments ("Expanding Attention", abstract:
the states are additive across chunks, so prefill admits a parallel scan), so
a sequence cut into contiguous segments, one per rank, is prefilled in three
steps:

  1. every rank sums its own segment's state (tsa_prefill_states, from zero);
  2. the segment sums are all-gathered over the group (the one exchange);
  3. every rank forms its prefix -- the initial state plus the sums of the
     segments before its own, added with tsa_state_merge -- and runs
     tsa_prefill on its segment with TSA_PREFILL_ACCUMULATE from it, which
     gives its segment's outputs; adding the later segments' sums then gives
     every rank the state after the whole sequence.

Every step on the data runs in the library's kernels; this module only picks
the segments and moves the sums between ranks (through host memory when the
group's backend is gloo, which the tests use on CPU-only machines).
"""
from __future__ import annotations


def shard_bounds(N: int, world: int, rank: int) -> tuple[int, int]:
    """Token range [start, end) of `rank`'s segment: contiguous, in rank
    order, lengths differing by at most one."""
    if world < 1 or not (0 <= rank < world) or N < 0:
        raise ValueError(f"bad shard request N={N} world={world} rank={rank}")
    base, extra = divmod(N, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def all_gather_states(x, group=None):
    """The list of every rank's `x` (same shape and dtype on every rank), in
    rank order. Under gloo, device tensors are staged through host memory."""
    import torch
    import torch.distributed as dist
    world = dist.get_world_size(group)
    staged = x
    if x.is_cuda and dist.get_backend(group) == "gloo":
        staged = x.detach().cpu()
    parts = [torch.empty_like(staged) for _ in range(world)]
    dist.all_gather(parts, staged.contiguous(), group=group)
    if staged is not x:
        parts = [p.to(x.device) for p in parts]
    return parts


class LibraryOps:
    """The three library calls the sharded prefill is made of."""

    def __init__(self, tsa_module=None):
        if tsa_module is None:
            from . import tsa as tsa_module
        self.T = tsa_module

    def new_states(self, cfg, like):
        return self.T.new_states(cfg, like.device)

    def segment_sum(self, cfg, n, k, v, states):
        self.T.prefill_states(cfg, n, k, v, states)

    def prefill(self, cfg, n, q, k, v, out, states, accumulate):
        self.T.prefill(cfg, n, q, k, v, out, states, accumulate=accumulate)

    def merge(self, cfg, a, b):
        self.T.state_merge(cfg, a, b)

    def zero(self, cfg, states):
        # a prefill of no tokens without ACCUMULATE zeroes the states
        self.T.prefill(cfg, 0, None, None, None, None, states, accumulate=False)


def sharded_prefill(cfg, q, k, v, out, states, accumulate: bool = False, group=None, ops=None):
    """Prefill of one sequence whose tokens are split over the group's ranks.

    On every rank: q, k, v are its segment ([B, H, n_r, d] with the segments
    in rank order, e.g. from shard_bounds); out receives the segment's outputs;
    states holds, with accumulate, the state before the whole sequence (the
    same on every rank), and on return the state after the whole sequence (the
    same on every rank)."""
    import torch.distributed as dist
    ops = ops or LibraryOps()
    rank = dist.get_rank(group)
    n = int(k.shape[2])
    delta = ops.new_states(cfg, states)
    if n > 0:
        ops.segment_sum(cfg, n, k, v, delta)
    else:
        ops.zero(cfg, delta)
    deltas = all_gather_states(delta, group)
    if not accumulate:
        ops.zero(cfg, states)
    for r in range(rank):
        ops.merge(cfg, states, deltas[r])
    ops.prefill(cfg, n, q, k, v, out, states, accumulate=True)
    for r in range(rank + 1, len(deltas)):
        ops.merge(cfg, states, deltas[r])
    return states
