"""Host-side partitioning of the chunked forward pass across ranks, one GPU per rank.

Two ways to spread the work:

* Independent items. Every (sequence, head) pair -- and every value column of a head's
  state -- evolves independently, so ranks can own disjoint sets of sequences (or of
  heads) and run ``chunk_fwd`` on their own slice with no collective on the data path.
  ``partition_sequences`` balances contiguous sequence ranges by token count;
  ``partition_heads`` splits heads evenly.

* One long sequence split in time. The inter-chunk recurrence is serial ("chunks run
  serially through the state recurrence", "From Numerical Stability to Load
  Balancing", §2.1), so a sequence cut into segments needs exactly one exchange per
  boundary: the final state of segment r is the initial state of segment r + 1.
  ``time_split_forward`` runs that hand-off with point-to-point send/recv (it
  pipelines rather than parallelises a single sequence). ``affine_time_split_forward``
  parallelises it: the recurrence is affine in its start state, so each rank first
  computes its segment's map S_end = M S_start + B (two ordinary forward passes: from
  h0 = I with v = 0, and from h0 = 0), one all-gather shares the maps, each rank chains
  the maps of the ranks before it to get its true start state, and all ranks replay
  their segments at once.

Nothing here computes any part of the method: ``fwd`` is the caller's forward function
(``chunk_fwd`` on a GPU).
"""
from __future__ import annotations

from typing import Callable, List, Sequence, Tuple


def partition_sequences(lengths: Sequence[int], world: int) -> List[Tuple[int, int]]:
    """Contiguous sequence ranges ``[begin, end)``, one per rank, with token counts as
    even as a greedy sweep allows. Every sequence belongs to exactly one rank; a rank
    may receive an empty range when there are fewer sequences than ranks."""
    if world <= 0:
        raise ValueError("world must be positive")
    n = len(lengths)
    total = sum(int(x) for x in lengths)
    bounds = [0]
    acc = 0
    for r in range(1, world):
        target = total * r / world
        i = bounds[-1]
        while i < n and acc + lengths[i] <= target:
            acc += int(lengths[i])
            i += 1
        # take one more sequence when that lands closer to the target
        if i < n and (target - acc) > (acc + lengths[i] - target):
            acc += int(lengths[i])
            i += 1
        bounds.append(max(i, bounds[-1]))
    bounds.append(n)
    return [(bounds[r], bounds[r + 1]) for r in range(world)]


def partition_heads(n_heads: int, world: int) -> List[Tuple[int, int]]:
    """Even contiguous head ranges ``[begin, end)``, one per rank."""
    if world <= 0:
        raise ValueError("world must be positive")
    base, extra = divmod(n_heads, world)
    out, h = [], 0
    for r in range(world):
        k = base + (1 if r < extra else 0)
        out.append((h, h + k))
        h += k
    return out


def segment_bounds(length: int, world: int, multiple: int = 16) -> List[Tuple[int, int]]:
    """Split ``length`` tokens into ``world`` segments whose cut points are multiples of
    ``multiple`` (the chunk size), so every segment but the last is whole chunks."""
    cuts = [0]
    for r in range(1, world):
        c = (length * r // world) // multiple * multiple
        cuts.append(min(max(c, cuts[-1]), length))
    cuts.append(length)
    return [(cuts[r], cuts[r + 1]) for r in range(world)]


def time_split_forward(fwd: Callable, segment_inputs: dict, h0, rank: int, world: int,
                       group=None):
    """Run this rank's segment of one sequence with the state hand-off.

    ``segment_inputs`` holds this rank's tokens (keys q, k, v, gate_logits, beta and
    cu_seqlens for the segment). Rank 0 starts from ``h0`` (or zeros when None is
    given and ``fwd`` accepts it); rank r > 0 first receives its start state from rank
    r - 1. After the forward pass the rank sends its final state to rank r + 1.
    Returns ``(out, h_final)`` of the segment. ``fwd(q, k, v, gate_logits, beta, h0,
    cu_seqlens)`` must return ``(out, h_final)`` as tensors.
    """
    import torch.distributed as dist
    if rank > 0:
        if h0 is None:
            raise ValueError("ranks after the first need a receive buffer in h0")
        dist.recv(h0, src=rank - 1, group=group)
    out, h_final = fwd(segment_inputs["q"], segment_inputs["k"], segment_inputs["v"],
                       segment_inputs["gate_logits"], segment_inputs["beta"], h0,
                       segment_inputs["cu_seqlens"])
    if rank < world - 1:
        dist.send(h_final.contiguous(), dst=rank + 1, group=group)
    return out, h_final


def affine_time_split_forward(fwd: Callable, combine: Callable, segment_inputs: dict, h0,
                              rank: int, world: int, group=None):
    """This rank's segment of one sequence, all ranks in parallel (see the module note).

    ``segment_inputs`` is as for ``time_split_forward``; ``h0`` is the sequence's start
    state ([1, H, d_k, d_v], or None for zeros) -- rank 0's copy is broadcast. ``fwd`` is
    the forward function (``fwd(q, k, v, gate_logits, beta, h0, cu_seqlens) -> (out,
    h_final)``), ``combine(M, S, B)`` returns M S + B per head (``affine_combine`` on a
    GPU). Returns ``(out, h_final)`` of the segment; the last rank's ``h_final`` is the
    sequence's.
    """
    import torch
    import torch.distributed as dist
    q, v = segment_inputs["q"], segment_inputs["v"]
    H, dk, dv = q.shape[1], q.shape[2], v.shape[2]
    cu = segment_inputs["cu_seqlens"]
    args = (segment_inputs["k"], segment_inputs["gate_logits"], segment_inputs["beta"])
    sdt = torch.float32 if h0 is None else h0.dtype
    zero = torch.zeros((1, H, dk, dv), dtype=sdt, device=q.device)
    start = zero.clone() if h0 is None else h0.clone()
    dist.broadcast(start, src=0, group=group)
    # this segment's affine map
    eye = torch.eye(dk, dtype=sdt, device=q.device).expand(1, H, dk, dk).contiguous()
    v0 = torch.zeros((q.shape[0], H, dk), dtype=v.dtype, device=q.device)
    _, M = fwd(q, args[0], v0, args[1], args[2], eye, cu)
    _, B = fwd(q, args[0], v, args[1], args[2], zero, cu)
    Ms = [torch.empty_like(M) for _ in range(world)]
    Bs = [torch.empty_like(B) for _ in range(world)]
    dist.all_gather(Ms, M.contiguous(), group=group)
    dist.all_gather(Bs, B.contiguous(), group=group)
    # exclusive scan of the maps of the ranks before this one
    for r in range(rank):
        start = combine(Ms[r][0], start[0], Bs[r][0]).unsqueeze(0)
    return fwd(q, args[0], v, args[1], args[2], start.contiguous(), cu)
