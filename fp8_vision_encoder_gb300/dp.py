"""Data-parallel pieces of the path: spreading a packed batch's segments over
ranks, and the one exchange dynamic scaling needs.

Segments (images) and heads never interact in the attention, so each rank can
quantize and attend its own segments.  Only the amax is global: the pages keep
one amax per tensor per forward over the whole batch ("FP8 ViT Encoder
Attention", Usage: a 16-entry circular buffer of observed Q/K/V amax values),
so with dynamic scaling the ranks combine their local amax values with one
all-reduce(MAX) of four floats before the ring push; every ring then equals the
single-GPU ring of the whole batch.  Static scales need no collective.
"""

import torch

from . import amax_local, ring_push


def shard_segments(seqlens, world_size):
    """Assign segments to ranks, longest first by attention cost L^2, each to
    the rank with the least cost so far (ties: lower rank).  Returns one sorted
    list of segment indices per rank."""
    if world_size < 1:
        raise ValueError("world_size must be >= 1")
    load = [0] * world_size
    parts = [[] for _ in range(world_size)]
    order = sorted(range(len(seqlens)), key=lambda i: (-int(seqlens[i]) ** 2, i))
    for i in order:
        r = min(range(world_size), key=lambda x: (load[x], x))
        parts[r].append(i)
        load[r] += int(seqlens[i]) ** 2
    return [sorted(p) for p in parts]


def shard_cu_seqlens(seqlens, segments):
    """cu_seqlens (Python list) of a rank's segments packed back to back, and
    the (start, end) token ranges of those segments in the full batch."""
    starts = [0]
    for L in seqlens:
        starts.append(starts[-1] + int(L))
    cu, ranges = [0], []
    for i in segments:
        cu.append(cu[-1] + int(seqlens[i]))
        ranges.append((starts[i], starts[i + 1]))
    return cu, ranges


def allreduce_amax(vals, group=None):
    """In-place all-reduce(MAX) of a float32[4] (a_q, a_k, a_v, any_tokens)."""
    import torch.distributed as dist
    dist.all_reduce(vals, op=dist.ReduceOp.MAX, group=group)
    return vals


def amax_update_dp(state, q, k, v, cu_seqlens, group=None, stream=None, **kwargs):
    """Dynamic scaling over ranks: local amax, all-reduce(MAX), ring push.
    With one rank (or no process group) it equals amax_update."""
    vals = amax_local(state, q, k, v, cu_seqlens, stream=stream, **kwargs)
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1:
        s = torch.cuda.current_stream() if stream is None else stream
        with torch.cuda.stream(s):
            allreduce_amax(vals, group)
    ring_push(state, vals, stream=stream)
    return vals
