"""Expert parallelism over several processes (one GPU each): host-side
partition of the routed experts and the sum of the shards' outputs.

Each rank holds a contiguous range of the routed experts (a ``Layer`` built
with ``expert_begin`` and that range's expert weights) plus a replica of the
router; the shared expert lives on rank 0.  Every rank receives all T tokens,
routes them over all E experts and computes its shard's part of y (the
pairs whose expert it holds, weighted by their gates, and the shared expert
on rank 0).  One all-reduce (sum) of y completes the layer.  The pages run
their models on one device or place whole layers across devices ("Step-5
Preview GGUF", "Files and memory requirements"); this split of one layer is
the library's own.
"""


def expert_ranges(E, world):
    """Balanced contiguous ranges [(begin, count)] of E experts over `world`
    ranks: the first E % world ranks hold one expert more."""
    if world < 1 or E < world:
        raise ValueError(f"cannot split {E} experts over {world} ranks")
    q, r = divmod(E, world)
    out, b = [], 0
    for i in range(world):
        n = q + (1 if i < r else 0)
        out.append((b, n))
        b += n
    return out


def holds_shared(rank):
    """The shared expert lives on rank 0."""
    return rank == 0


def all_reduce_output(y, group=None):
    """Sums the shards' outputs y [T, H] over the process group, in place.
    bf16 outputs are summed in fp32 and rounded once."""
    import torch
    import torch.distributed as dist
    if y.dtype == torch.float32:
        dist.all_reduce(y, op=dist.ReduceOp.SUM, group=group)
        return y
    acc = y.float()
    dist.all_reduce(acc, op=dist.ReduceOp.SUM, group=group)
    y.copy_(acc)
    return y
