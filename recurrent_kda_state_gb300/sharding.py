"""Head-sharded layout of the KDA path over several GPUs (host bookkeeping).

Every (sequence, head) unit of the path is independent, so a tensor-parallel
serving engine ("One node, 2.8x more throughput" on the vLLM Kimi K3 page
runs the model at TP8) gives each rank a contiguous range of heads: the rank
keeps the pools, rings and packed token tensors of its own heads only and
calls the library on them unchanged, with H = the size of its range.  Nothing
is exchanged between ranks on the path; the all-reduce after the output
projection lies outside it.  This module holds only the partition and the
slicing around it, none of the method's arithmetic.
"""


def head_range(num_heads, world, rank):
    """[h0, h1) of the heads rank `rank` of `world` owns: contiguous, sizes
    differing by at most one (num_heads / world each when it divides)."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("rank %d of world %d" % (rank, world))
    base, extra = divmod(num_heads, world)
    h0 = rank * base + min(rank, extra)
    return h0, h0 + base + (1 if rank < extra else 0)


def shard_heads(x, h0, h1, axis=1):
    """The heads [h0, h1) of a packed tensor ([N][H][d] tokens or [N][H] beta,
    axis 1; [P][H][...] pools and rings, axis 1) as a contiguous copy, the
    layout the rank's own buffers have."""
    idx = [slice(None)] * x.ndim
    idx[axis] = slice(h0, h1)
    part = x[tuple(idx)]
    return part.contiguous() if hasattr(part, "contiguous") else part.copy()


def gather_heads(parts, axis=1):
    """Concatenate per-rank results along the head axis (rank order)."""
    first = parts[0]
    if hasattr(first, "contiguous"):
        import torch
        return torch.cat(list(parts), dim=axis)
    import numpy as np
    return np.concatenate(list(parts), axis=axis)
