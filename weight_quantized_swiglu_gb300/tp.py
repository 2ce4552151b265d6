"""Host side of the tensor-parallel shard over the intermediate dimension.

vllm.cpp issue "tp>1 fp8w tail-MLP shard host-dequantizes every layer",
"Proposed fix": rank r of n keeps gate/up rows [r I/n, (r+1) I/n) and the same
columns of down; each rank's down projection is then a partial sum over its
slice, and one exchange gives the layer's output. Here the exchange is an
all-gather of every rank's fp32 [M, K] partial into a rank-major
[n, M, K] buffer followed by ``QuantMLP.combine`` (qmlp_shard_combine), which
adds the partials in rank order on the device: the same bytes on every rank,
where a ring all-reduce would add in an order that depends on the topology.

This module holds only the rank arithmetic and the collective call; the
partials, the sum and the rounding are computed by the library's kernels.
"""
from __future__ import annotations


def shard_range(I: int, rank: int, nranks: int) -> tuple[int, int]:
    """Intermediate rows [i0, i1) of rank `rank` (I % nranks == 0 and the
    slice a multiple of 16, as qmlp_create_shard requires)."""
    if nranks < 1 or not 0 <= rank < nranks:
        raise ValueError(f"rank {rank} of {nranks}")
    if I % nranks or (I // nranks) % 16:
        raise ValueError(f"I={I} does not split into {nranks} slices of a multiple of 16")
    s = I // nranks
    return rank * s, (rank + 1) * s


def gather_partials(partial, out=None, group=None):
    """All-gather this rank's partial [M, K] into a rank-major [n, M, K]
    tensor (every rank gets every partial; slot r holds rank r's). Works on
    NCCL (device tensors) and gloo (host tensors)."""
    import torch
    import torch.distributed as dist
    n = dist.get_world_size(group)
    if out is None:
        out = torch.empty((n,) + tuple(partial.shape), dtype=partial.dtype, device=partial.device)
    dist.all_gather(list(out.unbind(0)), partial.contiguous(), group=group)
    return out
