"""Data-parallel helpers for the NF4 LoRA linear layer.

The layer is row-independent in the tokens: Y, U, V and dX of a token depend
on that token alone, while the adapter gradients dA and dB are sums over the
tokens. A data-parallel step therefore gives each rank its own contiguous
slice of tokens and sums dA and dB over the ranks once per step; the frozen
NF4 weight is a read-only replica on every rank.
Sources: inquiringlines.com note on QLoRA (gradients flow into the adapters
only); serverroom.net "Fine-tuning an LLM on a GPU", data-parallel
fine-tuning (every GPU holds the model and a share of the batch).
"""
from __future__ import annotations


def token_shard(M_total: int, rank: int, world: int) -> tuple[int, int]:
    """[start, stop) of rank's tokens: contiguous, sizes differing by at most one."""
    if world < 1 or not 0 <= rank < world or M_total < 0:
        raise ValueError("bad shard request")
    base, extra = divmod(M_total, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def allreduce_adapter_grads(grads, group=None):
    """Sums each adapter gradient tensor (dA, dB, fp32) over the ranks of
    `group`, in place."""
    import torch.distributed as dist
    for g in grads:
        dist.all_reduce(g, op=dist.ReduceOp.SUM, group=group)
