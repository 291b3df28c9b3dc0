"""Data-parallel split of the forward over ranks (one process per GPU).

Every (batch, head) of attention is independent: the forward parallelises
over batch, heads and query blocks with no exchange between them ("FlashAttention
V2", section 2; "Lecture 6 — FlashAttention-2", parallelising over the
sequence).  N ranks therefore split a global batch into contiguous shards of
batch rows; each rank runs the whole forward on its own shard and nothing on
the data path crosses GPUs.  Only the measured step time is combined: the
slowest rank sets it (maximum over ranks).
"""
from __future__ import annotations


def batch_range(global_batch: int, world: int, rank: int) -> tuple[int, int]:
    """Rows ``[start, stop)`` of a global batch owned by ``rank`` of
    ``world``: contiguous, as even as possible (the first ``global_batch %
    world`` ranks hold one more row)."""
    if world < 1 or not 0 <= rank < world or global_batch < 0:
        raise ValueError("bad shard request")
    base, extra = divmod(global_batch, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def max_over_ranks(values, device=None) -> list[float]:
    """Element-wise maximum of ``values`` over all ranks of the default
    process group (the values unchanged without one, or with one rank)."""
    import torch
    import torch.distributed as dist

    vals = [float(v) for v in values]
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return vals
    t = torch.tensor(vals, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]
