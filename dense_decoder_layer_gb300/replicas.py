"""Independent replicas across GPUs: the stack does not shard.

Every rank runs the whole stack on its own GPU over its own batch; nothing
is exchanged on the data path.  The only collective is the bookkeeping of
a measurement: the slowest rank's time and the sum of all ranks' tokens.
"""

from __future__ import annotations

import torch
import torch.distributed as dist


def aggregate(local_ms: float, local_tokens: int) -> tuple[float, float]:
    """(max time over ranks in ms, whole-job tokens per second)."""
    if dist.is_available() and dist.is_initialized():
        dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
        t = torch.tensor([local_ms], dtype=torch.float64, device=dev)
        n = torch.tensor([float(local_tokens)], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        dist.all_reduce(n, op=dist.ReduceOp.SUM)
        ms, tokens = float(t.item()), float(n.item())
    else:
        ms, tokens = float(local_ms), float(local_tokens)
    return ms, tokens / (ms / 1e3)


def barrier() -> None:
    if dist.is_available() and dist.is_initialized():
        dist.barrier()
