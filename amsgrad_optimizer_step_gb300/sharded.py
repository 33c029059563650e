"""Host logic for running the step on parameter shards, one rank per GPU.

The update is independent per element, so a bucket can be split into
contiguous shards, one per rank, with no data exchange in the update itself.
The only exchange is the gradient statistics: the skip and the global-norm
clip are defined over the WHOLE gradient ("训练与状态保存", section "在 ruda:0 上
进行原生 PyTorch 训练": global L2 clipping over all active parameter groups, any
non-finite value skips the step).  Each rank reads back its own 12-byte
report; the ranks exchange (sum of squares, non-finite count) and every rank
sums them in rank order, so that all ranks take a bit-identical decision.
"""

from __future__ import annotations

from typing import Optional

import torch

from . import FaStats, fa_clip_decision


def shard_range(n: int, rank: int, world: int, align: int = 8) -> tuple[int, int]:
    """Contiguous [start, end) of rank's shard; boundaries are multiples of ``align``
    elements so that every shard of an aligned buffer stays 16-byte aligned."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad rank/world")
    units = (n + align - 1) // align
    lo = units * rank // world
    hi = units * (rank + 1) // world
    return min(lo * align, n), min(hi * align, n)


def report_totals(rep: FaStats) -> tuple[float, int]:
    """(sum of squares of the stored gradient, non-finite count) of one report."""
    return float(rep.sum_sq) + float(rep.sum_sq_lo), int(rep.nonfinite)


def gather_totals(sum_sq: float, nonfinite: int, group=None,
                  device: Optional[torch.device] = None) -> tuple[float, int]:
    """All ranks' (sum, count), added in rank order.  Single process: unchanged."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return sum_sq, nonfinite
    world = dist.get_world_size(group)
    dev = device
    if dev is None:  # NCCL exchanges device tensors, gloo host tensors
        dev = (torch.device("cuda", torch.cuda.current_device())
               if dist.get_backend(group) == "nccl" else torch.device("cpu"))
    mine = torch.tensor([sum_sq, float(nonfinite)], dtype=torch.float64, device=dev)
    parts = [torch.empty_like(mine) for _ in range(world)]
    dist.all_gather(parts, mine, group=group)
    total_s = 0.0
    total_c = 0
    for part in parts:  # fixed rank order: identical on every rank
        s, c = part.tolist()
        total_s += s
        total_c += int(c)
    return total_s, total_c


def global_clip_decision(rep: FaStats, gradient_scale: float, max_grad_norm: float, group=None,
                         device: Optional[torch.device] = None) -> tuple[bool, float, float]:
    """(skip, global norm, clip coefficient) over every rank's shard."""
    s, c = report_totals(rep)
    s, c = gather_totals(s, c, group=group, device=device)
    return fa_clip_decision(s, c, gradient_scale, max_grad_norm)
