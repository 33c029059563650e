"""Host logic for running the step on parameter shards, one rank per GPU.

The update is independent per element, so a bucket can be split into
contiguous shards, one per rank, with no data exchange in the update itself.
The skip and the global-norm clip are defined over the WHOLE gradient
("训练与状态保存", section "在 ruda:0 上进行原生 PyTorch 训练": global L2 clipping over
all active parameter groups, any non-finite value skips the step).  Each rank
reads back its own 12-byte report; the ranks exchange (sum of squares,
non-finite count) and every rank sums them in rank order, so that all ranks
take a bit-identical decision.

``Zero1Step`` is the whole data-parallel step around that exchange, with the
optimizer state sharded (ZeRO stage 1): every rank holds the replicated FP32
parameters and its own full gradient (its share of the batch); rank r owns the
moments of shard r only.  Per step: a reduce-scatter of the flat gradient
(each rank receives the sum over ranks of its shard; the mean is the
gradient_scale times the world size, so averaging costs no extra pass), the
analysis and merge of that shard, the 12-byte exchange and decision, the fused
update of the shard, and an all-gather of the updated parameter shards
("ruCCL 用户指南", section "6. 集合通信训练": gradients are reduced with Mean before
the optimizer step; section "7. 显式 rank 张量集合通信": reduce-scatter and all-gather
in rank order).  NCCL runs the collectives on the device buffers; gloo, which
takes host tensors, stages them through the host (used by tests whose ranks
share one GPU).
"""

from __future__ import annotations

from typing import Optional

import torch

from . import FaStats, fa_clip_decision, fa_stats_sum_sq


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
    return fa_stats_sum_sq(rep), int(rep.nonfinite)


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


def zero1_shard_len(n: int, world: int, align: int = 8) -> int:
    """Elements per shard: ceil(n / world) rounded up to ``align`` (16 bytes of FP32),
    so that every shard starts 16-byte aligned; the flat buffers hold world times
    that (the tail past n is padding, never analysed or updated)."""
    if world < 1 or n < 0:
        raise ValueError("bad n/world")
    per = (n + world - 1) // world
    return (per + align - 1) // align * align


class Zero1Step:
    """The sharded data-parallel step over one flat bucket (see the module text).

    ``p`` (FP32) and ``g`` (FP32/FP16/BF16) are the caller's flat device buffers of
    ``padded`` elements; the first ``n`` are the bucket.  The rank's moments (and
    AMSGrad maximum) for its shard are allocated here.  ``shard_ops`` replaces the
    per-shard statistics and update (an object with ``stats(g_shard) -> (sum of
    squares of the stored values, non-finite count)`` and ``update(p_shard, g_shard,
    m, v, vmax, t, coef, scale, opts)``, t the completed step count); without it the
    library's kernels run them.
    """

    def __init__(self, n: int, opts, grad_dtype: torch.dtype, device: torch.device,
                 row_len: int = 256, max_grad_norm: float = 0.0, gradient_scale: float = 1.0,
                 mean: bool = True, group=None, shard_ops=None):
        import torch.distributed as dist
        self.distributed = dist.is_available() and dist.is_initialized()
        self.world = dist.get_world_size(group) if self.distributed else 1
        self.rank = dist.get_rank(group) if self.distributed else 0
        self.group = group
        self.nccl = self.distributed and dist.get_backend(group) == "nccl"
        self.n = n
        self.shard = zero1_shard_len(n, self.world)
        self.padded = self.shard * self.world
        self.lo = min(self.rank * self.shard, n)
        self.hi = min(self.lo + self.shard, n)
        self.k = self.hi - self.lo  # elements of the bucket in this rank's shard
        self.opts = opts
        self.device = device
        self.row_len = row_len
        self.max_grad_norm = max_grad_norm
        # the reduced gradient is a sum over ranks: its mean divides by the world size too
        self.scale = gradient_scale * (self.world if mean else 1)
        self.t = 0
        self.ops = shard_ops or _LibraryShardOps(self.k, row_len, device)
        self.g_shard = torch.empty(self.shard, dtype=grad_dtype, device=device)
        self.m = torch.zeros(self.shard, dtype=torch.float32, device=device)
        self.v = torch.zeros(self.shard, dtype=torch.float32, device=device)
        self.vmax = (torch.zeros(self.shard, dtype=torch.float32, device=device)
                     if opts.amsgrad else None)

    def _reduce_scatter(self, g: torch.Tensor) -> None:
        import torch.distributed as dist
        if not self.distributed:
            self.g_shard.copy_(g[:self.shard])
        elif self.nccl:
            dist.reduce_scatter_tensor(self.g_shard, g, op=dist.ReduceOp.SUM, group=self.group)
        else:
            out = torch.empty(self.shard, dtype=g.dtype)
            dist.reduce_scatter_tensor(out, g.cpu(), op=dist.ReduceOp.SUM, group=self.group)
            self.g_shard.copy_(out)

    def _all_gather(self, p: torch.Tensor) -> None:
        import torch.distributed as dist
        mine = p[self.rank * self.shard:(self.rank + 1) * self.shard]
        if not self.distributed:
            return
        if self.nccl:  # in place: each rank's input is its own slice of the output
            dist.all_gather_into_tensor(p, mine, group=self.group)
        else:
            full = torch.empty(self.padded, dtype=p.dtype)
            dist.all_gather_into_tensor(full, mine.cpu(), group=self.group)
            p.copy_(full)

    def step(self, p: torch.Tensor, g: torch.Tensor, events=None) -> dict:
        """One step.  Returns the decision: skipped, nonfinite, grad_norm, clip_coef.

        ``events`` (optional, three CUDA events) are recorded on the current stream after
        the reduce-scatter and the statistics, right before the update and right after
        it, for timing the phases."""
        if p.numel() != self.padded or g.numel() != self.padded:
            raise ValueError(f"p and g must hold {self.padded} elements (padded bucket)")
        self._reduce_scatter(g)
        s, c = self.ops.stats(self.g_shard[:self.k]) if self.k else (0.0, 0)
        if events:
            events[0].record()
        s, c = gather_totals(s, c, group=self.group,
                             device=self.device if self.nccl else torch.device("cpu"))
        skip, norm, coef = fa_clip_decision(s, c, self.scale, self.max_grad_norm)
        if events:
            events[1].record()
        if not skip and self.k:
            self.ops.update(p[self.lo:self.hi], self.g_shard[:self.k], self.m[:self.k],
                            self.v[:self.k], None if self.vmax is None else self.vmax[:self.k],
                            self.t, coef, self.scale, self.opts)
        if events:
            events[2].record()
        if not skip:
            self.t += 1
            self._all_gather(p)
        return {"skipped": bool(skip), "nonfinite": int(c), "grad_norm": norm, "clip_coef": coef}


class _LibraryShardOps:
    """The shard's statistics and update in the library's kernels."""

    def __init__(self, k: int, row_len: int, device: torch.device):
        from . import fa_stats_rows, scratch_buffer, stats_buffer
        self.rows = fa_stats_rows(k, row_len) if k else 0
        self.row_len = row_len
        if k:
            self.rows_buf = stats_buffer(self.rows, device)
            self.scratch = scratch_buffer(self.rows, device)
            self.report = stats_buffer(1, device)

    def stats(self, g_shard: torch.Tensor) -> tuple[float, int]:
        from . import fa_analyze_gradient, fa_merge_gradient_stats, fa_read_report
        fa_analyze_gradient(g_shard, self.row_len, self.rows_buf)
        fa_merge_gradient_stats(self.rows_buf, self.rows, self.scratch, self.report)
        return report_totals(fa_read_report(self.report))

    def update(self, p, g, m, v, vmax, t, coef, scale, opts) -> None:
        from . import control, fa_bucket_step
        fa_bucket_step(None, p, g, m, v, vmax, t, opts, control(scale), coef)
