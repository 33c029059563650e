"""The sharded statistics exchange on two CPU ranks (gloo, world_size 2).

Each rank holds a contiguous shard of one gradient, forms its own 12-byte
report (here from the oracle, since there is no GPU), and the ranks take the
skip / clip decision together through ``sharded.global_clip_decision``.  The
decision must equal the single-process decision over the whole gradient and be
bit-identical on every rank.
"""

import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

from conftest import ROOT


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, n, inf_at, out_dir):
    import sys
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import torch.distributed as dist
    import oracle
    from amsgrad_optimizer_step_gb300 import FaStats, sharded
    from synthetic.configs import CONFIG5

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = CONFIG5.scaled(n)
    lo, hi = sharded.shard_range(n, rank, world)
    bits = w.grad_host(1, np.arange(lo, hi))
    if inf_at is not None and lo <= inf_at < hi:
        bits[inf_at - lo] = 0x7F80  # +Inf in BF16
    s, c = oracle.lib().gradient_stats(bits, "bf16", 1.0)
    rep = FaStats()
    rep.sum_sq = np.float32(s)
    rep.sum_sq_lo = np.float32(s - float(np.float32(s)))
    rep.nonfinite = c
    skip, norm, coef = sharded.global_clip_decision(rep, 4.0, 0.5)
    np.save(os.path.join(out_dir, f"r{rank}.npy"), np.array([float(skip), norm, coef, lo, hi]))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("inf_at", [None, 700_001])
def test_two_rank_decision_matches_whole_gradient(tmp_path, inf_at):
    import oracle
    import amsgrad_optimizer_step_gb300 as fa
    from amsgrad_optimizer_step_gb300 import build
    from synthetic.configs import CONFIG5
    build.build()
    n = 1_000_003
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), n, inf_at, str(tmp_path)),
                       nprocs=world, join=True, start_method="spawn")
    res = [np.load(tmp_path / f"r{r}.npy") for r in range(world)]
    # shards tile [0, n) with 8-element aligned boundaries
    assert res[0][3] == 0 and res[0][4] == res[1][3] and res[1][4] == n
    assert int(res[0][4]) % 8 == 0
    # every rank took the bit-identical decision
    assert np.array_equal(res[0][:3], res[1][:3])
    # ... equal to the decision over the whole gradient
    bits = CONFIG5.scaled(n).grad_host(1, np.arange(n))
    if inf_at is not None:
        bits[inf_at] = 0x7F80
    s, c = oracle.lib().gradient_stats(bits, "bf16", 1.0)
    skip, norm, coef = fa.fa_clip_decision(s, c, 4.0, 0.5)
    assert bool(res[0][0]) == skip == (inf_at is not None)
    if not skip:
        assert abs(res[0][1] - norm) <= 1e-6 * norm
        assert abs(res[0][2] - coef) <= 1e-6 * coef


def test_shard_ranges_tile_the_bucket():
    from amsgrad_optimizer_step_gb300 import sharded
    for n in (0, 1, 7, 8, 9, 1000, 1_073_741_824, 1_195_991_040):
        for world in (1, 2, 3, 4, 8):
            prev = 0
            for r in range(world):
                lo, hi = sharded.shard_range(n, r, world)
                assert lo == prev and hi >= lo
                assert lo % 8 == 0 or lo == n
                prev = hi
            assert prev == n


def _optim_worker(rank, world, port, out_dir):
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    from amsgrad_optimizer_step_gb300 import FaStats, fa_clip_decision
    from amsgrad_optimizer_step_gb300.optim import statistics_decision

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    rep = FaStats()
    rep.sum_sq = np.float32(3.0 + 5.0 * rank)  # rank 0: 3, rank 1: 8
    rep.sum_sq_lo = np.float32(0.0)
    rep.nonfinite = 0
    local = statistics_decision(rep, 2.0, 0.5)
    shards = statistics_decision(rep, 2.0, 0.5, shard_group=dist.group.WORLD)
    want_local = fa_clip_decision(3.0 + 5.0 * rank, 0, 2.0, 0.5)
    want_shards = fa_clip_decision(11.0, 0, 2.0, 0.5)
    np.save(os.path.join(out_dir, f"o{rank}.npy"),
            np.array([list(map(float, local)), list(map(float, shards)),
                      list(map(float, want_local)), list(map(float, want_shards))]))
    dist.barrier()
    dist.destroy_process_group()


def test_fused_adamw_sums_statistics_only_over_a_shard_group(tmp_path):
    """FusedAdamW's decision with torch.distributed initialised: replicas (no
    shard_group) decide from their own report, which already covers the whole reduced
    gradient; shards (shard_group set) sum the ranks' totals first."""
    from amsgrad_optimizer_step_gb300 import build
    build.build()
    world = 2
    mp.start_processes(_optim_worker, args=(world, _free_port(), str(tmp_path)),
                       nprocs=world, join=True, start_method="spawn")
    res = [np.load(tmp_path / f"o{r}.npy") for r in range(world)]
    for r in res:
        local, shards, want_local, want_shards = r
        assert np.array_equal(local, want_local)
        assert np.array_equal(shards, want_shards)
    # the sharded decision is the same on every rank; the local ones differ
    assert np.array_equal(res[0][1], res[1][1])
    assert not np.array_equal(res[0][0], res[1][0])
