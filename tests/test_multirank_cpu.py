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


# ---- the sharded (ZeRO-1) data-parallel step -----------------------------------------

class _OracleShardOps:
    """Per-shard statistics and update from the oracle (no GPU here), so that the
    step's host logic -- padding, reduce-scatter, the exchange and decision, the
    step count, the all-gather -- runs on CPU ranks."""

    def __init__(self, dtype):
        import oracle
        self.lib = oracle.lib()
        self.dtype = dtype

    def _bits(self, g):
        return g.numpy() if self.dtype == "f32" else g.view(__import__("torch").int16).numpy().view(np.uint16)

    def stats(self, g_shard):
        return self.lib.gradient_stats(self._bits(g_shard), self.dtype, 1.0)

    def update(self, p, g, m, v, vmax, t, coef, scale, opts):
        import torch
        o = dict(lr=opts.lr, beta1=opts.beta1, beta2=opts.beta2, eps=opts.eps,
                 weight_decay=opts.weight_decay, amsgrad=bool(opts.amsgrad),
                 maximize=bool(opts.maximize))
        arrs = [x.double().numpy().copy() for x in (p, m, v)]
        vm = vmax.double().numpy().copy() if vmax is not None else np.zeros(p.numel())
        self.lib.update(self._bits(g), self.dtype, o, scale, coef, t + 1, t > 0, True, *arrs, vm)
        for dst, src in zip((p, m, v), arrs):
            dst.copy_(torch.from_numpy(src.astype(np.float32)))
        if vmax is not None:
            vmax.copy_(torch.from_numpy(vm.astype(np.float32)))


def _zero1_worker(rank, world, port, n, dtype, ams, inf, out_dir):
    import sys
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import torch
    import torch.distributed as dist
    import amsgrad_optimizer_step_gb300 as fa
    from amsgrad_optimizer_step_gb300 import sharded
    import zero1_inputs as Z

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    opts = fa.options(lr=2e-3, weight_decay=0.01, amsgrad=ams)
    step = sharded.Zero1Step(n, opts, tdt, torch.device("cpu"), max_grad_norm=0.5,
                             gradient_scale=2.0, shard_ops=_OracleShardOps(dtype))
    p = torch.zeros(step.padded)
    p[:n] = torch.from_numpy(Z.params(n))
    decisions = []
    for call in range(1, 5):
        at = inf[2] if inf is not None and inf[0] == call and inf[1] == rank else None
        bits = Z.rank_gradient(n, step.padded, rank, call, dtype, at)
        g = torch.from_numpy(bits) if dtype == "f32" else \
            torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)
        d = step.step(p, g)
        decisions.append([d["skipped"], d["nonfinite"], repr(d["grad_norm"]), repr(d["clip_coef"])])
    np.savez(os.path.join(out_dir, f"z{rank}.npz"), p=p.numpy(), m=step.m[:step.k].numpy(),
             v=step.v[:step.k].numpy(), lo=step.lo, hi=step.hi, t=step.t, shard=step.shard)
    import json
    with open(os.path.join(out_dir, f"z{rank}.json"), "w") as f:
        json.dump(decisions, f)
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world,n,dtype,ams,inf", [
    (2, 10_000, "f32", False, None),
    (3, 10_007, "bf16", True, (3, 1, 4321)),   # uneven split; +Inf in rank 1's gradient
    (3, 9, "f32", True, (2, 0, 0)),            # the third shard holds no element
])
def test_zero1_step_on_cpu_ranks_matches_the_whole_bucket_oracle(tmp_path, world, n, dtype,
                                                                 ams, inf):
    """The ZeRO-1 step on gloo CPU ranks: every rank ends with the same full parameters,
    equal to the oracle run over the whole bucket on the exact sum of the ranks'
    gradients with gradient_scale x world (the mean); the shards' moments tile the
    oracle's; a +Inf in one rank's gradient skips the step on every rank."""
    import json
    import oracle
    import zero1_inputs as Z
    mp.start_processes(_zero1_worker, args=(world, _free_port(), n, dtype, ams, inf,
                                            str(tmp_path)),
                       nprocs=world, join=True, start_method="spawn")
    res = [np.load(tmp_path / f"z{r}.npz") for r in range(world)]
    dec = [json.load(open(tmp_path / f"z{r}.json")) for r in range(world)]
    assert all(d == dec[0] for d in dec), "the ranks decided differently"
    lib = oracle.lib()
    opts = dict(lr=2e-3, beta1=0.9, beta2=0.999, eps=1e-5, weight_decay=0.01, amsgrad=ams,
                maximize=False)
    ref = oracle.OracleAdamW(Z.params(n).astype(np.float64), opts, storage="f32", lib_=lib)
    for call in range(1, 5):
        bits = Z.reduced_gradient(n, world, call, dtype, inf)
        s, c = lib.gradient_stats(bits, dtype, 2.0 * world)
        skip, norm, coef = lib.clip_decision(s, c, 0.5)
        got = dec[0][call - 1]
        assert got[0] == skip and got[1] == c
        if not skip:
            assert abs(float(got[2]) - norm) <= 1e-12 * norm
        ref.step(bits, dtype, 2.0 * world, skip_update=skip, clip_coef=coef)
    for r in res:
        assert int(r["t"]) == ref.state.t
        np.testing.assert_allclose(r["p"][:n], ref.p, rtol=1e-6, atol=1e-9)
        assert not r["p"][n:].any(), "padding written"
    m = np.concatenate([r["m"] for r in res])
    v = np.concatenate([r["v"] for r in res])
    np.testing.assert_allclose(m, ref.state.m, rtol=1e-6, atol=1e-12)
    np.testing.assert_allclose(v, ref.state.v, rtol=1e-6, atol=1e-15)
    assert [int(r["lo"]) for r in res] == [min(k * int(res[0]["shard"]), n) for k in range(world)]
