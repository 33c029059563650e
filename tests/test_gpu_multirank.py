"""Two logical ranks on one GPU running the sharded, globally clipped step end to end.

Each rank is its own process on cuda:0 with a contiguous shard of one bucket: it
analyses and merges its shard's gradient in the library's kernels, reads its 12-byte
report, exchanges (sum of squares, non-finite count) with the other rank over gloo
(`sharded.global_clip_decision`), and updates its shard with the global decision.  The
ranks' kernels never wait on one another: the only exchange is on the host.  The union
of the shards must match the oracle run on the whole bucket, and every rank must take
the same decision.
"""

import json
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

from conftest import ROOT

pytestmark = pytest.mark.gpu


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, n, out_dir):
    import sys
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import torch
    import torch.distributed as dist
    import amsgrad_optimizer_step_gb300 as fa
    from amsgrad_optimizer_step_gb300 import sharded
    from synthetic.configs import CONFIG5

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w = CONFIG5.scaled(n, calls=4, inf_call=3)
    lo, hi = sharded.shard_range(n, rank, world)
    k = hi - lo
    idx = np.arange(lo, hi)
    p = torch.from_numpy(w.params_host(idx)).to(dev)
    m, v = torch.zeros_like(p), torch.zeros_like(p)
    rows = fa.fa_stats_rows(k, w.row_len)
    rows_buf, scratch, report = (fa.stats_buffer(rows, dev), fa.scratch_buffer(rows, dev),
                                 fa.stats_buffer(1, dev))
    opts = fa.options(**w.options())
    t = 0
    decisions = []
    for call in range(1, w.calls + 1):
        bits = w.grad_host(call, idx)
        g = torch.from_numpy(bits.view(np.int16)).to(dev).view(torch.bfloat16)
        fa.fa_analyze_gradient(g, w.row_len, rows_buf)
        fa.fa_merge_gradient_stats(rows_buf, rows, scratch, report)
        skip, norm, coef = sharded.global_clip_decision(fa.fa_read_report(report),
                                                        w.gradient_scale, w.max_grad_norm)
        if not skip:
            t, _ = fa.fa_bucket_step(None, p, g, m, v, None, t, opts,
                                     fa.control(w.gradient_scale), coef)
        decisions.append([bool(skip), repr(norm), repr(coef)])
    torch.cuda.synchronize()
    np.savez(os.path.join(out_dir, f"rank{rank}.npz"), p=p.cpu().numpy(), m=m.cpu().numpy(),
             v=v.cpu().numpy(), lo=lo, hi=hi, t=t)
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump(decisions, f)
    dist.destroy_process_group()


def test_two_logical_ranks_match_the_oracle(tmp_path, oracle_lib):
    import oracle
    from amsgrad_optimizer_step_gb300 import build
    from synthetic.configs import CONFIG5
    build.build()
    n = 2_000_017
    world = 2
    mp.spawn(_rank, args=(world, _free_port(), n, str(tmp_path)), nprocs=world, join=True)

    w = CONFIG5.scaled(n, calls=4, inf_call=3)
    shards = [np.load(tmp_path / f"rank{r}.npz") for r in range(world)]
    decisions = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    assert decisions[0] == decisions[1], "the ranks decided differently"
    assert [d[0] for d in decisions[0]] == [False, False, True, False]
    assert shards[0]["hi"] == shards[1]["lo"] and shards[1]["hi"] == n
    assert all(int(s["t"]) == 3 for s in shards)

    idx = np.arange(n)
    ref = oracle.OracleAdamW(w.params_host(idx), w.options(), lib_=oracle_lib)
    for call in range(1, w.calls + 1):
        bits = w.grad_host(call, idx)
        s, c = oracle_lib.gradient_stats(bits, "bf16", w.gradient_scale)
        skip, norm, coef = oracle_lib.clip_decision(s, c, w.max_grad_norm)
        got = decisions[0][call - 1]
        assert got[0] == skip
        if not skip:
            assert abs(float(got[1]) - norm) <= 1e-5 * norm
        ref.step(bits, "bf16", w.gradient_scale, skip_update=skip, clip_coef=coef)
    from gpu_harness import gate
    for name, want in (("p", ref.p), ("m", ref.state.m), ("v", ref.state.v)):
        got = np.concatenate([sh[name] for sh in shards])
        gate(got, want, 1e-5, f"two ranks, {name}")


def _zero1_rank(rank, world, port, n, dtype, ams, inf, out_dir):
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
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    opts = fa.options(lr=2e-3, weight_decay=0.01, amsgrad=ams)
    step = sharded.Zero1Step(n, opts, tdt, dev, max_grad_norm=0.5, gradient_scale=2.0)
    p = torch.zeros(step.padded, device=dev)
    p[:n] = torch.from_numpy(Z.params(n)).to(dev)
    g = torch.empty(step.padded, dtype=tdt, device=dev)
    decisions = []
    for call in range(1, 5):
        at = inf[2] if inf is not None and inf[0] == call and inf[1] == rank else None
        bits = Z.rank_gradient(n, step.padded, rank, call, dtype, at)
        host = torch.from_numpy(bits) if dtype == "f32" else \
            torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)
        g.copy_(host)
        d = step.step(p, g)
        decisions.append([d["skipped"], d["nonfinite"], repr(d["grad_norm"]),
                          repr(d["clip_coef"])])
    torch.cuda.synchronize()
    np.savez(os.path.join(out_dir, f"z{rank}.npz"), p=p.cpu().numpy(),
             m=step.m[:step.k].cpu().numpy(), v=step.v[:step.k].cpu().numpy(),
             vmax=(step.vmax[:step.k].cpu().numpy() if ams else np.zeros(0)), t=step.t)
    with open(os.path.join(out_dir, f"z{rank}.json"), "w") as f:
        json.dump(decisions, f)
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world,n,dtype,ams,inf", [
    (2, 2_000_017, "bf16", False, None),
    (3, 3_000_001, "f32", True, (3, 2, 2_999_999)),  # uneven split; +Inf in rank 2's gradient
])
def test_zero1_step_logical_ranks_match_the_whole_bucket_oracle(tmp_path, oracle_lib, world, n,
                                                                dtype, ams, inf):
    """The ZeRO-1 data-parallel step with logical ranks sharing cuda:0 (gloo collectives
    staged through the host, so no kernel waits on another rank): reduce-scatter of the
    ranks' gradients, each shard analysed, merged and updated in the library's kernels,
    the 12-byte totals exchanged, the parameters all-gathered.  Every rank's full
    parameters and the shards' moments against the oracle over the whole bucket on the
    exact sum of the gradients with gradient_scale x world (the mean), the trajectory
    within 1e-5; the decisions identical on every rank and the norm within 1e-5 of the
    oracle's; a +Inf in one rank's gradient skips the step everywhere."""
    import oracle
    import zero1_inputs as Z
    from amsgrad_optimizer_step_gb300 import build
    from gpu_harness import gate
    build.build()
    mp.spawn(_zero1_rank, args=(world, _free_port(), n, dtype, ams, inf, str(tmp_path)),
             nprocs=world, join=True)
    res = [np.load(tmp_path / f"z{r}.npz") for r in range(world)]
    dec = [json.load(open(tmp_path / f"z{r}.json")) for r in range(world)]
    assert all(d == dec[0] for d in dec), "the ranks decided differently"
    opts = dict(lr=2e-3, beta1=0.9, beta2=0.999, eps=1e-5, weight_decay=0.01, amsgrad=ams,
                maximize=False)
    ref = oracle.OracleAdamW(Z.params(n).astype(np.float64), opts, storage="f32",
                             lib_=oracle_lib)
    for call in range(1, 5):
        bits = Z.reduced_gradient(n, world, call, dtype, inf)
        s, c = oracle_lib.gradient_stats(bits, dtype, 2.0 * world)
        skip, norm, coef = oracle_lib.clip_decision(s, c, 0.5)
        got = dec[0][call - 1]
        assert got[0] == skip and got[1] == c, (call, got, skip, c)
        if not skip:
            assert abs(float(got[2]) - norm) <= 1e-5 * norm
        ref.step(bits, dtype, 2.0 * world, skip_update=skip, clip_coef=coef)
    for r in res:
        assert int(r["t"]) == ref.state.t
        gate(r["p"][:n], ref.p, 1e-5, "gathered p")
        assert not r["p"][n:].any(), "padding written"
    gate(np.concatenate([r["m"] for r in res]), ref.state.m, 1e-5, "sharded m")
    gate(np.concatenate([r["v"] for r in res]), ref.state.v, 1e-5, "sharded v")
    if ams:
        gate(np.concatenate([r["vmax"] for r in res]), ref.state.vmax, 1e-5, "sharded vmax")


def test_bench_runs_the_zero1_step_with_two_ranks_on_one_gpu():
    """bench.py --gpus 2 under torchrun, the two ranks sharing cuda:0 with gloo
    collectives staged through the host: the ZeRO-1 step runs and rank 0 prints one
    JSON line for the whole job (both ranks' parameters counted), with the data-parallel
    configuration named and the step's kernel launches counted."""
    import subprocess
    import sys
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--gpus", "2", "--steps", "3", "--warmup", "3",
           "--params", "1048576", "--e2e-steps", "2", "--next-rows-steps", "0",
           "--no-cpu-baseline", "--dist-backend", "gloo"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, (r.stdout[-2000:], r.stderr[-3000:])
    lines = [x for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    line = json.loads(lines[0])
    assert line["n_gpus"] == 2 and line["value"] > 0 and line["scaling"] == "weak"
    assert line["config"]["parallelism"].startswith("dp2, ZeRO-1")
    # per step: one analysis, two merge levels (4096 rows), one update
    assert line["gpu_launches"] == 3 * 4
    assert line["e2e"]["h2d_bytes_per_step"] == 2 * 1048576 * 2


def _zero1_nccl_rank(rank, port, n, out_dir):
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
    os.environ["NCCL_NVLS_ENABLE"] = "0"
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    dist.init_process_group("nccl", rank=rank, world_size=1, device_id=dev)
    opts = fa.options(lr=2e-3, weight_decay=0.01, amsgrad=True)
    step = sharded.Zero1Step(n, opts, torch.bfloat16, dev, max_grad_norm=0.5, gradient_scale=2.0)
    assert step.nccl and step.distributed
    p = torch.zeros(step.padded, device=dev)
    p[:n] = torch.from_numpy(Z.params(n)).to(dev)
    g = torch.empty(step.padded, dtype=torch.bfloat16, device=dev)
    decisions = []
    for call in range(1, 4):
        bits = Z.rank_gradient(n, step.padded, 0, call, "bf16", 77 if call == 2 else None)
        g.copy_(torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16))
        d = step.step(p, g)
        decisions.append([d["skipped"], d["nonfinite"], repr(d["grad_norm"])])
    torch.cuda.synchronize()
    np.savez(os.path.join(out_dir, "nccl.npz"), p=p.cpu().numpy(), m=step.m.cpu().numpy(),
             v=step.v.cpu().numpy(), vmax=step.vmax.cpu().numpy(), t=step.t)
    with open(os.path.join(out_dir, "nccl.json"), "w") as f:
        json.dump(decisions, f)
    dist.destroy_process_group()


def test_zero1_step_on_a_one_rank_nccl_group_matches_the_oracle(tmp_path, oracle_lib):
    """The ZeRO-1 step's NCCL branch on the one GPU there is: a one-rank NCCL group, so
    reduce_scatter_tensor and the in-place all_gather_into_tensor run on the device buffers
    (moving data within the GPU).  Against the oracle over the whole bucket, with a +Inf
    in the second of three calls."""
    import oracle
    import zero1_inputs as Z
    from amsgrad_optimizer_step_gb300 import build
    from gpu_harness import gate
    build.build()
    n = 1_000_003
    mp.spawn(_zero1_nccl_rank, args=(_free_port(), n, str(tmp_path)), nprocs=1, join=True)
    res = np.load(tmp_path / "nccl.npz")
    dec = json.load(open(tmp_path / "nccl.json"))
    opts = dict(lr=2e-3, beta1=0.9, beta2=0.999, eps=1e-5, weight_decay=0.01, amsgrad=True,
                maximize=False)
    ref = oracle.OracleAdamW(Z.params(n).astype(np.float64), opts, storage="f32",
                             lib_=oracle_lib)
    inf = (2, 0, 77)
    for call in range(1, 4):
        bits = Z.reduced_gradient(n, 1, call, "bf16", inf)
        s, c = oracle_lib.gradient_stats(bits, "bf16", 2.0)
        skip, norm, coef = oracle_lib.clip_decision(s, c, 0.5)
        assert dec[call - 1][0] == skip and dec[call - 1][1] == c
        if not skip:
            assert abs(float(dec[call - 1][2]) - norm) <= 1e-5 * norm
        ref.step(bits, "bf16", 2.0, skip_update=skip, clip_coef=coef)
    assert int(res["t"]) == ref.state.t == 2
    gate(res["p"][:n], ref.p, 1e-5, "p")
    gate(res["m"][:n], ref.state.m, 1e-5, "m")
    gate(res["v"][:n], ref.state.v, 1e-5, "v")
    gate(res["vmax"][:n], ref.state.vmax, 1e-5, "vmax")


def test_bench_zero1_step_over_nccl_checks_its_own_parity():
    """bench.py --zero1 under torchrun with one rank over NCCL: the ZeRO-1 step's NCCL
    collectives on the device buffers, timed, and the bench's own oracle replay of the
    timed run must pass (parity.ok)."""
    import subprocess
    import sys
    env = dict(os.environ, NCCL_NVLS_ENABLE="0")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "1",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--gpus", "1", "--steps", "3", "--warmup", "3",
           "--params", "1048576", "--e2e-steps", "2", "--no-cpu-baseline", "--zero1"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=900, env=env)
    assert r.returncode == 0, (r.stdout[-2000:], r.stderr[-3000:])
    line = json.loads([x for x in r.stdout.splitlines() if x.startswith("{")][-1])
    assert line["config"]["parallelism"].startswith("dp1, ZeRO-1")
    assert line["parity"]["ok"] is True and line["parity"]["t"] == 6
    assert line["value"] > 0 and line["gpu_launches"] == 3 * 4
