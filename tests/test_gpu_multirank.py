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
