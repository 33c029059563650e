"""The bench's host-side bookkeeping, without a GPU: the DRAM-traffic figure is taken
from the committed ncu summary only while the kernel source it was captured from is
unchanged, and the workload record names the configuration it times."""

import os
import shutil

import bench


def test_traffic_is_scaled_from_the_committed_capture():
    n = 1 << 30
    t = bench.update_kernel_traffic(n)
    assert t is not None, "the committed capture no longer matches the kernel source"
    # 14 B read + ~11.8 B written per parameter: within the algorithmic 26 B/param
    assert 25.5 * n <= t <= 26.0 * n


def test_traffic_is_void_once_the_kernel_changes(tmp_path, monkeypatch):
    root = tmp_path / "repo"
    csrc = root / "amsgrad_optimizer_step_gb300" / "csrc"
    os.makedirs(csrc)
    os.makedirs(root / "profiles")
    src = os.path.join(bench.ROOT, "amsgrad_optimizer_step_gb300", "csrc")
    for f in ("update_kernels.cu", "internal.h"):
        shutil.copy(os.path.join(src, f), csrc / f)
    shutil.copy(os.path.join(bench.ROOT, "profiles", "update_kernel_traffic_flat256M_bf16.txt"),
                root / "profiles")
    monkeypatch.setattr(bench, "ROOT", str(root))
    assert bench.update_kernel_traffic(1 << 28) is not None
    with open(csrc / "update_kernels.cu", "a") as f:
        f.write("\n// edited\n")
    assert bench.update_kernel_traffic(1 << 28) is None


def test_default_workload_is_the_1e9_bucket():
    w = bench.workload()
    cfg = bench.config_dict(w)
    assert cfg["workload"] == "flat1G_bf16_stats_clip" and cfg["params"] == 1_073_741_824
    assert cfg["grad_dtype"] == "bf16" and cfg["row_len"] == 256
    assert cfg["merge_fan_in"] == 1024 and cfg["max_grad_norm"] == 1.0


def test_reference_arm_prints_the_contract_line():
    """`bench.py --impl reference` times the oracle on the host cores and prints one JSON
    line with the arm's keys; it needs no GPU."""
    import json
    import subprocess
    import sys
    r = subprocess.run([sys.executable, os.path.join(bench.ROOT, "bench.py"), "--impl",
                        "reference", "--steps", "2", "--warmup", "1"],
                       capture_output=True, text=True, timeout=600, cwd=bench.ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "params/s" and line["value"] > 0
    assert line["config"]["workload"] == "flat1G_bf16_stats_clip"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"] == {"value": line["value"], "unit": "params/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert line["higher_is_better"] is True and line["steps"] == 2 and line["warmup"] == 1


def _oracle_snapshot(w, steps):
    """What a correct device run would leave at the sampled indices: the oracle's own
    trajectory (built here from the oracle, as a stand-in for the GPU's results)."""
    import numpy as np
    import oracle
    lib = oracle.lib()
    idx = bench.parity_indices(w.n, k=500)
    g_all = w.grad_host(1, np.arange(w.n))
    s, c = lib.gradient_stats(g_all, "bf16", w.gradient_scale)
    skip, norm, coef = lib.clip_decision(s, c, w.max_grad_norm)
    o = oracle.OracleAdamW(w.params_host(idx), w.options(), storage="f32", lib_=lib)
    for _ in range(steps):
        o.step(w.grad_host(1, idx), "bf16", w.gradient_scale, skip_update=skip, clip_coef=coef)
    return {"idx": idx, "p": o.p.astype(np.float32), "m": o.state.m.astype(np.float32),
            "v": o.state.v.astype(np.float32), "norm": norm, "nonfinite": c, "skipped": skip,
            "t": steps, "g_bits": g_all}


def test_bench_parity_check_passes_the_oracle_and_catches_errors():
    """The bench's end-of-run parity check: a snapshot equal to the oracle's trajectory
    passes; a parameter off by 1e-4, a moment off by 2e-5, a norm off by 1e-4 relative,
    a wrong count, a wrong step count or a gradient that differs from the generator
    each fail it."""
    import dataclasses
    w = bench.workload(256 * 40 + 3)
    w = dataclasses.replace(w, max_grad_norm=0.05)  # so the clip is active at this size
    snap = _oracle_snapshot(w, 4)
    good = bench.parity_check(w, snap, 4)
    assert good["ok"] and good["max_rel_err"] <= 1e-6 and good["elements"] == len(snap["idx"])
    assert good["norm_rel_err"] <= 1e-12
    bad_cases = [("p", lambda s: s["p"].__setitem__(3, s["p"][3] + 1e-4)),
                 ("m", lambda s: s["m"].__setitem__(-1, s["m"][-1] + 2e-5)),
                 ("norm", lambda s: s.__setitem__("norm", s["norm"] * (1 + 1e-4))),
                 ("nonfinite", lambda s: s.__setitem__("nonfinite", 1)),
                 ("t", lambda s: s.__setitem__("t", 3)),
                 ("g", lambda s: s["g_bits"].__setitem__(int(s["idx"][5]), 0x7f80))]
    for name, spoil in bad_cases:
        s = {k: (v.copy() if hasattr(v, "copy") else v) for k, v in snap.items()}
        spoil(s)
        assert not bench.parity_check(w, s, 4)["ok"], name


def _row_record(w, idx, t0, steps):
    """A next-row record as the bench builds it, with the device side played by the
    oracle itself: the state after t0 steps from the generator's parameters, and after
    t0 + steps."""
    import numpy as np
    import oracle
    lib = oracle.lib()
    gh = w.grad_host(1, idx)
    o = oracle.OracleAdamW(w.params_host(idx), w.options(), storage="f32", lib_=lib)

    def snap(t):
        st = o.state
        zero = np.zeros(len(idx), np.float32)
        out = {"p": o.p.copy(), "m": zero if st.m is None else st.m.copy(),
               "v": zero if st.v is None else st.v.copy(), "t": t}
        if w.amsgrad:
            out["vmax"] = zero if st.vmax is None else st.vmax.copy()
        return out

    for _ in range(t0):
        o.step(gh, w.grad_dtype, w.gradient_scale)
    before = snap(t0)
    for _ in range(steps):
        o.step(gh, w.grad_dtype, w.gradient_scale)
    return {"w": w, "idx": idx, "gdt": w.grad_dtype, "g_bits": gh.copy(),
            "p0_from_generator": t0 == 0, "before": before, "after": snap(t0 + steps)}


def test_bench_next_row_replay_passes_the_oracle_and_catches_errors():
    """The bench's next-row check (the in-place 124M row and the decoder bucket rows):
    a batch equal to the oracle's replay passes, from the first step and from a state
    mid-run, with AMSGrad and maximize; a parameter off by 1e-4, a moment or vmax off
    by 2e-5, a step count off by one, or a gradient other than the generator's fails."""
    import dataclasses
    import numpy as np
    from synthetic.configs import CONFIG3, CONFIG4_MAX
    w3 = CONFIG3.scaled(4099)
    w4 = dataclasses.replace(CONFIG4_MAX, segments=None).scaled(5003)
    for w, t0 in ((w3, 0), (w4, 3)):
        idx = np.unique(np.concatenate([np.arange(0, w.n, 7), [w.n - 1]])).astype(np.int64)
        rec = _row_record(w, idx, t0, 4)
        good = bench.row_parity_check(rec)
        assert good["ok"] and good["steps"] == 4 and good["max_rel_err"] <= 1e-7, good
        spoils = [("p", lambda r: r["after"]["p"].__setitem__(2, r["after"]["p"][2] + 1e-4)),
                  ("m", lambda r: r["after"]["m"].__setitem__(-1, r["after"]["m"][-1] + 2e-5)),
                  ("t", lambda r: r["after"].__setitem__("t", r["after"]["t"] - 1)),
                  ("g", lambda r: r["g_bits"].__setitem__(5, r["g_bits"][5] ^ 1))]
        if w.amsgrad:
            spoils.append(("vmax", lambda r: r["after"]["vmax"].__setitem__(
                0, r["after"]["vmax"][0] + 2e-5)))
        for name, spoil in spoils:
            r = {k: v for k, v in rec.items()}
            r["after"] = {k: (v.copy() if hasattr(v, "copy") else v) for k, v in rec["after"].items()}
            r["g_bits"] = rec["g_bits"].copy()
            spoil(r)
            assert not bench.row_parity_check(r)["ok"], (w.name, name)


def test_bench_next_row_replay_takes_per_segment_decisions():
    """The per-segment clipped rows: each sampled element replays with its own
    segment's coefficient, which the oracle decides from that segment's whole
    gradient.  A device state made with those coefficients passes; one made with a
    single global coefficient, or a gradient changed outside the sampled elements,
    fails."""
    import dataclasses
    import numpy as np
    import oracle
    from synthetic.configs import CONFIG4
    lib = oracle.lib()
    seg = np.array([0, 700, 700, 2500, 2501, 6000], np.int64)  # one empty, one of 1 element
    w = dataclasses.replace(CONFIG4, segments=None).scaled(int(seg[-1]))
    g_all = w.grad_host(1, np.arange(w.n))
    max_norm = 1e-3
    coefs = [lib.clip_decision(*lib.gradient_stats(g_all[a:b], "f16", 1.0), max_norm)[2]
             for a, b in zip(seg[:-1], seg[1:])]
    assert min(coefs) < 1.0
    idx = np.unique(np.concatenate([np.arange(0, w.n, 5), seg[1:-1], seg[1:-1] - 1]))
    idx = idx[idx < w.n].astype(np.int64)
    kseg = np.searchsorted(seg, idx, side="right") - 1

    def device_like(coef_of):
        p = np.empty(len(idx), np.float32)
        m, v, vm = p.copy(), p.copy(), p.copy()
        for k in np.unique(kseg):
            sel = np.flatnonzero(kseg == k)
            o = oracle.OracleAdamW(w.params_host(idx[sel]), w.options(), lib_=lib)
            for _ in range(3):
                o.step(w.grad_host(1, idx[sel]), "f16", clip_coef=coef_of(k))
            p[sel], m[sel], v[sel], vm[sel] = o.p, o.state.m, o.state.v, o.state.vmax
        return {"p": p, "m": m, "v": v, "vmax": vm, "t": 3}

    zero = np.zeros(len(idx), np.float32)
    before = {"p": w.params_host(idx), "m": zero, "v": zero, "vmax": zero, "t": 0}
    rec = {"w": w, "idx": idx, "gdt": "f16", "g_bits": g_all[idx].copy(),
           "p0_from_generator": True, "seg": seg, "max_grad_norm": max_norm,
           "g_full_bits": g_all, "before": before, "after": device_like(lambda k: coefs[k])}
    good = bench.row_parity_check(rec)
    assert good["ok"] and good["segments"] == 5 and good["max_rel_err"] <= 1e-7, good
    assert abs(good["min_clip_coef_oracle"] - min(coefs)) == 0
    bad = dict(rec, after=device_like(lambda k: min(coefs)))
    assert not bench.row_parity_check(bad)["ok"]
    off = np.setdiff1d(np.arange(w.n), idx)[3]
    g2 = g_all.copy()
    g2[off] = np.uint16(0x3C00)  # 1.0 in FP16: a larger norm for that segment
    assert not bench.row_parity_check(dict(rec, g_full_bits=g2))["ok"]
