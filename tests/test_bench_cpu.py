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
