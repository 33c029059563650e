"""The C ABI used from plain C, with no Python binding in between.

`tests/c_consumer/consumer.c` includes only `include/fused_adamw.h` and the CUDA
runtime, allocates its own device buffers and runs three statistics-guarded steps
(the second with a +Inf, so skipped).  On the CPU the header and the program must
compile as strict C; on the GPU the program is built, linked against the library and
run, and its output is compared with the oracle.  Run again with the update decided on
the device (fa_bucket_step_clipped_gated), and composed from the separate calls (the
descriptor update fa_bucket_update deciding from the device report), it must write the
same bits.
"""

import os
import shutil
import struct
import subprocess

import numpy as np
import pytest

from conftest import ROOT

SRC = os.path.join(ROOT, "tests", "c_consumer", "consumer.c")
INCLUDE = os.path.join(ROOT, "include")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _gcc():
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    return gcc


def test_header_is_strict_c():
    r = subprocess.run([_gcc(), "-std=c99", "-pedantic", "-Wall", "-Wextra", "-Werror", "-x", "c",
                        "-fsyntax-only", "-I", INCLUDE, "-"],
                       input='#include "fused_adamw.h"\nint main(void) { return 0; }\n',
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_consumer_compiles_as_c11():
    if not os.path.exists(os.path.join(CUDA, "include", "cuda_runtime.h")):
        pytest.skip("CUDA headers not available")
    r = subprocess.run([_gcc(), "-std=c11", "-pedantic", "-Wall", "-Wextra", "-Werror",
                        "-fsyntax-only", "-I", INCLUDE, "-I", os.path.join(CUDA, "include"), SRC],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def _mix(x):
    x = x.astype(np.uint64)
    x ^= x >> np.uint64(16)
    x = (x * np.uint64(0x7FEB352D)) & np.uint64(0xFFFFFFFF)
    x ^= x >> np.uint64(15)
    x = (x * np.uint64(0x846CA68B)) & np.uint64(0xFFFFFFFF)
    x ^= x >> np.uint64(16)
    return x


def _sample(stream, n, scale):
    """The program's inputs, rebuilt bit for bit."""
    i = np.arange(n, dtype=np.uint64)
    u = (_mix(_mix(np.array([stream], dtype=np.uint64)) ^ i) >> np.uint64(16)).astype(np.int64)
    return ((u - 32768).astype(np.float32) / np.float32(32768.0)) * np.float32(scale)


@pytest.mark.gpu
def test_consumer_runs_and_matches_the_oracle(oracle_lib, tmp_path):
    import oracle
    from amsgrad_optimizer_step_gb300 import build
    lib_path = build.build()
    pkg = os.path.dirname(lib_path)
    n = 100_003
    exe = str(tmp_path / "consumer")
    r = subprocess.run([_gcc(), "-std=c11", "-O2", SRC, "-I", INCLUDE,
                        "-I", os.path.join(CUDA, "include"), "-L", pkg, "-lfused_adamw",
                        "-L", os.path.join(CUDA, "lib64"), "-lcudart",
                        f"-Wl,-rpath,{pkg}:{os.path.join(CUDA, 'lib64')}", "-o", exe],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = str(tmp_path / "out.bin")
    r = subprocess.run([exe, str(n), out], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    raw = open(out, "rb").read()
    out_gated = str(tmp_path / "out_gated.bin")
    r = subprocess.run([exe, str(n), out_gated, "gated"], capture_output=True, text=True,
                       timeout=120)
    assert r.returncode == 0, r.stderr
    assert open(out_gated, "rb").read() == raw, "the device-decided steps wrote other bits"
    out_desc = str(tmp_path / "out_descriptor.bin")
    r = subprocess.run([exe, str(n), out_desc, "descriptor"], capture_output=True, text=True,
                       timeout=120)
    assert r.returncode == 0, r.stderr
    assert open(out_desc, "rb").read() == raw, "the steps composed from the separate calls differ"
    t = struct.unpack_from("<Q", raw, 0)[0]
    reps = [struct.unpack_from("<iiQdd", raw, 8 + 32 * k) for k in range(3)]
    arrays = np.frombuffer(raw, dtype=np.float32, offset=8 + 96).reshape(3, n)

    opts = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-5, weight_decay=1e-4, amsgrad=False,
                maximize=False)
    ref = oracle.OracleAdamW(_sample(1, n, 0.03125), opts, lib_=oracle_lib)
    for call in range(1, 4):
        g = _sample(100 + call, n, 0.0625)
        if call == 2:
            g[n // 2] = np.inf
        s, c = oracle_lib.gradient_stats(g, "f32", 4.0)
        skip, norm, coef = oracle_lib.clip_decision(s, c, 0.5)
        updated, skipped, nonfinite, dev_norm, dev_coef = reps[call - 1]
        assert (updated, skipped, nonfinite) == (int(not skip), int(skip), c)
        if not skip:
            assert abs(dev_norm - norm) <= 1e-5 * norm and abs(dev_coef - coef) <= 1e-5 * coef
            assert coef < 1.0
        ref.step(g, "f32", 4.0, skip_update=skip, clip_coef=coef)
    assert t == ref.state.t == 2
    from gpu_harness import gate
    for got, want, name in zip(arrays, (ref.p, ref.state.m, ref.state.v), "pmv"):
        gate(got, want, 1e-5, f"C consumer {name}")
