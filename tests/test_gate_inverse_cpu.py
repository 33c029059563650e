"""The exact inverse behind the device-side decision's multiplications (no GPU).

The device decides skip and clip with the host's FP64 operations, but divides by a
power-of-two gradient scale by multiplying with its inverse, which the host computes
with ``power_of_two_inverse`` (csrc/internal.h).  That is bit-identical only if the
inverse is exact and IEEE arithmetic rounds x / s and x * (1 / s) to the same double.
This compiles the header's function with the host compiler and checks both: which
scales get an inverse, and, for every exponent of s and random x of every exponent
(subnormal and overflowing quotients included), that the two results have the same
bits.
"""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CXX = shutil.which("g++")

PROGRAM = r'''
#include "internal.h"
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <limits>

static uint64_t state = 0x2545F4914F6CDD1Dull;
static uint64_t next() {  // splitmix64
    uint64_t z = (state += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}
static uint64_t bits(double x) { uint64_t u; std::memcpy(&u, &x, 8); return u; }
static double from_bits(uint64_t u) { double x; std::memcpy(&x, &u, 8); return x; }

int main() {
    long bad = 0, checked = 0, with_inverse = 0;
    for (int k = -1074; k <= 1023; ++k) {
        const double s = std::ldexp(1.0, k);
        const double inv = fa::power_of_two_inverse(s);
        const bool expect = k >= -1022 && k <= 1022;
        if ((inv != 0.0) != expect) { std::printf("scale 2^%d: inverse %a\n", k, inv); ++bad; }
        if (inv == 0.0) continue;
        ++with_inverse;
        if (inv * s != 1.0) { std::printf("2^%d: inverse not exact\n", k); ++bad; }
        for (int i = 0; i < 400; ++i) {
            // any finite double: random sign, exponent and mantissa
            double x = from_bits(next() & 0xFFEFFFFFFFFFFFFFull);
            if (!std::isfinite(x)) continue;
            ++checked;
            if (bits(x / s) != bits(x * inv)) { std::printf("x=%a s=2^%d\n", x, k); ++bad; }
        }
    }
    const double others[] = {3.0, 0.1, 1000.0, 1.5, 0.0, -2.0, -0.5,
                             std::numeric_limits<double>::infinity(),
                             std::numeric_limits<double>::quiet_NaN(),
                             std::nextafter(1.0, 2.0), std::nextafter(2.0, 1.0)};
    for (double s : others)
        if (fa::power_of_two_inverse(s) != 0.0) { std::printf("scale %a got an inverse\n", s); ++bad; }
    std::printf("checked %ld with_inverse %ld bad %ld\n", checked, with_inverse, bad);
    return bad != 0;
}
'''


@pytest.mark.skipif(CXX is None, reason="needs g++")
def test_power_of_two_inverse_gives_the_division_bits(tmp_path):
    src = tmp_path / "inverse.cpp"
    src.write_text(PROGRAM)
    exe = tmp_path / "inverse"
    cuda_inc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")
    subprocess.run([CXX, "-std=c++17", "-O2", "-ffp-contract=off",
                    "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(ROOT, "amsgrad_optimizer_step_gb300", "csrc"),
                    "-I", cuda_inc, str(src), "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout[-3000:]
    last = r.stdout.strip().splitlines()[-1].split()
    assert int(last[1]) > 700_000 and int(last[3]) == 2045 and int(last[5]) == 0, r.stdout
