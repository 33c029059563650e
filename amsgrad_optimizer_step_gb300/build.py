"""Ahead-of-time build of ``libfused_adamw.so`` for sm_103a with nvcc.

Each translation unit compiles in parallel; the objects are linked into one
shared library next to this file, against the shared CUDA runtime (the same
``libcudart.so.13`` soname that PyTorch loads).
"""

from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_NAME = "libfused_adamw.so"
LIB_PATH = os.path.join(PKG, LIB_NAME)
BUILD_DIR = os.path.join(PKG, "_build")

# Build variants: the normal library, and the bounds-checked test variant whose
# kernels count and skip any access outside their arrays (-DFA_BOUNDS_CHECK=1).
VARIANTS = {
    "normal": (LIB_PATH, BUILD_DIR, []),
    "checked": (os.path.join(PKG, "libfused_adamw_checked.so"),
                os.path.join(PKG, "_build_checked"), ["-DFA_BOUNDS_CHECK=1"]),
}

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# Host code without floating-point contraction: the FP64 coefficient arithmetic then
# rounds the same on x86-64 and AArch64 (whose compilers may otherwise fuse 1 - lr*wd).
COMMON = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O2,-ffp-contract=off",
          "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC)
                  if f.endswith((".cu", ".cpp")))


def _deps() -> list[str]:
    hdrs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".h")]
    hdrs += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    return sources() + hdrs + [os.path.abspath(__file__)]


# ELF e_machine of a shared object built for this host (x86-64: 62, AArch64: 183).
_ELF_MACHINE = {"x86_64": 62, "amd64": 62, "aarch64": 183, "arm64": 183}


def _built_for_this_host(path: str) -> bool:
    """False for a library built for another architecture (e.g. copied from an x86
    host to an AArch64 one), which must be rebuilt rather than loaded."""
    import platform
    want = _ELF_MACHINE.get(platform.machine().lower())
    try:
        with open(path, "rb") as f:
            head = f.read(20)
    except OSError:
        return False
    if len(head) < 20 or head[:4] != b"\x7fELF":
        return False
    machine = int.from_bytes(head[18:20], "little" if head[5] == 1 else "big")
    return want is None or machine == want


def up_to_date(lib_path: str = LIB_PATH) -> bool:
    if not os.path.exists(lib_path) or not _built_for_this_host(lib_path):
        return False
    t = os.path.getmtime(lib_path)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False,
          variant: str = "normal") -> str:
    """Compile and link the library if any source is newer; returns its path."""
    lib_path, build_dir, defines = VARIANTS[variant]
    if not force and up_to_date(lib_path):
        return lib_path
    os.makedirs(build_dir, exist_ok=True)
    cc = nvcc()
    extra = (["-Xptxas", "-v"] if ptxas_info else []) + defines

    def compile_one(src: str) -> str:
        obj = os.path.join(build_dir, os.path.basename(src) + ".o")
        cmd = [cc, *ARCH, *COMMON, *extra, "-c", src, "-o", obj]
        if src.endswith(".cpp"):
            cmd[1:1] = ["-x", "cu"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose or ptxas_info:
            print(r.stdout + r.stderr)
        return obj

    with concurrent.futures.ThreadPoolExecutor(max_workers=8) as ex:
        objs = list(ex.map(compile_one, sources()))
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
           "-Xlinker", "-rpath,/usr/local/cuda/lib64"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv,
                variant="checked" if "--checked" in sys.argv else "normal"))
