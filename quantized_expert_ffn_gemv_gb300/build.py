"""In-tree build of the package's native libraries.

- libmoe_synth.so: the seeded input generator (plain C, gcc).
- libmoe_gb300.so: the CUDA library behind include/moe.h (nvcc, sm_103a only).

Both land in quantized_expert_ffn_gemv_gb300/_build/ (git-ignored).  Sources are
recompiled when they are newer than the library.
"""
import glob
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT = os.path.join(PKG, "_build")
SYNTH_LIB = os.path.join(OUT, "libmoe_synth.so")
CUDA_LIB = os.path.join(OUT, "libmoe_gb300.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _stale(target, sources):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(s) > t for s in sources)


def build_synth(force=False):
    src = os.path.join(CSRC, "synth.c")
    os.makedirs(OUT, exist_ok=True)
    if force or _stale(SYNTH_LIB, [src]):
        tmp = SYNTH_LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=gnu11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
                        "-pthread", "-Wall", "-o", tmp, src, "-lm"], check=True)
        os.replace(tmp, SYNTH_LIB)
    return SYNTH_LIB


def cuda_sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def cuda_headers():
    return sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
                  + glob.glob(os.path.join(ROOT, "include", "*.h")))


def build_cuda(force=False, verbose=False):
    srcs = cuda_sources()
    if not srcs:
        raise RuntimeError("no CUDA sources")
    os.makedirs(OUT, exist_ok=True)
    deps = srcs + cuda_headers()
    if not force and not _stale(CUDA_LIB, deps):
        return CUDA_LIB
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
                    "-I", os.path.join(ROOT, "include"), "-I", CSRC, "--expt-relaxed-constexpr"]
    if verbose:
        flags += ["-Xptxas", "-v"]
    objs = []

    def compile_one(src):
        obj = os.path.join(OUT, os.path.basename(src) + f".{os.getpid()}.o")
        r = subprocess.run([NVCC] + flags + ["-c", src, "-o", obj], capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and r.stderr:
            sys.stderr.write(r.stderr)
        return obj

    objs = [os.path.join(OUT, os.path.basename(src) + f".{os.getpid()}.o") for src in srcs]
    tmp = CUDA_LIB + f".tmp{os.getpid()}"
    try:
        with ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
            list(ex.map(compile_one, srcs))
        r = subprocess.run([NVCC] + ARCH + ["-shared", "-o", tmp] + objs + ["-lpthread"], capture_output=True,
                           text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, CUDA_LIB)
    finally:  # no objects or partial library left behind, whether the build worked or not
        for f in objs + [tmp]:
            if os.path.exists(f):
                os.remove(f)
    return CUDA_LIB


def build_all(force=False, verbose=False):
    return build_synth(force), build_cuda(force, verbose)


if __name__ == "__main__":
    print(build_all(force="--force" in sys.argv, verbose="-v" in sys.argv))
