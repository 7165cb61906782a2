"""Build libconvrot.so (the sm_103a kernels and their C ABI) in-tree.

Each CUDA source is compiled in parallel with nvcc for sm_103a only, then the
objects are linked into ``int8_hadamard_rotated_gb300/_lib/libconvrot.so``.
The benchmark's own measurement kernels (a size-matched copy and a probe of
the legacy s8 tensor instruction) go into a separate small library,
``_lib/libconvrot_bench.so``, which the product never loads.
Rebuilds are skipped when the libraries are newer than every source.

    python -m int8_hadamard_rotated_gb300.build [--force] [--verbose]
"""
from __future__ import annotations

import argparse
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build", "libconvrot")
LIB_DIR = os.path.join(PKG, "_lib")
LIB_PATH = os.path.join(LIB_DIR, "libconvrot.so")
BENCH_LIB_PATH = os.path.join(LIB_DIR, "libconvrot_bench.so")

SOURCES = ["api.cu", "pack.cu", "gemm.cu", "gemm_w4.cu", "noalloc.cu", "host_pipeline.cu", "mlp.cu"]
BENCH_CSRC = os.path.join(PKG, "bench_csrc")
BENCH_SOURCES = ["copy_ceiling.cu", "mma_s8_probe.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
              "--expt-relaxed-constexpr", "-I" + INCLUDE]


def nvcc_path() -> str:
    cand = shutil.which("nvcc")
    if cand:
        return cand
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    p = os.path.join(home, "bin", "nvcc")
    if os.path.exists(p):
        return p
    raise RuntimeError("nvcc not found (set CUDA_HOME or put nvcc on PATH)")


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files += [os.path.join(BENCH_CSRC, f) for f in os.listdir(BENCH_CSRC)]
    files.append(os.path.join(INCLUDE, "convrot.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date() -> bool:
    if not (os.path.exists(LIB_PATH) and os.path.exists(BENCH_LIB_PATH)):
        return False
    t = min(os.path.getmtime(LIB_PATH), os.path.getmtime(BENCH_LIB_PATH))
    return all(os.path.getmtime(f) <= t for f in _deps())


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    """Compile the library if needed; returns its path. Raises on failure."""
    if not force and not ptxas_info and up_to_date():
        return LIB_PATH
    nvcc = nvcc_path()
    os.makedirs(BUILD_DIR, exist_ok=True)
    os.makedirs(LIB_DIR, exist_ok=True)

    def compile_one(job):
        src_dir, src = job
        obj = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, "-c", os.path.join(src_dir, src), "-o", obj]
        if ptxas_info:
            cmd += ["-Xptxas", "-v"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, obj, r

    jobs = [(CSRC, s) for s in SOURCES] + [(BENCH_CSRC, s) for s in BENCH_SOURCES]
    with ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        results = list(ex.map(compile_one, jobs))
    objs = {}
    for src, obj, r in results:
        if verbose or ptxas_info or r.returncode != 0:
            sys.stderr.write(f"== {src}\n{r.stdout}{r.stderr}")
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}")
        objs[src] = obj
    for path, srcs in ((LIB_PATH, SOURCES), (BENCH_LIB_PATH, BENCH_SOURCES)):
        tmp = path + ".tmp"
        cmd = [nvcc, *ARCH, "-shared", *[objs[s] for s in srcs], "-o", tmp]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            sys.stderr.write(r.stdout + r.stderr)
            raise RuntimeError(f"link of {os.path.basename(path)} failed")
        os.replace(tmp, path)
    return LIB_PATH


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--ptxas-info", action="store_true")
    a = ap.parse_args(argv)
    print(build(force=a.force, verbose=a.verbose, ptxas_info=a.ptxas_info))


if __name__ == "__main__":
    main()
