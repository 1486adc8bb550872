"""Build libdecode_attn.so in-tree with nvcc (sm_103a only).

Each .cu file under csrc/ is compiled in parallel into csrc/../_build/*.o
and linked into decode_attention_kv_split_gb300/libdecode_attn.so.  Objects
are rebuilt when their source or any header is newer.  Run as
``python -m decode_attention_kv_split_gb300.build``.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libdecode_attn.so")
INCLUDE = os.path.join(ROOT, "include")
# The same sources built with DA_TEST_HOOKS (short wait limits, a switch that
# makes one producer withhold a stage) and DA_BOUNDS_CHECK (every global
# index the kernels compute checked against its buffer; a bad one is skipped
# and reported as DA_DEVERR_BOUNDS).  Only the tests load it.
BUILD_TEST = os.path.join(PKG, "_build_test")
LIB_TEST = os.path.join(PKG, "libdecode_attn_test.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-I", INCLUDE]


def _nvcc() -> str:
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cand = os.path.join(cuda, "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _headers() -> list[str]:
    return glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h"))


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose: bool = False, ptxas_info: bool = False, test_hooks: bool = False) -> str:
    """Build the library (``test_hooks``: the test-only variant) and return its path."""
    build_dir, lib = (BUILD_TEST, LIB_TEST) if test_hooks else (BUILD, LIB)
    os.makedirs(build_dir, exist_ok=True)
    sources = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    headers = _headers()
    nvcc = _nvcc()
    jobs = []
    objects = []
    for src in sources:
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        objects.append(obj)
        if ptxas_info or _stale(obj, [src, *headers]):
            cmd = [nvcc, *ARCH, *NVCC_FLAGS, *(["-DDA_TEST_HOOKS", "-DDA_BOUNDS_CHECK"] if test_hooks else []), "-c",
                   src, "-o", obj]
            if ptxas_info:
                cmd.insert(1, "-Xptxas=-v")
            jobs.append(cmd)

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    failed = []
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
        for cmd, r in ex.map(run, jobs):
            if verbose or ptxas_info or r.returncode != 0:
                sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
            if r.returncode != 0:
                failed.append(cmd[-3])
    if failed:
        raise RuntimeError(f"nvcc failed for: {failed}")
    if jobs or _stale(lib, objects):
        tmp = lib + f".tmp{os.getpid()}"
        cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objects, "-lcudart_static", "-lrt", "-ldl",
               "-lpthread"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
            raise RuntimeError("link failed")
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, ptxas_info="--ptxas" in sys.argv))
