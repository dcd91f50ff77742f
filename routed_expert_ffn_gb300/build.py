"""Build the CUDA library ``libmoe_gb300.so`` in-tree for sm_103a.

Each ``csrc/*.cu`` file is compiled by nvcc in parallel, then linked into one
shared library next to this file.  ``python -m routed_expert_ffn_gb300.build``
runs it from the command line.
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libmoe_gb300.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else (shutil.which("nvcc") or "nvcc")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _stale(obj: str, src: str) -> bool:
    if not os.path.exists(obj):
        return True
    # every header the sources include (csrc/*.cuh, include/*.h)
    inc = os.path.join(ROOT, "include")
    deps = [src] + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    deps += [os.path.join(inc, f) for f in os.listdir(inc) if f.endswith(".h")]
    t = os.path.getmtime(obj)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False,
          defines=None, lib_path: str = None) -> str:
    """Compile the library.  ``defines`` ({name: value}) override the kernels'
    compile-time parameters (``-D`` macros of the sources); such a variant is built in its own directory into
    ``lib_path``."""
    build_dir, lib = BUILD, LIB
    extra = []
    if defines:
        tag = "_".join(f"{k}{v}" for k, v in sorted(defines.items()))
        build_dir = os.path.join(BUILD, tag)
        lib = lib_path or os.path.join(build_dir, "libmoe_gb300.so")
        extra = [f"-D{k}={v}" for k, v in sorted(defines.items())]
    os.makedirs(build_dir, exist_ok=True)
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                    "-I", os.path.join(ROOT, "include"), "--expt-relaxed-constexpr"] + extra
    if ptxas_verbose:
        flags += ["-Xptxas", "-v"]
    jobs = []
    for src in sources():
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        if force or ptxas_verbose or _stale(obj, src):
            jobs.append([nvcc(), *flags, "-c", src, "-o", obj])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    failed = []
    if jobs:
        with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            for cmd, r in ex.map(run, jobs):
                if verbose or ptxas_verbose or r.returncode != 0:
                    sys.stderr.write(r.stdout + r.stderr)
                if r.returncode != 0:
                    failed.append(os.path.basename(cmd[-3]))
    if failed:
        raise RuntimeError(f"nvcc failed for {failed}")
    objs = [os.path.join(build_dir, os.path.basename(s)[:-3] + ".o") for s in sources()]
    if force or jobs or not os.path.exists(lib):
        tmp = lib + f".tmp{os.getpid()}"
        cuda_lib = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "lib64")
        subprocess.check_call([nvcc(), *ARCH, "-shared", "-cudart", "shared", *objs, "-o", tmp,
                               "-Xlinker", f"-rpath,{cuda_lib}"])
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, ptxas_verbose="--ptxas-v" in sys.argv)
    print(LIB)
