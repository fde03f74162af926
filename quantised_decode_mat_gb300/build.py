"""Build libqmd.so (the CUDA kernels + C ABI) in-tree for sm_103a.

    python -m quantised_decode_mat_gb300.build [--force] [-v] [--trace]

Each translation unit is compiled by its own nvcc process in parallel, then linked into
quantised_decode_mat_gb300/libqmd.so.  Objects go to quantised_decode_mat_gb300/_build/.

--trace builds the traced variant instead (libqmd_trace.so, objects in _build_trace/): the same
kernels compiled with -DQMD_TRACE, which adds per-CTA phase time stamps and the two entry points
of include/qmd_trace.h.  It is a measurement tool, never the product library.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libqmd.so")
BUILD_TRACE = os.path.join(HERE, "_build_trace")
LIB_TRACE = os.path.join(HERE, "libqmd_trace.so")
UNITS = ("api", "pack", "rmsnorm", "qmv_q4k", "qmv_q5k", "qmv_q6k", "bind", "alu")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xptxas", "-v"] + ARCH


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    if os.path.exists(cand):
        return cand
    import shutil
    found = shutil.which("nvcc")
    if not found:
        raise RuntimeError("nvcc not found")
    return os.path.realpath(found)


def _sources_mtime() -> float:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(HERE, "..", "include", "qmd.h"))
    files.append(os.path.join(HERE, "..", "include", "qmd_trace.h"))
    files.append(os.path.abspath(__file__))
    return max(os.path.getmtime(f) for f in files)


def build(force: bool = False, verbose: bool = False, trace: bool = False) -> str:
    lib_path, build_dir = (LIB_TRACE, BUILD_TRACE) if trace else (LIB, BUILD)
    if not force and os.path.exists(lib_path) and os.path.getmtime(lib_path) >= _sources_mtime():
        return lib_path
    os.makedirs(build_dir, exist_ok=True)
    nvcc = _nvcc()
    procs = []
    defines = ["-DQMD_TRACE"] if trace else []
    for u in UNITS:
        obj = os.path.join(build_dir, u + ".o")
        log = open(os.path.join(build_dir, u + ".log"), "w")
        cmd = [nvcc, *NVCC_FLAGS, *defines, "-c", os.path.join(CSRC, u + ".cu"), "-o", obj]
        procs.append((u, subprocess.Popen(cmd, stdout=log, stderr=subprocess.STDOUT), log))
    failed = []
    for u, p, log in procs:
        if p.wait() != 0:
            failed.append(u)
        log.close()
    if failed:
        for u in failed:
            sys.stderr.write(open(os.path.join(build_dir, u + ".log")).read())
        raise RuntimeError(f"nvcc failed for {failed}")
    tmp = lib_path + f".tmp{os.getpid()}"
    cuda_lib = os.path.join(os.path.dirname(os.path.dirname(nvcc)), "lib64")
    subprocess.run([nvcc, "-shared", "--cudart", "shared", *ARCH, "-o", tmp]
                   + [os.path.join(build_dir, u + ".o") for u in UNITS]
                   + ["-Xlinker", f"-rpath,{cuda_lib}"], check=True)
    os.replace(tmp, lib_path)
    if verbose:
        for u in UNITS:
            sys.stdout.write(open(os.path.join(build_dir, u + ".log")).read())
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, trace="--trace" in sys.argv))
