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


# The spill gate: ptxas reports, per kernel instance, the bytes it spills to local memory; a
# spill in a product instance fails the build.  The one exemption is the test-only recording
# variant (mode 1 of the mat-vec kernels: qmd_debug_qmatvec_dump), which stores every integer
# dot it computes and is never on a timed path.  Template argument (0-based) that holds the mode:
_MODE_ARG = {"qmv_kernel": 3, "qmv_tc_kernel": 1, "qmv_rl_kernel": 2}
_RECORDING_MODE = 1


def spills(log_text: str) -> list[tuple[str, int, int]]:
    """(mangled kernel name, spill store bytes, spill load bytes) for every entry function of a
    ptxas -v log that spills."""
    import re
    out, cur = [], None
    for line in log_text.splitlines():
        m = re.search(r"Compiling entry function '(\S+)'", line)
        if m:
            cur = m.group(1)
            continue
        m = re.search(r"(\d+) bytes spill stores, (\d+) bytes spill loads", line)
        if m and cur and (int(m.group(1)) or int(m.group(2))):
            out.append((cur, int(m.group(1)), int(m.group(2))))
    return out


def spill_exempt(mangled: str) -> bool:
    """True for the recording variant of a mat-vec kernel, read from the mangled template
    arguments (Itanium ABI: L<i|b><value>E in order)."""
    import re
    for kern, pos in _MODE_ARG.items():
        m = re.search(r"\d+" + kern + r"I((?:L[ib]\d+E)+)E", mangled)
        if m:
            args = [int(v) for v in re.findall(r"L[ib](\d+)E", m.group(1))]
            return len(args) > pos and args[pos] == _RECORDING_MODE
    return False


def check_spills(build_dir: str) -> None:
    """Raise if any product kernel instance in the build's ptxas logs spills."""
    bad = []
    for u in UNITS:
        path = os.path.join(build_dir, u + ".log")
        if os.path.exists(path):
            with open(path) as f:
                bad += [(u,) + s for s in spills(f.read()) if not spill_exempt(s[0])]
    if bad:
        raise RuntimeError("register spills in product kernel instances: " +
                           "; ".join(f"{u}: {k} ({st} B stored, {ld} B loaded)" for u, k, st, ld in bad))


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
    check_spills(build_dir)
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
