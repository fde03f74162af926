"""The split-K kernel's host-visible arithmetic, checked on the CPU from its own header
(tests/splitk/splitk_partition_check.cu, compiled by nvcc, no device code run): every row's groups
of four blocks split over the cluster's CTAs without gap or overlap, each group sum read from the
CTA that wrote it, the clusters' tile ranges covering every tile once within the size the plan
reserves, and the shared-memory regions in order, aligned and large enough."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "splitk", "splitk_partition_check.cu")
OUT = os.path.join(ROOT, "tests", "splitk", "_build")


def _nvcc():
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else shutil.which("nvcc")


def test_split_k_partition_and_layout():
    nvcc = _nvcc()
    if not nvcc:
        pytest.skip("no nvcc")
    os.makedirs(OUT, exist_ok=True)
    exe = os.path.join(OUT, "splitk_partition_check")
    cmd = [nvcc, "-std=c++17", "-O1", "-gencode", "arch=compute_103a,code=sm_103a",
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(ROOT, "quantised_decode_mat_gb300", "csrc"),
           SRC, "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-3000:]
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
