"""The C ABI as a C program uses it: tests/c_abi/qmd_c_caller.c, plain C99, includes only
include/qmd.h and the CUDA runtime's C header and links against libqmd.so.  On the CPU: it must
compile with warnings as errors and link.  On a GPU: it packs and multiplies a small Q4_K case
through qmd_q8k_pack + qmd_qmatvec and through qmd_qmatvec_x, and both results must equal the
oracle's same-order result bit for bit."""
import os
import subprocess

import numpy as np
import pytest

import oracle as O
from quantised_decode_mat_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_abi", "qmd_c_caller.c")
OUT_DIR = os.path.join(ROOT, "tests", "c_abi", "_build")
PKG = os.path.join(ROOT, "quantised_decode_mat_gb300")


def _cuda_home():
    return os.environ.get("CUDA_HOME", "/usr/local/cuda")


def build_caller() -> str:
    from quantised_decode_mat_gb300 import build as qbuild
    qbuild.build()
    os.makedirs(OUT_DIR, exist_ok=True)
    exe = os.path.join(OUT_DIR, "qmd_c_caller")
    cuda = _cuda_home()
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-O1",
           "-I", os.path.join(ROOT, "include"), "-isystem", os.path.join(cuda, "include"), SRC, "-o", exe,
           "-L", PKG, "-lqmd", f"-Wl,-rpath,{PKG}", "-L", os.path.join(cuda, "lib64"), "-lcudart",
           f"-Wl,-rpath,{os.path.join(cuda, 'lib64')}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_c_caller_compiles_as_c99_and_links():
    if not os.path.exists(os.path.join(_cuda_home(), "include", "cuda_runtime_api.h")):
        pytest.skip("no CUDA headers")
    assert os.path.exists(build_caller())


@pytest.mark.gpu
def test_c_caller_results_match_the_oracle(tmp_path):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    exe = build_caller()
    rows, K, batch = 37, 1280, 2
    W = synth.q4k_weights(81, rows, K)
    x = synth.activations(81, batch, K)
    inp, outp = tmp_path / "in.bin", tmp_path / "out.bin"
    with open(inp, "wb") as f:
        f.write(np.array([rows, K], np.int64).tobytes())
        f.write(np.array([batch], np.int32).tobytes())
        f.write(np.ascontiguousarray(W).tobytes())
        f.write(np.ascontiguousarray(x, np.float32).tobytes())
    r = subprocess.run([exe, str(inp), str(outp)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    y = np.fromfile(outp, np.float32).reshape(2, batch, rows)
    oqs, od, obs = O.q8k_pack(x)
    ref = O.qmatvec(O.FMT_Q4_K, W, oqs, od, obs, O.ORDER_RUNS_OF_SIXTEEN)
    for k in range(2):
        assert np.array_equal(y[k].view(np.uint32), ref.view(np.uint32))
