"""CPU oracle for the Q4_K / Q6_K x q8_K decode mat-vec (ctypes wrapper over qmd_oracle.c).

TEST INFRASTRUCTURE ONLY.  Only `tests/`, `__graft_entry__.smoke()` and the benchmark's
CPU-baseline leg may import this package.  It shares no code with the CUDA path and never
imports it; the library's product path never imports this package.

Arrays are numpy; weights are canonical GGUF blocks (uint8 [rows, K/256, 144 or 210]).
Formats are named by their GGUF type ids: 12 = Q4_K, 13 = Q5_K, 14 = Q6_K.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "qmd_oracle.c")
BUILD_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD_DIR, "liboracle.so")

FMT_Q4_K = 12
FMT_Q5_K = 13
FMT_Q6_K = 14
QK = 256
BLOCK_BYTES = {FMT_Q4_K: 144, FMT_Q5_K: 176, FMT_Q6_K: 210}
ORDER_SEQUENTIAL = 0
ORDER_GROUPS_OF_FOUR = 1
ORDER_RUNS_OF_SIXTEEN = 2

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile qmd_oracle.c with gcc (portable C99, no FMA contraction)."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        tmp = LIB + f".tmp{os.getpid()}"
        subprocess.run(
            ["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-o", tmp, SRC, "-lm"],
            check=True,
        )
        os.replace(tmp, LIB)
    return LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(LIB)
            p = ctypes.c_void_p
            i64 = ctypes.c_int64
            i32 = ctypes.c_int
            L.oracle_f16_to_f32.argtypes = [ctypes.c_uint16]
            L.oracle_f16_to_f32.restype = ctypes.c_float
            L.oracle_q4k_fields.argtypes = [p, p, p, p, p, p]
            L.oracle_q4k_dequant.argtypes = [p, p]
            L.oracle_q6k_fields.argtypes = [p, p, p, p]
            L.oracle_q5k_fields.argtypes = [p, p, p, p, p, p]
            L.oracle_q5k_dequant.argtypes = [p, p]
            L.oracle_q5k_subdots.argtypes = [p, p, i64, p]
            L.oracle_q6k_dequant.argtypes = [p, p]
            L.oracle_q8k_pack.argtypes = [p, i64, p, p, p]
            L.oracle_q4k_subdots.argtypes = [p, p, i64, p]
            L.oracle_q6k_subdots.argtypes = [p, p, i64, p]
            L.oracle_block_terms.argtypes = [i32, p, p, p, p, i64, p]
            L.oracle_qmatvec.argtypes = [i32, p, p, p, p, i64, i64, i32, i32, p]
            L.oracle_qmatvec_f64.argtypes = [i32, p, p, p, i64, i64, i32, p]
            L.oracle_q6k_split.argtypes = [p, i64, i64, p, p, i64]
            L.oracle_rmsnorm.argtypes = [p, p, p, ctypes.c_float, i64, p, p]
            L.oracle_rmsnorm_q8k_pack.argtypes = [p, p, p, ctypes.c_float, i64, p, p, p, p, p]
            for name in ("oracle_q4k_fields", "oracle_q4k_dequant", "oracle_q6k_fields",
                         "oracle_q6k_dequant", "oracle_q8k_pack", "oracle_q4k_subdots",
                         "oracle_q6k_subdots", "oracle_block_terms",
                         "oracle_q5k_fields", "oracle_q5k_dequant", "oracle_q5k_subdots",
                         "oracle_qmatvec_f64", "oracle_q6k_split", "oracle_rmsnorm",
                         "oracle_rmsnorm_q8k_pack"):
                getattr(L, name).restype = None
            L.oracle_qmatvec.restype = ctypes.c_int  # 0, or non-zero for a refused call
            _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


# ---- scalar / block helpers -------------------------------------------------------------------
def f16_to_f32(h: int) -> float:
    return float(lib().oracle_f16_to_f32(int(h) & 0xFFFF))


def q4k_fields(block: np.ndarray):
    """-> (d, dmin, sc[8], m[8], q[256]) of one 144-byte block."""
    b = _c(block, np.uint8)
    assert b.size == 144
    d = np.zeros(1, np.float32)
    dm = np.zeros(1, np.float32)
    sc = np.zeros(8, np.int32)
    m = np.zeros(8, np.int32)
    q = np.zeros(256, np.int32)
    lib().oracle_q4k_fields(_ptr(b), _ptr(d), _ptr(dm), _ptr(sc), _ptr(m), _ptr(q))
    return float(d[0]), float(dm[0]), sc, m, q


def q5k_fields(block: np.ndarray):
    """-> (d, dmin, sc[8], m[8], q[256] in 0..31) of one 176-byte block."""
    b = _c(block, np.uint8)
    assert b.size == 176
    d = np.zeros(1, np.float32)
    dm = np.zeros(1, np.float32)
    sc = np.zeros(8, np.int32)
    m = np.zeros(8, np.int32)
    q = np.zeros(256, np.int32)
    lib().oracle_q5k_fields(_ptr(b), _ptr(d), _ptr(dm), _ptr(sc), _ptr(m), _ptr(q))
    return float(d[0]), float(dm[0]), sc, m, q


def q6k_fields(block: np.ndarray):
    """-> (d, sc[16] (signed), q[256] in 0..63) of one 210-byte block."""
    b = _c(block, np.uint8)
    assert b.size == 210
    d = np.zeros(1, np.float32)
    sc = np.zeros(16, np.int32)
    q = np.zeros(256, np.int32)
    lib().oracle_q6k_fields(_ptr(b), _ptr(d), _ptr(sc), _ptr(q))
    return float(d[0]), sc, q


def dequant(fmt: int, block: np.ndarray) -> np.ndarray:
    """f64 weight values of one block."""
    b = _c(block, np.uint8)
    w = np.zeros(256, np.float64)
    if fmt == FMT_Q4_K:
        lib().oracle_q4k_dequant(_ptr(b), _ptr(w))
    elif fmt == FMT_Q5_K:
        lib().oracle_q5k_dequant(_ptr(b), _ptr(w))
    else:
        lib().oracle_q6k_dequant(_ptr(b), _ptr(w))
    return w


# ---- q8_K -------------------------------------------------------------------------------------
def q8k_pack(x: np.ndarray):
    """x f32 [batch, K] -> (qs int8 [batch, K], d f32 [batch, K/256], bsums int16 [batch, K/256, 8])."""
    x = _c(np.atleast_2d(x), np.float32)
    batch, K = x.shape
    assert K % QK == 0
    nb = K // QK
    qs = np.zeros((batch, K), np.int8)
    d = np.zeros((batch, nb), np.float32)
    bs = np.zeros((batch, nb, 8), np.int16)
    L = lib()
    for v in range(batch):
        L.oracle_q8k_pack(x[v].ctypes.data, K, qs[v].ctypes.data, d[v].ctypes.data, bs[v].ctypes.data)
    return qs, d, bs


# ---- integer dots, block terms and the mat-vec -------------------------------------------------
def subdots(fmt: int, row: np.ndarray, qs: np.ndarray) -> np.ndarray:
    """One row's int32 sub-block dots against one packed vector: [nb, 8] (Q4_K, Q5_K) or [nb, 16] (Q6_K)."""
    row = _c(row, np.uint8)
    qs = _c(qs, np.int8).reshape(-1)
    K = qs.size
    nb = K // QK
    per = 16 if fmt == FMT_Q6_K else 8
    out = np.zeros((nb, per), np.int32)
    if fmt == FMT_Q4_K:
        lib().oracle_q4k_subdots(_ptr(row), _ptr(qs), K, _ptr(out))
    elif fmt == FMT_Q5_K:
        lib().oracle_q5k_subdots(_ptr(row), _ptr(qs), K, _ptr(out))
    else:
        lib().oracle_q6k_subdots(_ptr(row), _ptr(qs), K, _ptr(out))
    return out


def block_terms(fmt: int, row: np.ndarray, qs: np.ndarray, xd: np.ndarray, bsums: np.ndarray) -> np.ndarray:
    row = _c(row, np.uint8)
    qs = _c(qs, np.int8).reshape(-1)
    xd = _c(xd, np.float32).reshape(-1)
    bsums = _c(bsums, np.int16).reshape(-1)
    K = qs.size
    out = np.zeros(K // QK, np.float32)
    lib().oracle_block_terms(fmt, _ptr(row), _ptr(qs), _ptr(xd), _ptr(bsums), K, _ptr(out))
    return out


def qmatvec(fmt: int, W: np.ndarray, qs: np.ndarray, xd: np.ndarray, bsums: np.ndarray,
            order: int = ORDER_SEQUENTIAL) -> np.ndarray:
    """y f32 [batch, rows] from canonical GGUF W [rows, nb, bytes] and packed vectors."""
    W = _c(W, np.uint8)
    rows = W.shape[0]
    qs = _c(np.atleast_2d(qs), np.int8)
    batch, K = qs.shape
    nb = K // QK
    assert W.size == rows * nb * BLOCK_BYTES[fmt], "W shape does not match K"
    xd = _c(xd, np.float32).reshape(batch, nb)
    bsums = _c(bsums, np.int16).reshape(batch, nb, 8)
    y = np.zeros((batch, rows), np.float32)
    rc = lib().oracle_qmatvec(fmt, _ptr(W), _ptr(qs), _ptr(xd), _ptr(bsums), rows, K, batch, order, _ptr(y))
    if rc != 0:
        raise RuntimeError(f"oracle_qmatvec refused the call (status {rc}, K={K}, batch={batch})")
    return y


def qmatvec_f64(fmt: int, W: np.ndarray, qs: np.ndarray, xd: np.ndarray) -> np.ndarray:
    """Brute force: f64 dequantised W times f64 (dx * q8), summed in f64.  [batch, rows]."""
    W = _c(W, np.uint8)
    rows = W.shape[0]
    qs = _c(np.atleast_2d(qs), np.int8)
    batch, K = qs.shape
    nb = K // QK
    assert W.size == rows * nb * BLOCK_BYTES[fmt]
    xd = _c(xd, np.float32).reshape(batch, nb)
    y = np.zeros((batch, rows), np.float64)
    lib().oracle_qmatvec_f64(fmt, _ptr(W), _ptr(qs), _ptr(xd), rows, K, batch, _ptr(y))
    return y


def q6k_split(gguf: np.ndarray, prefix_stride: int):
    """Canonical Q6_K [rows, nb, 210] -> (body uint8 [rows, nb, 208], prefix uint16 [rows, prefix_stride])."""
    g = _c(gguf, np.uint8)
    rows, nb = g.shape[0], g.shape[1]
    body = np.zeros((rows, nb, 208), np.uint8)
    prefix = np.zeros((rows, prefix_stride), np.uint16)
    lib().oracle_q6k_split(_ptr(g), rows, nb * QK, _ptr(body), _ptr(prefix), prefix_stride)
    return body, prefix


# ---- RMSNorm (+ residual) before the pack ------------------------------------------------------
def rmsnorm(x: np.ndarray, r: np.ndarray | None, g: np.ndarray, eps: float):
    """x, r f32 [batch, K] (r may be None), g f32 [K] -> (h, n) f32 [batch, K]: h = x + r, n the
    RMS-normalised h times g, in the declared order (oracle_rmsnorm)."""
    x = _c(np.atleast_2d(x), np.float32)
    batch, K = x.shape
    assert K % QK == 0
    r = None if r is None else _c(np.atleast_2d(r), np.float32).reshape(batch, K)
    g = _c(g, np.float32).reshape(K)
    h = np.zeros((batch, K), np.float32)
    n = np.zeros((batch, K), np.float32)
    L = lib()
    for v in range(batch):
        L.oracle_rmsnorm(x[v].ctypes.data, None if r is None else r[v].ctypes.data, _ptr(g), eps, K,
                         h[v].ctypes.data, n[v].ctypes.data)
    return h, n


def rmsnorm_q8k_pack(x: np.ndarray, r: np.ndarray | None, g: np.ndarray, eps: float):
    """-> (h f32 [batch, K], qs, d, bsums) as q8k_pack of the RMS-normalised x + r."""
    h, n = rmsnorm(x, r, g, eps)
    qs, d, bs = q8k_pack(n)
    return h, qs, d, bs


def rel_err(y: np.ndarray, ref: np.ndarray, floor_frac: float = 1e-3) -> np.ndarray:
    """Per-element |y - ref| / max(|ref|, floor_frac * rms(ref over that output vector)).

    y, ref: [batch, rows].  The floor keeps outputs that cancel to near zero from turning a
    rounding difference into a large relative error."""
    y = np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    rms = np.sqrt(np.mean(ref * ref, axis=-1, keepdims=True))
    den = np.maximum(np.abs(ref), floor_frac * rms)
    den = np.where(den == 0, 1.0, den)
    return np.abs(y - ref) / den
