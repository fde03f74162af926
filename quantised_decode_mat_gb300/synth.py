"""Seeded synthetic inputs for the decode mat-vec: GGUF-shaped weight bytes and f32 activations.

This module only draws random numbers.  It holds none of the method's arithmetic: no block
decoding, no quantisation, no dot products.  Both the CPU oracle's tests and the GPU path's
tests and benchmark take their inputs from here, so the two sides see the same bytes.

Generator: SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number generators",
OOPSLA 2014), used counter-style: word i of a stream with key k is mix(k + (i + 1) * GAMMA),
where mix is the SplitMix64 output function.  Any block of any tensor can therefore be
regenerated alone, which is how full-size outputs are sampled for the oracle.

Value distributions follow the workloads the pages measure (7B-class projection layers):
  * Q4_K blocks: f16 d, dmin ~ U[1e-3, 1e-2] (an f32 draw rounded to f16, nearest-even),
    12 scale bytes uniform (so every packed 6-bit scale and min is uniform on 0..63),
    128 nibble bytes uniform (so every 4-bit code is uniform on 0..15).
  * Q6_K blocks: 128 ql bytes and 64 qh bytes uniform, 16 int8 scales ~ U{-32..31},
    f16 d ~ U[1e-3, 1e-2].
  * activations: x ~ N(0, 1) in f32 via the Box-Muller transform computed in f64.
"""
from __future__ import annotations

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

QK_K = 256
Q4K_BLOCK_BYTES = 144
Q5K_BLOCK_BYTES = 176
Q6K_BLOCK_BYTES = 210

# tensor ids used in stream keys
T_Q4K, T_Q6K, T_ACT, T_RES, T_GAIN, T_Q5K = 1, 2, 3, 4, 5, 6
# sub-streams inside a tensor
_S_D, _S_DMIN, _S_SCALES, _S_QS, _S_QL, _S_QH, _S_U1, _S_U2 = range(8)


_S30, _S27, _S31 = np.uint64(30), np.uint64(27), np.uint64(31)


def _mix(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output function (z ^= z >> 30; z *= M1; z ^= z >> 27; z *= M2; z ^= z >> 31)."""
    z = np.array(z, dtype=np.uint64, copy=True)
    with np.errstate(over="ignore"):
        z ^= np.right_shift(z, _S30)
        np.multiply(z, _M1, out=z)
        z ^= np.right_shift(z, _S27)
        np.multiply(z, _M2, out=z)
        z ^= np.right_shift(z, _S31)
    return z


def stream_key(*ids: int) -> np.uint64:
    """Fold a tuple of small non-negative ints into one 64-bit stream key."""
    k = np.uint64(0)
    for v in ids:
        with np.errstate(over="ignore"):
            k = _mix(np.asarray(k ^ np.uint64(v & 0xFFFFFFFFFFFFFFFF), dtype=np.uint64) + GAMMA)
    return np.uint64(k)


def u64(key: np.uint64, n: int, start: int = 0) -> np.ndarray:
    """Words start .. start+n-1 of the stream `key`."""
    z = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        np.multiply(z, GAMMA, out=z)
        np.add(z, np.uint64(key), out=z)
    return _mix(z)


def rand_bytes(key: np.uint64, n: int) -> np.ndarray:
    words = u64(key, (n + 7) // 8)
    return words.view(np.uint8)[:n].copy()


def uniform01(key: np.uint64, n: int) -> np.ndarray:
    """f64 in (0, 1]: (top 53 bits + 1) / 2^53, never 0 so that log() is finite."""
    return ((u64(key, n) >> np.uint64(11)).astype(np.float64) + 1.0) * (1.0 / 9007199254740992.0)


def _f16_uniform(key: np.uint64, n: int, lo: float = 1e-3, hi: float = 1e-2) -> np.ndarray:
    u = uniform01(key, n)
    v = (lo + (hi - lo) * u).astype(np.float32)
    return v.astype(np.float16)  # IEEE round-to-nearest-even


def q4k_weights(seed: int, rows: int, K: int, layer: int = 0, tensor: int = 0) -> np.ndarray:
    """uint8 [rows, K/256, 144]: canonical GGUF Q4_K blocks in row-major block order."""
    assert K % QK_K == 0
    nb = K // QK_K
    n = rows * nb
    base = (seed, T_Q4K, layer, tensor)
    out = np.empty((n, Q4K_BLOCK_BYTES), dtype=np.uint8)
    out[:, 0:2] = _f16_uniform(stream_key(*base, _S_D), n).view(np.uint8).reshape(n, 2)
    out[:, 2:4] = _f16_uniform(stream_key(*base, _S_DMIN), n).view(np.uint8).reshape(n, 2)
    out[:, 4:16] = rand_bytes(stream_key(*base, _S_SCALES), n * 12).reshape(n, 12)
    out[:, 16:144] = rand_bytes(stream_key(*base, _S_QS), n * 128).reshape(n, 128)
    return out.reshape(rows, nb, Q4K_BLOCK_BYTES)


def q5k_weights(seed: int, rows: int, K: int, layer: int = 0, tensor: int = 0) -> np.ndarray:
    """uint8 [rows, K/256, 176]: canonical GGUF Q5_K blocks (d, dmin, 12 scale/min bytes, 32
    bytes of fifth bits, 128 bytes of low nibbles); the same value distributions as Q4_K with
    uniform fifth bits."""
    assert K % QK_K == 0
    nb = K // QK_K
    n = rows * nb
    base = (seed, T_Q5K, layer, tensor)
    out = np.empty((n, Q5K_BLOCK_BYTES), dtype=np.uint8)
    out[:, 0:2] = _f16_uniform(stream_key(*base, _S_D), n).view(np.uint8).reshape(n, 2)
    out[:, 2:4] = _f16_uniform(stream_key(*base, _S_DMIN), n).view(np.uint8).reshape(n, 2)
    out[:, 4:16] = rand_bytes(stream_key(*base, _S_SCALES), n * 12).reshape(n, 12)
    out[:, 16:48] = rand_bytes(stream_key(*base, _S_QH), n * 32).reshape(n, 32)
    out[:, 48:176] = rand_bytes(stream_key(*base, _S_QS), n * 128).reshape(n, 128)
    return out.reshape(rows, nb, Q5K_BLOCK_BYTES)


def q6k_weights(seed: int, rows: int, K: int, layer: int = 0, tensor: int = 0) -> np.ndarray:
    """uint8 [rows, K/256, 210]: canonical GGUF Q6_K blocks (ql, qh, scales, d)."""
    assert K % QK_K == 0
    nb = K // QK_K
    n = rows * nb
    base = (seed, T_Q6K, layer, tensor)
    out = np.empty((n, Q6K_BLOCK_BYTES), dtype=np.uint8)
    out[:, 0:128] = rand_bytes(stream_key(*base, _S_QL), n * 128).reshape(n, 128)
    out[:, 128:192] = rand_bytes(stream_key(*base, _S_QH), n * 64).reshape(n, 64)
    sc = (rand_bytes(stream_key(*base, _S_SCALES), n * 16).astype(np.int16) % 64) - 32
    out[:, 192:208] = sc.astype(np.int8).view(np.uint8).reshape(n, 16)
    out[:, 208:210] = _f16_uniform(stream_key(*base, _S_D), n).view(np.uint8).reshape(n, 2)
    return out.reshape(rows, nb, Q6K_BLOCK_BYTES)


def activations(seed: int, batch: int, K: int, layer: int = 0, tensor: int = 0) -> np.ndarray:
    """f32 [batch, K] ~ N(0, 1) (Box-Muller in f64, rounded once to f32)."""
    n = batch * K
    base = (seed, T_ACT, layer, tensor)
    u1 = uniform01(stream_key(*base, _S_U1), n)
    u2 = uniform01(stream_key(*base, _S_U2), n)
    x = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
    return x.astype(np.float32).reshape(batch, K)


def residual(seed: int, batch: int, K: int, layer: int = 0, tensor: int = 0) -> np.ndarray:
    """f32 [batch, K] ~ N(0, 1): the residual stream added before an RMSNorm."""
    n = batch * K
    base = (seed, T_RES, layer, tensor)
    u1 = uniform01(stream_key(*base, _S_U1), n)
    u2 = uniform01(stream_key(*base, _S_U2), n)
    x = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
    return x.astype(np.float32).reshape(batch, K)


def norm_gain(seed: int, K: int, layer: int = 0, tensor: int = 0) -> np.ndarray:
    """f32 [K] ~ U[0.5, 1.5]: an RMSNorm's per-element gain."""
    u = uniform01(stream_key(seed, T_GAIN, layer, tensor, _S_D), K)
    return (0.5 + u).astype(np.float32)


# ---------------------------------------------------------------------------------------------
# The five workloads: shapes and seeds.  Config 4 is a 32-layer 7B-shaped decode step; each
# projection of each layer consumes its own activation vector(s).
# ---------------------------------------------------------------------------------------------
CONFIGS = {
    0: dict(name="q4k_256x2048_b1", fmt="q4k", rows=256, K=2048, batches=(1,), seed=0),
    1: dict(name="q4k_4096x4096_b1", fmt="q4k", rows=4096, K=4096, batches=(1,), seed=1),
    2: dict(name="q6k_4096x14336_b1", fmt="q6k", rows=4096, K=14336, batches=(1,), seed=2),
    3: dict(name="q4k_28672x4096_b1248", fmt="q4k", rows=28672, K=4096, batches=(1, 2, 4, 8), seed=3),
}

# config 4: per layer (name, fmt, rows, K)
STEP_LAYERS = 32
STEP_PROJECTIONS = (
    ("qkv", "q4k", 6144, 4096),
    ("o", "q4k", 4096, 4096),
    ("gate_up", "q4k", 28672, 4096),
    ("down", "q6k", 4096, 14336),
)


def step_seed(layer: int) -> int:
    """Config 4 layer l draws from seed 4*1000 + l."""
    return 4 * 1000 + layer


def weights(fmt: str, seed: int, rows: int, K: int, layer: int = 0, tensor: int = 0) -> np.ndarray:
    if fmt == "q4k":
        return q4k_weights(seed, rows, K, layer, tensor)
    if fmt == "q5k":
        return q5k_weights(seed, rows, K, layer, tensor)
    if fmt == "q6k":
        return q6k_weights(seed, rows, K, layer, tensor)
    raise ValueError(fmt)
