"""Counter-based seeded random numbers for the synthetic workloads (host side).

This module holds input generation only -- none of the attention or
quantisation arithmetic.  The CUDA twin in ``synth/csrc/synth_fill.cu``
implements the same counter-based generator bit for bit, so large caches can be
filled on the device while the CPU oracle regenerates exactly the rows it needs.

Generator (both sides):

* hash: the SplitMix64 output function (Steele, Lea and Flood, "Fast splittable
  pseudorandom number generators", OOPSLA 2014), applied to
  ``key + (counter + 1) * 0x9E3779B97F4A7C15`` (mod 2^64).
* normal variates: the classical "sum of twelve uniforms minus six" (Irwin-Hall,
  n = 12) approximation of N(0, 1).  Element ``i`` draws three 64-bit hashes at
  counters ``3i, 3i+1, 3i+2``, splits each into four 16-bit uniforms
  ``u in [0, 65535]``, sums the twelve (``S``), and returns
  ``(S - 393210) / 65536`` -- exact in fp32 (``|S - 393210| < 2^19``), mean 0,
  variance ``1 - 2^-32``, support ``[-6, 6]``.
* bf16: round-to-nearest-even of that fp32 value (never NaN).
"""
from __future__ import annotations

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_MASK16 = np.uint64(0xFFFF)

# Tensor identities mixed into the key (any distinct constants would do).
TENSOR_Q = 1
TENSOR_K = 2
TENSOR_V = 3
TENSOR_CKV = 4
TENSOR_QMLA = 5
TENSOR_CTX = 6
TENSOR_PERM = 7
TENSOR_TOPK = 8


def mix64(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output function on uint64 arrays (wrapping arithmetic)."""
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        z = z ^ (z >> np.uint64(31))
    return z


def make_key(seed: int, tensor: int) -> int:
    """64-bit stream key for (seed, tensor)."""
    with np.errstate(over="ignore"):
        k = mix64(np.array([np.uint64(seed) * GOLDEN + np.uint64(tensor)], dtype=np.uint64))[0]
    return int(k)


def hash_at(key: int, counter: np.ndarray) -> np.ndarray:
    c = np.asarray(counter, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return mix64(np.uint64(key) + (c + np.uint64(1)) * GOLDEN)


def normal_f32(key: int, idx: np.ndarray) -> np.ndarray:
    """Irwin-Hall(12) normal variates (fp32) for element indices ``idx``."""
    idx = np.asarray(idx, dtype=np.uint64)
    s = np.zeros(idx.shape, dtype=np.int64)
    with np.errstate(over="ignore"):
        base = idx * np.uint64(3)
        for j in range(3):
            h = hash_at(key, base + np.uint64(j))
            for k in range(4):
                s += ((h >> np.uint64(16 * k)) & _MASK16).astype(np.int64)
    return ((s - 393210).astype(np.float32)) * np.float32(1.0 / 65536.0)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even fp32 -> bf16 (inputs here are finite)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal_bf16(key: int, idx: np.ndarray) -> np.ndarray:
    return f32_to_bf16_bits(normal_f32(key, idx))


def uniform_u64(key: int, idx: np.ndarray) -> np.ndarray:
    return hash_at(key, np.asarray(idx, dtype=np.uint64))


def uniform_int(key: int, idx: np.ndarray, lo: int, hi: int) -> np.ndarray:
    """Integers in [lo, hi] (inclusive) by reduction of one hash modulo the span."""
    span = np.uint64(hi - lo + 1)
    return (uniform_u64(key, idx) % span).astype(np.int64) + lo


def permutation(key: int, n: int) -> np.ndarray:
    """A uniform random permutation of range(n): argsort of n hashed keys."""
    h = uniform_u64(key, np.arange(n, dtype=np.uint64))
    return np.argsort(h, kind="stable").astype(np.int64)


def sample_sorted_unique(key: int, row: int, n_pool: int, k: int) -> np.ndarray:
    """k distinct integers from [0, n_pool), sorted: the k smallest hash keys."""
    idx = np.uint64(row) * np.uint64(n_pool) + np.arange(n_pool, dtype=np.uint64)
    h = uniform_u64(key, idx)
    pick = np.argpartition(h, k - 1)[:k] if k < n_pool else np.arange(n_pool)
    return np.sort(pick).astype(np.int32)
