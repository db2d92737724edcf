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

import ctypes
import os
import subprocess
import threading

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
TENSOR_SPREAD = 9


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


_HERE = os.path.dirname(os.path.abspath(__file__))
_HOST_SRC = os.path.join(_HERE, "csrc", "synth_host.c")
_HOST_LIB = os.path.join(_HERE, "_build", "libsynth_host.so")
_host = None
_host_lock = threading.Lock()


def build_host() -> str:
    """Compile the host C twin of this generator (gcc, strict IEEE)."""
    os.makedirs(os.path.dirname(_HOST_LIB), exist_ok=True)
    if os.path.exists(_HOST_LIB) and os.path.getmtime(_HOST_LIB) >= os.path.getmtime(_HOST_SRC):
        return _HOST_LIB
    tmp = _HOST_LIB + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
                    "-o", tmp, _HOST_SRC], check=True)
    os.replace(tmp, _HOST_LIB)
    return _HOST_LIB


def _host_lib():
    global _host
    with _host_lock:
        if _host is None:
            try:
                L = ctypes.CDLL(build_host())
            except (OSError, subprocess.CalledProcessError):
                _host = False
                return None
            L.synth_normal_bf16_idx.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_void_p, ctypes.c_int64]
            L.synth_normal_bf16_range.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint64,
                                                  ctypes.c_int64]
            L.synth_normal_bf16_rows.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint64,
                                                 ctypes.c_int64, ctypes.c_int64, ctypes.c_uint64]
            _host = L
    return _host or None


def normal_bf16_numpy(key: int, idx: np.ndarray) -> np.ndarray:
    return f32_to_bf16_bits(normal_f32(key, idx))


def normal_bf16(key: int, idx: np.ndarray) -> np.ndarray:
    """bf16 normals at counters idx (C twin when available; same bits)."""
    idx = np.ascontiguousarray(np.asarray(idx, dtype=np.uint64))
    L = _host_lib()
    if L is None:
        return normal_bf16_numpy(key, idx)
    out = np.empty(idx.shape, dtype=np.uint16)
    L.synth_normal_bf16_idx(out.ctypes.data_as(ctypes.c_void_p), np.uint64(key), idx.ctypes.data_as(ctypes.c_void_p),
                            idx.size)
    return out


def normal_bf16_range(key: int, base: int, n: int) -> np.ndarray:
    """bf16 normals at counters base .. base + n - 1."""
    L = _host_lib()
    if L is None:
        return normal_bf16_numpy(key, np.arange(base, base + n, dtype=np.uint64))
    out = np.empty(n, dtype=np.uint16)
    L.synth_normal_bf16_range(out.ctypes.data_as(ctypes.c_void_p), np.uint64(key), np.uint64(base), n)
    return out


def normal_bf16_rows(key: int, base: int, rows: int, row_len: int, row_stride: int) -> np.ndarray:
    """[rows][row_len] bf16 normals; row r covers counters base + r*row_stride + (0..row_len-1)."""
    L = _host_lib()
    if L is None:
        idx = (np.uint64(base) + np.arange(rows, dtype=np.uint64)[:, None] * np.uint64(row_stride)
               + np.arange(row_len, dtype=np.uint64)[None, :])
        return normal_bf16_numpy(key, idx.reshape(-1)).reshape(rows, row_len)
    out = np.empty((rows, row_len), dtype=np.uint16)
    L.synth_normal_bf16_rows(out.ctypes.data_as(ctypes.c_void_p), np.uint64(key), np.uint64(base), rows, row_len,
                             np.uint64(row_stride))
    return out


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
