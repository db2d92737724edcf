"""CPU oracle for paged FP8 (e4m3) KV decode attention -- TEST INFRASTRUCTURE.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library (``libpfkv``) shares
no code with it.  The arithmetic lives in plain C (``pfkv_oracle.c``, IEEE
double for attention); this module only compiles it with gcc and marshals numpy
arrays through ctypes.  ctypes releases the GIL during each call, so callers may
spread independent (request, head) units over threads without touching the
arithmetic.

Parity pins: every function here is pinned by ``tests/test_oracle_*.py``
against the e4m3 format definition, library routines (torch's float8_e4m3fn
cast, torch's scaled_dot_product_attention in float64), closed forms and
invariants stated on the source pages.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pfkv_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libpfkv_oracle.so")

ORC_OK = 0
ORC_ERR_ARG = -1
ORC_ERR_INDEX = -4
ORC_CACHE_FP8_E4M3 = 0
ORC_CACHE_BF16 = 1

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (strict IEEE: no contraction, no fast-math)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    newest_src = max(os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "pfkv_oracle.h")))
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= newest_src:
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O1", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
            L.orc_e4m3_value.restype = ctypes.c_double
            L.orc_e4m3_value.argtypes = [ctypes.c_uint8]
            L.orc_e4m3_encode.restype = ctypes.c_uint8
            L.orc_e4m3_encode.argtypes = [f32]
            L.orc_e4m3_encode_array.restype = None
            L.orc_e4m3_encode_array.argtypes = [vp, vp, i64]
            L.orc_bf16_to_f32.restype = f32
            L.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
            L.orc_kv_append.restype = i32
            L.orc_kv_append.argtypes = [vp, vp, vp, i32, i32, i32, i32, i64, f32]
            L.orc_kv_append_bf16.restype = i32
            L.orc_kv_append_bf16.argtypes = [vp, vp, vp, i32, i32, i32, i32, i64]
            L.orc_kv_append_head.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i64]
            L.orc_kv_append_token.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i64]
            L.orc_paged_decode_scaled_one.argtypes = [vp, vp, vp, vp, vp, i32, vp, vp, vp, i32, i32,
                                                      i32, i32, i32, i64, f32]
            L.orc_paged_prefill.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32, vp, vp, i32, i32, i32, i32,
                                            i32, i64, f32, f32, f32, i64, i64]
            L.orc_paged_decode_scaled.argtypes = [vp, vp, vp, vp, vp, i32, vp, vp, vp, i32, vp, i32,
                                                  i32, i32, i32, i32, i64, f32, i64, i64]
            L.orc_paged_decode_one.restype = i32
            L.orc_paged_decode_one.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32,
                                               i64, f32, f32, f32]
            L.orc_paged_decode.restype = i32
            L.orc_paged_decode.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32, vp, i32, i32, i32, i32,
                                           i32, i64, f32, f32, f32, i64, i64]
            L.orc_paged_decode_split_one.restype = i32
            L.orc_paged_decode_split_one.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32,
                                                     i32, i64, f32, f32, f32, i32]
            L.orc_mla_decode_one.restype = i32
            L.orc_mla_decode_one.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i64,
                                             f32, f32]
            L.orc_mla_decode.restype = i32
            L.orc_mla_decode.argtypes = [vp, vp, vp, vp, vp, i32, vp, vp, i32, i32, i32, i32, i32,
                                         i32, i64, f32, f32, i64, i64]
            L.orc_verify_page_tags.restype = i32
            L.orc_verify_page_tags.argtypes = [vp, vp, i32, vp, i32, i32, vp, i64, vp]
            L.orc_kv_bytes.restype = i64
            L.orc_kv_bytes.argtypes = [i64, i64, i64, i64, i64]
            _lib = L
    return _lib


class OracleError(RuntimeError):
    pass


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _chk(rc):
    if rc != ORC_OK:
        raise OracleError(f"oracle returned {rc}")


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------- e4m3 format
def e4m3_value(code: int) -> float:
    return lib().orc_e4m3_value(int(code))


def e4m3_table() -> np.ndarray:
    """float64[256]: the value of every e4m3 code (NaN for 0x7F and 0xFF)."""
    return np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)


def e4m3_encode(x) -> np.ndarray:
    """Round fp32 values to e4m3 codes (RNE, saturating, NaN -> 0x7F)."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32).reshape(-1))
    out = np.empty(x.shape[0], np.uint8)
    lib().orc_e4m3_encode_array(_ptr(x), _ptr(out), x.shape[0])
    return out


def bf16_to_f32(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


# --------------------------------------------------------------------- append
def kv_append(x_new_bf16, cache, slot_mapping, page_size: int, scale: float):
    """In place: quantise x_new [T][H][D] (bf16 bits) into cache [pages][H][P][D] (u8)."""
    x = _c(x_new_bf16, np.uint16)
    T, H, D = x.shape
    assert cache.dtype == np.uint8 and cache.flags.c_contiguous
    num_pages = cache.shape[0]
    sm = _c(slot_mapping, np.int64)
    _chk(lib().orc_kv_append(_ptr(x), _ptr(cache), _ptr(sm), T, H, D, page_size, num_pages,
                             ctypes.c_float(scale)))


def kv_append_bf16(x_new_bf16, cache, slot_mapping, page_size: int):
    x = _c(x_new_bf16, np.uint16)
    T, H, D = x.shape
    assert cache.dtype == np.uint16 and cache.flags.c_contiguous
    sm = _c(slot_mapping, np.int64)
    _chk(lib().orc_kv_append_bf16(_ptr(x), _ptr(cache), _ptr(sm), T, H, D, page_size,
                                  cache.shape[0]))


SCALE_TENSOR = 0
SCALE_HEAD = 1
SCALE_TOKEN = 2


def kv_append_head(x_new_bf16, cache, slot_mapping, page_size: int, head_scales):
    """In place: quantise x_new [T][H][D] with one scale per KV head (float32 [H])."""
    x = _c(x_new_bf16, np.uint16)
    T, H, D = x.shape
    assert cache.dtype == np.uint8 and cache.flags.c_contiguous
    hs = _c(head_scales, np.float32)
    assert hs.shape == (H,)
    sm = _c(slot_mapping, np.int64)
    _chk(lib().orc_kv_append_head(_ptr(x), _ptr(cache), _ptr(hs), _ptr(sm), T, H, D, page_size,
                                  cache.shape[0]))


def kv_append_token(x_new_bf16, cache, scales, slot_mapping, page_size: int):
    """In place: quantise x_new [T][H][D] with one scale per (token, KV head) row,
    written to scales float32 [pages][H][P] beside the row."""
    x = _c(x_new_bf16, np.uint16)
    T, H, D = x.shape
    assert cache.dtype == np.uint8 and cache.flags.c_contiguous
    assert scales.dtype == np.float32 and scales.flags.c_contiguous
    assert scales.shape == cache.shape[:3]
    sm = _c(slot_mapping, np.int64)
    _chk(lib().orc_kv_append_token(_ptr(x), _ptr(cache), _ptr(scales), _ptr(sm), T, H, D,
                                   page_size, cache.shape[0]))


# ------------------------------------------------------------------ attention
def paged_decode_scaled(q_bf16, k_cache, v_cache, granularity: int, k_scales, v_scales,
                        block_tables, context_lens, page_size: int, softmax_scale: float,
                        num_kv_heads: int, units=None):
    """Double-precision decode over an e4m3 cache with per-tensor ([1]), per-head
    ([Hkv]) or per-token ([pages][Hkv][P]) float32 scales."""
    q = _c(q_bf16, np.uint16)
    B, Hq, D = q.shape
    assert k_cache.dtype == np.uint8 and v_cache.dtype == np.uint8
    ks = _c(k_scales, np.float32)
    vs = _c(v_scales, np.float32)
    bt = _c(block_tables, np.int32)
    cl = _c(context_lens, np.int32)
    out = np.zeros((B, Hq, D), np.float64)
    lse = np.full((B, Hq), -np.inf, np.float64)
    u0, u1 = (0, B * Hq) if units is None else units
    _chk(lib().orc_paged_decode_scaled(_ptr(out), _ptr(lse), _ptr(q), _ptr(k_cache),
                                       _ptr(v_cache), granularity, _ptr(ks), _ptr(vs), _ptr(bt),
                                       bt.shape[1], _ptr(cl), B, Hq, num_kv_heads, D, page_size,
                                       k_cache.shape[0], softmax_scale, u0, u1))
    return out, lse


def paged_decode_scaled_one(q_head_bf16, k_cache, v_cache, granularity: int, k_scales, v_scales,
                            bt_row, L: int, kvh: int, page_size: int, softmax_scale: float):
    q = _c(q_head_bf16, np.uint16).reshape(-1)
    D = q.shape[0]
    ks = _c(k_scales, np.float32)
    vs = _c(v_scales, np.float32)
    bt = _c(bt_row, np.int32)
    out = np.zeros(D, np.float64)
    lse = ctypes.c_double(0.0)
    _chk(lib().orc_paged_decode_scaled_one(_ptr(out), ctypes.byref(lse), _ptr(q), _ptr(k_cache),
                                           _ptr(v_cache), granularity, _ptr(ks), _ptr(vs),
                                           _ptr(bt), L, k_cache.shape[1], kvh, D, page_size,
                                           k_cache.shape[0], softmax_scale))
    return out, lse.value


def paged_decode(q_bf16, k_cache, v_cache, block_tables, context_lens, page_size: int,
                 k_scale: float, v_scale: float, softmax_scale: float, num_kv_heads: int,
                 units=None):
    """Double-precision decode attention.  q [B][Hq][D] bf16 bits; caches
    [pages][Hkv][P][D] u8 (e4m3) or u16 (bf16).  Returns (out [B][Hq][D], lse [B][Hq])."""
    q = _c(q_bf16, np.uint16)
    B, Hq, D = q.shape
    dt = ORC_CACHE_BF16 if k_cache.dtype == np.uint16 else ORC_CACHE_FP8_E4M3
    bt = _c(block_tables, np.int32)
    cl = _c(context_lens, np.int32)
    out = np.zeros((B, Hq, D), np.float64)
    lse = np.full((B, Hq), -np.inf, np.float64)
    u0, u1 = (0, B * Hq) if units is None else units
    _chk(lib().orc_paged_decode(_ptr(out), _ptr(lse), _ptr(q), _ptr(k_cache), _ptr(v_cache), dt,
                                _ptr(bt), bt.shape[1], _ptr(cl), B, Hq, num_kv_heads, D, page_size,
                                k_cache.shape[0], k_scale, v_scale, softmax_scale, u0, u1))
    return out, lse


def paged_prefill(q_bf16, k_cache, v_cache, block_tables, context_lens, q_start, page_size: int,
                  k_scale: float, v_scale: float, softmax_scale: float, num_kv_heads: int, rows=None):
    """Several new query tokens per request, causal among themselves: q
    [total_q][Hq][D] bf16 bits with request b's rows q_start[b] .. q_start[b+1]-1
    at positions L_b - n_b + i.  Returns (out [total_q][Hq][D], lse [total_q][Hq])."""
    q = _c(q_bf16, np.uint16)
    T, Hq, D = q.shape
    dt = ORC_CACHE_BF16 if k_cache.dtype == np.uint16 else ORC_CACHE_FP8_E4M3
    bt = _c(block_tables, np.int32)
    cl = _c(context_lens, np.int32)
    qs = _c(q_start, np.int32)
    B = cl.shape[0]
    assert qs.shape == (B + 1,) and qs[-1] == T
    out = np.zeros((T, Hq, D), np.float64)
    lse = np.full((T, Hq), -np.inf, np.float64)
    r0, r1 = (0, T * Hq) if rows is None else rows
    _chk(lib().orc_paged_prefill(_ptr(out), _ptr(lse), _ptr(q), _ptr(k_cache), _ptr(v_cache), dt,
                                 _ptr(bt), bt.shape[1], _ptr(cl), _ptr(qs), B, Hq, num_kv_heads, D,
                                 page_size, k_cache.shape[0], k_scale, v_scale, softmax_scale, r0, r1))
    return out, lse


def paged_decode_one(q_head_bf16, k_cache, v_cache, bt_row, L: int, kvh: int, page_size: int,
                     k_scale: float, v_scale: float, softmax_scale: float, chunk: int = 0):
    """One query head of one request; chunk > 0 runs the split-KV + LSE-merge form."""
    q = _c(q_head_bf16, np.uint16).reshape(-1)
    D = q.shape[0]
    Hkv = k_cache.shape[1]
    dt = ORC_CACHE_BF16 if k_cache.dtype == np.uint16 else ORC_CACHE_FP8_E4M3
    bt = _c(bt_row, np.int32)
    out = np.zeros(D, np.float64)
    lse = ctypes.c_double(0.0)
    if chunk > 0:
        rc = lib().orc_paged_decode_split_one(_ptr(out), ctypes.byref(lse), _ptr(q), _ptr(k_cache),
                                              _ptr(v_cache), dt, _ptr(bt), L, Hkv, kvh, D,
                                              page_size, k_cache.shape[0], k_scale, v_scale,
                                              softmax_scale, chunk)
    else:
        rc = lib().orc_paged_decode_one(_ptr(out), ctypes.byref(lse), _ptr(q), _ptr(k_cache),
                                        _ptr(v_cache), dt, _ptr(bt), L, Hkv, kvh, D, page_size,
                                        k_cache.shape[0], k_scale, v_scale, softmax_scale)
    _chk(rc)
    return out, lse.value


def mla_decode(q_bf16, ckv_cache, block_tables, context_lens, topk, page_size: int, d_v: int,
               ckv_scale: float, softmax_scale: float, units=None):
    """q [B][H][Dqk] bf16 bits; ckv_cache [pages][P][Dqk] u8; topk [B][k] int32 or None.
    Returns (out [B][H][Dv], lse [B][H])."""
    q = _c(q_bf16, np.uint16)
    B, H, Dqk = q.shape
    bt = _c(block_tables, np.int32)
    cl = _c(context_lens, np.int32)
    tk = None if topk is None else _c(topk, np.int32)
    kn = 0 if tk is None else tk.shape[1]
    out = np.zeros((B, H, d_v), np.float64)
    lse = np.full((B, H), -np.inf, np.float64)
    u0, u1 = (0, B * H) if units is None else units
    _chk(lib().orc_mla_decode(_ptr(out), _ptr(lse), _ptr(q), _ptr(ckv_cache), _ptr(bt), bt.shape[1],
                              _ptr(cl), _ptr(tk), kn, B, H, Dqk, d_v, page_size,
                              ckv_cache.shape[0], ckv_scale, softmax_scale, u0, u1))
    return out, lse


def mla_decode_one(q_head_bf16, ckv_cache, bt_row, L: int, topk_row, page_size: int, d_v: int,
                   ckv_scale: float, softmax_scale: float):
    q = _c(q_head_bf16, np.uint16).reshape(-1)
    bt = _c(bt_row, np.int32)
    tk = None if topk_row is None else _c(topk_row, np.int32).reshape(-1)
    out = np.zeros(d_v, np.float64)
    lse = ctypes.c_double(0.0)
    _chk(lib().orc_mla_decode_one(_ptr(out), ctypes.byref(lse), _ptr(q), _ptr(ckv_cache), _ptr(bt),
                                  L, _ptr(tk), 0 if tk is None else tk.shape[0], q.shape[0], d_v,
                                  page_size, ckv_cache.shape[0], ckv_scale, softmax_scale))
    return out, lse.value


def kv_bytes(layers: int, kv_heads: int, head_dim: int, tokens: int, bytes_per_elem: int) -> int:
    return int(lib().orc_kv_bytes(layers, kv_heads, head_dim, tokens, bytes_per_elem))


REQ_TAG_MISMATCH = 0x1
REQ_BAD_INDEX = 0x2


def verify_page_tags(block_tables, table_tags, context_lens, page_size: int, page_tags) -> np.ndarray:
    """Per-request status of the page-tag check: 0 or an OR of REQ_TAG_MISMATCH / REQ_BAD_INDEX."""
    bt = _c(block_tables, np.int32)
    tt = _c(np.asarray(table_tags).astype(np.uint32, copy=False), np.uint32)
    cl = _c(context_lens, np.int32)
    pt = _c(np.asarray(page_tags).astype(np.uint32, copy=False), np.uint32)
    status = np.zeros(cl.shape[0], np.int32)
    _chk(lib().orc_verify_page_tags(_ptr(bt), _ptr(tt), bt.shape[1], _ptr(cl), cl.shape[0], page_size,
                                    _ptr(pt), pt.shape[0], _ptr(status)))
    return status
