"""paged_fp8_kv_02_gb300 -- decode attention over a paged FP8 (e4m3) KV cache
for NVIDIA GB300 (sm_103a).

A thin Python binding over the C ABI in ``include/pfkv.h`` (``libpfkv.so``).
Every function below has the name of the C entry point without the ``pfkv_``
prefix and only marshals arguments: tensors become device pointers, the current
torch CUDA stream becomes the ``stream`` argument, and a negative status raises
``PfkvError``.  PyTorch supplies device memory and streams; all arithmetic runs
in the library's CUDA kernels.  There is no fallback: if ``libpfkv.so`` is
missing or fails to load, importing the binding's functions raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import _build

__all__ = [
    "PfkvError", "load", "lib_path", "kv_append_fp8", "kv_append_bf16",
    "paged_decode_workspace_size", "paged_decode_attn", "paged_decode_attn_noalloc",
    "mla_decode_workspace_size",
    "mla_decode_attn", "validate_tables", "verify_page_tags", "workspace_status", "selftest_barrier_timeout",
    "last_error", "version",
    "CACHE_FP8_E4M3", "CACHE_BF16", "DEVERR", "REQ_TAG_MISMATCH", "REQ_BAD_INDEX",
    "PagePool", "block_hash", "slots_from_table",
]

CACHE_FP8_E4M3 = 0
CACHE_BF16 = 1
DEVERR = {
    "WAIT_TIMEOUT": 0x01, "BAD_PAGE": 0x02, "BAD_CONTEXT": 0x04, "WORKSPACE": 0x08,
    "BAD_TOPK": 0x10, "BAD_SLOT": 0x20,
}

REQ_TAG_MISMATCH = 0x1  # verify_page_tags: a page the request reads carries another tag
REQ_BAD_INDEX = 0x2     # verify_page_tags: a page id or context length out of range

_lock = threading.Lock()
_lib = None


class PfkvError(RuntimeError):
    def __init__(self, fn: str, code: int, msg: str):
        super().__init__(f"{fn} failed with status {code}: {msg}")
        self.code = code


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libpfkv.so (building it first if it is absent and allowed)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if not os.path.exists(path):
            if not build_if_missing:
                raise OSError(f"libpfkv not built: {path}")
            _build.build_pfkv()
        L = ctypes.CDLL(path)
        vp, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
        sig = {
            "pfkv_kv_append_fp8": (i32, [vp, vp, vp, vp, vp, i32, i32, i32, i32, i64, f32, f32, vp]),
            "pfkv_kv_append_bf16": (i32, [vp, vp, vp, vp, vp, i32, i32, i32, i32, i64, vp]),
            "pfkv_kv_append_fp8_scaled": (i32, [vp, vp, vp, vp, vp, i32, i32, i32, i32, i64, i32, vp, vp,
                                                vp]),
            "pfkv_paged_decode_workspace_size": (sz, [i32, i32, i32, i32, i32, i64]),
            "pfkv_paged_decode_attn": (i32, [vp, vp, vp, vp, i32, vp, i32, vp, i32, i32, i32, i32, i32,
                                             i64, f32, f32, f32, i32, vp, sz, vp, vp]),
            "pfkv_paged_decode_attn_noalloc": (i32, [vp, vp, vp, vp, i32, vp, i32, vp, i32, i32, i32, i32,
                                                     i32, i64, f32, f32, f32, i32, i64, vp, vp, vp]),
            "pfkv_paged_decode_attn_scaled": (i32, [vp, vp, vp, vp, i32, vp, vp, vp, i32, vp, i32, i32, i32,
                                                    i32, i32, i64, f32, i32, vp, sz, vp, vp]),
            "pfkv_paged_prefill_workspace_size": (sz, [i32, i32, i32, i32, i32, i32, i32]),
            "pfkv_paged_prefill_attn": (i32, [vp, vp, vp, vp, vp, i32, vp, vp, i32, i32, i32, i32, i32, i64,
                                              i32, i32, f32, f32, f32, i32, vp, sz, vp, vp]),
            "pfkv_mla_decode_workspace_size": (sz, [i32, i32, i32, i32]),
            "pfkv_mla_decode_attn": (i32, [vp, vp, vp, vp, i32, vp, vp, i32, i32, i32, i32, i32, i32,
                                           i64, f32, f32, vp, sz, vp, vp]),
            "pfkv_validate_tables": (i32, [vp, i32, vp, i32, i32, i64, vp, i32, vp, i32, vp, vp]),
            "pfkv_verify_page_tags": (i32, [vp, vp, i32, vp, i32, i32, vp, i64, vp, vp]),
            "pfkv_workspace_status": (i32, [vp, vp, vp]),
            "pfkv_pool_create": (vp, [i64, i32]),
            "pfkv_pool_destroy": (None, [vp]),
            "pfkv_pool_num_free": (i64, [vp]),
            "pfkv_pool_refcount": (i32, [vp, ctypes.c_int32]),
            "pfkv_pool_page_tags": (i32, [vp, vp]),
            "pfkv_pool_map_request": (i32, [vp, vp, i32, vp, vp, i32, vp]),
            "pfkv_pool_release": (i32, [vp, vp, i32]),
            "pfkv_block_hash": (ctypes.c_uint64, [ctypes.c_uint64, vp, i32]),
            "pfkv_slots_from_table": (i32, [vp, i32, i32, i32, i32, vp]),
            "pfkv_selftest_barrier_timeout": (i32, [vp, vp]),
            "pfkv_last_error": (ctypes.c_char_p, []),
            "pfkv_version": (ctypes.c_char_p, []),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
        return _lib


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(fn: str, rc: int):
    if rc != 0:
        raise PfkvError(fn, rc, last_error())


def last_error() -> str:
    return load().pfkv_last_error().decode()


def version() -> str:
    return load().pfkv_version().decode()


# ---------------------------------------------------------------- append
def kv_append_fp8(k_new, v_new, k_cache, v_cache, slot_mapping, k_scale: float, v_scale: float = 1.0,
                  stream=None):
    """Quantise bf16 rows k_new/v_new [T][H][D] to e4m3 and scatter them into
    k_cache/v_cache [pages][H][P][D] (uint8) at slot_mapping [T] (int64).
    For one latent tensor pass v_new = v_cache = None."""
    T, H, D = k_new.shape
    pages, _, P, _ = k_cache.shape
    rc = load().pfkv_kv_append_fp8(_ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                   _ptr(slot_mapping), T, H, D, P, pages, float(k_scale),
                                   float(v_scale), _stream(stream))
    _check("kv_append_fp8", rc)


def kv_append_bf16(k_new, v_new, k_cache, v_cache, slot_mapping, stream=None):
    T, H, D = k_new.shape
    pages, _, P, _ = k_cache.shape
    rc = load().pfkv_kv_append_bf16(_ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                    _ptr(slot_mapping), T, H, D, P, pages, _stream(stream))
    _check("kv_append_bf16", rc)


SCALE_TENSOR = 0
SCALE_HEAD = 1
SCALE_TOKEN = 2


def kv_append_fp8_scaled(k_new, v_new, k_cache, v_cache, slot_mapping, granularity: int, k_scales,
                         v_scales=None, stream=None):
    """kv_append_fp8 with float32 device scales: SCALE_TENSOR [1] / SCALE_HEAD
    [H] are read; SCALE_TOKEN [pages][H][P] receives each appended row's
    scale (its amax / 448)."""
    T, H, D = k_new.shape
    pages, _, P, _ = k_cache.shape
    rc = load().pfkv_kv_append_fp8_scaled(_ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                          _ptr(slot_mapping), T, H, D, P, pages, int(granularity),
                                          _ptr(k_scales), _ptr(v_scales), _stream(stream))
    _check("kv_append_fp8_scaled", rc)


# ---------------------------------------------------------------- decode
def paged_decode_workspace_size(batch: int, num_q_heads: int, num_kv_heads: int, head_dim: int = 128,
                                kv_split_tokens: int = 0, max_total_chunks: int = 0) -> int:
    return int(load().pfkv_paged_decode_workspace_size(batch, num_q_heads, num_kv_heads, head_dim,
                                                       kv_split_tokens, max_total_chunks))


def paged_decode_attn(out, q, k_cache, v_cache, block_tables, context_lens, k_scale: float,
                      v_scale: float, softmax_scale: float, kv_split_tokens: int = 0, workspace=None,
                      lse_out=None, stream=None, max_total_chunks: int = 0):
    """out/q bf16 [B][Hq][D]; caches uint8 (e4m3) or bf16 [pages][Hkv][P][D];
    block_tables int32 [B][max_pages]; context_lens int32 [B].  Returns the
    workspace used (allocated with torch when not given)."""
    import torch
    B, Hq, D = q.shape
    pages, Hkv, P, _ = k_cache.shape
    dt = CACHE_BF16 if k_cache.dtype == torch.bfloat16 else CACHE_FP8_E4M3
    if workspace is None:
        n = paged_decode_workspace_size(B, Hq, Hkv, D, kv_split_tokens, max_total_chunks)
        workspace = torch.empty(n, dtype=torch.uint8, device=q.device)
    rc = load().pfkv_paged_decode_attn(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), dt,
                                       _ptr(block_tables), block_tables.shape[1], _ptr(context_lens), B,
                                       Hq, Hkv, D, P, pages, float(k_scale), float(v_scale),
                                       float(softmax_scale), int(kv_split_tokens), _ptr(workspace),
                                       workspace.numel(), _ptr(lse_out), _stream(stream))
    _check("paged_decode_attn", rc)
    return workspace


def paged_decode_attn_scaled(out, q, k_cache, v_cache, granularity: int, k_scales, v_scales,
                             block_tables, context_lens, softmax_scale: float, kv_split_tokens: int = 0,
                             workspace=None, lse_out=None, stream=None, max_total_chunks: int = 0):
    """paged_decode_attn over an e4m3 cache with float32 device scales of the
    given granularity (SCALE_TENSOR [1], SCALE_HEAD [Hkv], SCALE_TOKEN
    [pages][Hkv][P]).  Returns the workspace used."""
    import torch
    B, Hq, D = q.shape
    pages, Hkv, P, _ = k_cache.shape
    if workspace is None:
        n = paged_decode_workspace_size(B, Hq, Hkv, D, kv_split_tokens, max_total_chunks)
        workspace = torch.empty(n, dtype=torch.uint8, device=q.device)
    rc = load().pfkv_paged_decode_attn_scaled(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                              int(granularity), _ptr(k_scales), _ptr(v_scales),
                                              _ptr(block_tables), block_tables.shape[1],
                                              _ptr(context_lens), B, Hq, Hkv, D, P, pages,
                                              float(softmax_scale), int(kv_split_tokens),
                                              _ptr(workspace), workspace.numel(), _ptr(lse_out),
                                              _stream(stream))
    _check("paged_decode_attn_scaled", rc)
    return workspace


def paged_decode_attn_noalloc(out, q, k_cache, v_cache, block_tables, context_lens, k_scale: float,
                              v_scale: float, softmax_scale: float, kv_split_tokens: int = 0,
                              max_total_chunks: int = 0, lse_out=None, status_out=None, stream=None):
    """paged_decode_attn without a workspace: for callers that cannot allocate
    device memory on the decode path.  The library's fixed 64 MiB device
    scratch is used instead (shared by all calls; order calls that could
    overlap).  status_out: optional int32 device tensor of one element."""
    import torch
    B, Hq, D = q.shape
    pages, Hkv, P, _ = k_cache.shape
    dt = CACHE_BF16 if k_cache.dtype == torch.bfloat16 else CACHE_FP8_E4M3
    rc = load().pfkv_paged_decode_attn_noalloc(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), dt,
                                               _ptr(block_tables), block_tables.shape[1], _ptr(context_lens),
                                               B, Hq, Hkv, D, P, pages, float(k_scale), float(v_scale),
                                               float(softmax_scale), int(kv_split_tokens),
                                               int(max_total_chunks), _ptr(lse_out), _ptr(status_out),
                                               _stream(stream))
    _check("paged_decode_attn_noalloc", rc)


def paged_prefill_workspace_size(batch: int, num_q_heads: int, num_kv_heads: int, max_q_len: int,
                                 max_context_len: int, kv_split_tokens: int = 0, head_dim: int = 128) -> int:
    return int(load().pfkv_paged_prefill_workspace_size(batch, num_q_heads, num_kv_heads, head_dim, max_q_len,
                                                        max_context_len, kv_split_tokens))


def paged_prefill_attn(out, q, k_cache, v_cache, block_tables, context_lens, q_start, max_q_len: int,
                       max_context_len: int, k_scale: float, v_scale: float, softmax_scale: float,
                       kv_split_tokens: int = 0, workspace=None, lse_out=None, stream=None):
    """Several new query tokens per request, causal among themselves: q/out
    bf16 [q_start[B]][Hq][D]; q_start int32 [B+1]; caches uint8 (e4m3)
    [pages][Hkv][P][D].  Returns the workspace used."""
    import torch
    T, Hq, D = q.shape
    pages, Hkv, P, _ = k_cache.shape
    B = context_lens.shape[0]
    if workspace is None:
        n = paged_prefill_workspace_size(B, Hq, Hkv, max_q_len, max_context_len, kv_split_tokens, D)
        workspace = torch.empty(max(n, 256), dtype=torch.uint8, device=q.device)
    rc = load().pfkv_paged_prefill_attn(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                        block_tables.shape[1], _ptr(context_lens), _ptr(q_start), B, Hq, Hkv, D,
                                        P, pages, int(max_q_len), int(max_context_len), float(k_scale),
                                        float(v_scale), float(softmax_scale), int(kv_split_tokens),
                                        _ptr(workspace), workspace.numel(), _ptr(lse_out), _stream(stream))
    _check("paged_prefill_attn", rc)
    return workspace


def mla_decode_workspace_size(batch: int, num_heads: int, d_latent: int = 512, topk: int = 0) -> int:
    return int(load().pfkv_mla_decode_workspace_size(batch, num_heads, d_latent, topk))


def mla_decode_attn(out, q, ckv_cache, block_tables, context_lens, topk_idx, ckv_scale: float,
                    softmax_scale: float, d_latent: int = 512, workspace=None, lse_out=None, stream=None):
    """out bf16 [B][H][d_latent]; q bf16 [B][H][Dqk]; ckv_cache uint8 [pages][P][Dqk];
    topk_idx int32 [B][k] or None."""
    import torch
    B, H, Dqk = q.shape
    pages, P, _ = ckv_cache.shape
    k = 0 if topk_idx is None else topk_idx.shape[1]
    if workspace is None:
        workspace = torch.empty(mla_decode_workspace_size(B, H, d_latent, k), dtype=torch.uint8,
                                device=q.device)
    rc = load().pfkv_mla_decode_attn(_ptr(out), _ptr(q), _ptr(ckv_cache), _ptr(block_tables),
                                     block_tables.shape[1], _ptr(context_lens), _ptr(topk_idx), k, B, H,
                                     d_latent, Dqk - d_latent, P, pages, float(ckv_scale),
                                     float(softmax_scale), _ptr(workspace), workspace.numel(),
                                     _ptr(lse_out), _stream(stream))
    _check("mla_decode_attn", rc)
    return workspace


def validate_tables(block_tables, context_lens, page_size: int, num_pages: int, err_word,
                    topk_idx=None, slot_mapping=None, stream=None):
    B = context_lens.shape[0]
    k = 0 if topk_idx is None else topk_idx.shape[1]
    ns = 0 if slot_mapping is None else slot_mapping.shape[0]
    rc = load().pfkv_validate_tables(_ptr(block_tables), block_tables.shape[1], _ptr(context_lens), B,
                                     page_size, num_pages, _ptr(topk_idx), k, _ptr(slot_mapping), ns,
                                     _ptr(err_word), _stream(stream))
    _check("validate_tables", rc)


def verify_page_tags(block_tables, table_tags, context_lens, page_size: int, page_tags, request_status,
                     stream=None):
    """Page-tag integrity check before decode: request_status[b] (int32, device) receives 0 or an
    OR of REQ_TAG_MISMATCH / REQ_BAD_INDEX.  table_tags (uint32 or int32 bits) has the shape of
    block_tables; page_tags holds one tag per physical page."""
    B = context_lens.shape[0]
    if tuple(table_tags.shape) != tuple(block_tables.shape):
        raise ValueError("table_tags must have the shape of block_tables")
    rc = load().pfkv_verify_page_tags(_ptr(block_tables), _ptr(table_tags), block_tables.shape[1],
                                      _ptr(context_lens), B, page_size, _ptr(page_tags), page_tags.shape[0],
                                      _ptr(request_status), _stream(stream))
    _check("verify_page_tags", rc)


def selftest_barrier_timeout(status, stream=None):
    """Run the bounded-wait self-test; `status` is an int32 device tensor of one element."""
    _check("selftest_barrier_timeout", load().pfkv_selftest_barrier_timeout(_ptr(status), _stream(stream)))


def workspace_status(workspace, stream=None) -> int:
    v = ctypes.c_int32(0)
    rc = load().pfkv_workspace_status(_ptr(workspace), ctypes.byref(v), _stream(stream))
    _check("workspace_status", rc)
    return int(v.value)


# ------------------------------------------------------ page pool (host side)
def _host(a, dtype):
    import numpy as np
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data_as(ctypes.c_void_p)


class PagePool:
    """Host page pool with reference counts, generation tags and a block-hash
    prefix cache (``pfkv_pool_*``).  Arrays are numpy, on the host."""

    def __init__(self, num_pages: int, page_size: int):
        self._h = load().pfkv_pool_create(num_pages, page_size)
        if not self._h:
            raise PfkvError("pool_create", -1, last_error())
        self.num_pages, self.page_size = num_pages, page_size

    def close(self):
        if self._h:
            load().pfkv_pool_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def num_free(self) -> int:
        return int(load().pfkv_pool_num_free(self._h))

    def refcount(self, page: int) -> int:
        return int(load().pfkv_pool_refcount(self._h, page))

    def page_tags(self):
        import numpy as np
        out = np.zeros(self.num_pages, np.uint32)
        _check("pool_page_tags", load().pfkv_pool_page_tags(self._h, out.ctypes.data_as(ctypes.c_void_p)))
        return out

    def map_request(self, tokens, max_pages: int):
        """-> (block-table row int32 [max_pages], tags uint32 [max_pages], cached token count)."""
        import numpy as np
        t, tp = _host(tokens, np.int32)
        row = np.zeros(max_pages, np.int32)
        tags = np.zeros(max_pages, np.uint32)
        cached = ctypes.c_int(0)
        rc = load().pfkv_pool_map_request(self._h, tp, t.shape[0], row.ctypes.data_as(ctypes.c_void_p),
                                          tags.ctypes.data_as(ctypes.c_void_p), max_pages, ctypes.byref(cached))
        _check("pool_map_request", rc)
        return row, tags, int(cached.value)

    def release(self, row, n_pages: int):
        import numpy as np
        r, rp = _host(row, np.int32)
        if not 0 <= n_pages <= r.shape[0]:
            raise ValueError(f"n_pages {n_pages} outside the row's {r.shape[0]} entries")
        _check("pool_release", load().pfkv_pool_release(self._h, rp, n_pages))


def block_hash(parent: int, tokens) -> int:
    import numpy as np
    t, tp = _host(tokens, np.int32)
    return int(load().pfkv_block_hash(ctypes.c_uint64(parent), tp, t.shape[0]))


def slots_from_table(row, page_size: int, first_token: int, n_tokens: int):
    import numpy as np
    r, rp = _host(row, np.int32)
    out = np.zeros(n_tokens, np.int64)
    _check("slots_from_table", load().pfkv_slots_from_table(rp, r.shape[0], page_size, first_token, n_tokens,
                                                            out.ctypes.data_as(ctypes.c_void_p)))
    return out
