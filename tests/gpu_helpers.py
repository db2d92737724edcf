"""Helpers for the GPU parity tests: run the product path through the C ABI
(via the thin binding) and build the oracle's expectations from the same seeded
inputs.  No oracle input comes from the GPU: the oracle re-encodes the host
generator's bf16 rows itself, and the GPU cache bytes are compared with the
oracle's bytes."""
from __future__ import annotations

import numpy as np

import oracle

TOL_REL = 2e-3
TOL_ABS = 1e-3


def pf():
    import paged_fp8_kv_02_gb300 as m
    m.load()
    return m


def bf16_half_ulp(ref):
    """Half a bf16 unit in the last place at |ref|: the rounding every bf16
    output carries even when its fp32 value is exact."""
    a = np.abs(np.asarray(ref, np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.exp2(e - 8), 0.0)


def assert_within_tolerance(got, ref, what=""):
    """Per element |err| <= 2e-3 * max|ref| + 1e-3 (+ half a bf16 ulp of ref for
    the bf16 output format), with max|ref| taken over the whole compared
    reference (a scalar, as the bound is stated)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    bound = TOL_REL * np.abs(ref).max() + TOL_ABS + bf16_half_ulp(ref)
    err = np.abs(got - ref)
    bad = err > bound
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {int(bad.sum())} elements outside tolerance; worst excess "
                             f"{float((err - bound).max()):.3e}; first at {idx.tolist()}")


def append_fp8_fn(p, w):
    return lambda k, v, kc, vc, s: p.kv_append_fp8(k, v, kc, vc, s, w.k_scale, w.v_scale)


def append_bf16_fn(p):
    return lambda k, v, kc, vc, s: p.kv_append_bf16(k, v, kc, vc, s)


def oracle_caches(w, bf16=False):
    """Full caches built by the oracle from the host generator (all tokens)."""
    shape = (w.num_pages, w.Hkv, w.P, w.D)
    kc = np.zeros(shape, np.uint16 if bf16 else np.uint8)
    vc = np.zeros_like(kc)
    for b in range(w.B):
        t0, _ = w.prefill_range(b)
        t1 = int(w.context_lens[b])
        if t1 <= t0:
            continue
        sl = w.slots(b, t0, t1)
        if bf16:
            oracle.kv_append_bf16(w.kv_bits("k", b, t0, t1), kc, sl, w.P)
            oracle.kv_append_bf16(w.kv_bits("v", b, t0, t1), vc, sl, w.P)
        else:
            oracle.kv_append(w.kv_bits("k", b, t0, t1), kc, sl, w.P, w.k_scale)
            oracle.kv_append(w.kv_bits("v", b, t0, t1), vc, sl, w.P, w.v_scale)
    return kc, vc


def gpu_pages_of(cache_dev, bt_row, kvh, L, P):
    """Rows t < L of one KV head of one request, gathered from a device cache
    through its block table -> host array [L][D]."""
    import torch
    npg = (L + P - 1) // P
    pages = torch.as_tensor(bt_row[:npg].astype(np.int64), device=cache_dev.device)
    rows = cache_dev[:, kvh].index_select(0, pages)  # [npg][P][D], this head only
    if rows.dtype == torch.bfloat16:
        rows = rows.view(torch.int16)
    return rows.reshape(npg * P, -1)[:L].cpu().numpy()


def oracle_one_head(w, b, kvh, bf16=False):
    """Oracle K/V rows [L][D] of one (request, KV head), encoded by the oracle
    from the host generator, in a private contiguous mini cache."""
    L = int(w.context_lens[b])
    P = w.P
    npg = (L + P - 1) // P
    kc = np.zeros((max(npg, 1), 1, P, w.D), np.uint16 if bf16 else np.uint8)
    vc = np.zeros_like(kc)
    slots = np.arange(L, dtype=np.int64)
    kb = w.kv_head_bits("k", b, kvh, 0, L)[:, None, :]
    vb = w.kv_head_bits("v", b, kvh, 0, L)[:, None, :]
    if bf16:
        oracle.kv_append_bf16(kb, kc, slots, P)
        oracle.kv_append_bf16(vb, vc, slots, P)
    else:
        oracle.kv_append(kb, kc, slots, P, w.k_scale)
        oracle.kv_append(vb, vc, slots, P, w.v_scale)
    return kc, vc, np.arange(max(npg, 1), dtype=np.int32)


def oracle_one_head_token(w, b, kvh):
    """As oracle_one_head for per-token scales: the oracle's codes and scales
    of one (request, KV head) in a private mini cache, plus its block-table row."""
    L = int(w.context_lens[b])
    P = w.P
    npg = max((L + P - 1) // P, 1)
    kc = np.zeros((npg, 1, P, w.D), np.uint8)
    vc = np.zeros_like(kc)
    ks = np.zeros((npg, 1, P), np.float32)
    vs = np.zeros_like(ks)
    slots = np.arange(L, dtype=np.int64)
    oracle.kv_append_token(w.kv_head_bits("k", b, kvh, 0, L)[:, None, :], kc, ks, slots, P)
    oracle.kv_append_token(w.kv_head_bits("v", b, kvh, 0, L)[:, None, :], vc, vs, slots, P)
    return kc, vc, ks, vs, np.arange(npg, dtype=np.int32)


def gpu_scales_of(scales_dev, bt_row, kvh, L, P):
    """Per-token scales t < L of one KV head of one request -> host float32 [L]."""
    import torch
    npg = (L + P - 1) // P
    pages = torch.as_tensor(bt_row[:npg].astype(np.int64), device=scales_dev.device)
    return scales_dev.index_select(0, pages)[:, kvh].reshape(-1)[:L].cpu().numpy()


def to_np_bf16(t):
    import torch
    return t.float().cpu().numpy().astype(np.float64) if t.dtype == torch.bfloat16 else t.cpu().numpy()
