"""Host-side helpers for tests: fill caches through the oracle, and build the
independent dense reference (torch casts + scaled_dot_product_attention)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from synth import gen


def oracle_fill_paged(w, include_new=True):
    """K/V caches [pages][Hkv][P][D] (u8) filled by the oracle's append:
    every prefill token, then (optionally) the step's new tokens."""
    shape = (w.num_pages, w.Hkv, w.P, w.D)
    kc = np.zeros(shape, np.uint8)
    vc = np.zeros(shape, np.uint8)
    for b in range(w.B):
        t0, t1 = w.prefill_range(b)
        if include_new:
            t1 = int(w.context_lens[b])
        if t1 <= t0:
            continue
        sl = w.slots(b, t0, t1)
        oracle.kv_append(w.kv_bits("k", b, t0, t1), kc, sl, w.P, w.k_scale)
        oracle.kv_append(w.kv_bits("v", b, t0, t1), vc, sl, w.P, w.v_scale)
    return kc, vc


def oracle_fill_paged_bf16(w):
    shape = (w.num_pages, w.Hkv, w.P, w.D)
    kc = np.zeros(shape, np.uint16)
    vc = np.zeros(shape, np.uint16)
    for b in range(w.B):
        t0, _ = w.prefill_range(b)
        t1 = int(w.context_lens[b])
        sl = w.slots(b, t0, t1)
        oracle.kv_append_bf16(w.kv_bits("k", b, t0, t1), kc, sl, w.P)
        oracle.kv_append_bf16(w.kv_bits("v", b, t0, t1), vc, sl, w.P)
    return kc, vc


def oracle_fill_mla(m):
    cache = np.zeros((m.num_pages, m.P, m.Dqk), np.uint8)
    for b in range(m.B):
        L = int(m.context_lens[b])
        oracle.kv_append(m.ckv_bits(b, 0, L), cache.reshape(m.num_pages, 1, m.P, m.Dqk),
                         m.slots(b, 0, L), m.P, m.ckv_scale)
    return cache


# ------------------------------------------------------- scale granularities
def spread_rows(w, which, b, t0, t1, spread=6, zero_rows=False):
    """bf16 rows [t1-t0][Hkv][D] whose magnitudes vary by token and head
    (PagedWorkload.kv_spread_bits); zero_rows also blanks every 13th token of
    head 0 (K) or every 11th (V) so that all-zero rows occur."""
    x = w.kv_spread_bits(which, b, t0, t1, spread)
    if zero_rows:
        t = np.arange(t0, t1)
        x[(t % (13 if which == "k" else 11)) == 0, 0, :] = 0
    return x


def spread_scales(w, gran, spread=6, zero_rows=False):
    """Per-tensor [1] or per-head [Hkv] scales (amax / 448 in fp32) of the
    spread rows of every attended token of w; None for per-token."""
    if gran == oracle.SCALE_TOKEN:
        return None, None
    out = []
    for which in ("k", "v"):
        m = np.zeros(w.Hkv, np.float32)
        for b in range(w.B):
            L = int(w.context_lens[b])
            t0 = w.shared_tokens if 0 < b < w.shared_requests else 0
            if L > t0:
                x = np.abs(gen.bf16_bits_to_f32(spread_rows(w, which, b, t0, L, spread, zero_rows)))
                m = np.maximum(m, x.max(axis=(0, 2)))
        if gran == oracle.SCALE_TENSOR:
            m = np.array([m.max()], np.float32)
        out.append((m / np.float32(448.0)).astype(np.float32))
    return out[0], out[1]


def oracle_fill_scaled(w, gran, spread=6, zero_rows=False):
    """Caches [pages][Hkv][P][D] (u8) and scales of w filled by the oracle at
    granularity gran from the spread rows: (kc, vc, ks, vs)."""
    shape = (w.num_pages, w.Hkv, w.P, w.D)
    kc, vc = np.zeros(shape, np.uint8), np.zeros(shape, np.uint8)
    ks, vs = spread_scales(w, gran, spread, zero_rows)
    if gran == oracle.SCALE_TOKEN:
        ks = np.zeros(shape[:3], np.float32)
        vs = np.zeros(shape[:3], np.float32)
    for b in range(w.B):
        L = int(w.context_lens[b])
        t0 = w.shared_tokens if 0 < b < w.shared_requests else 0
        if L <= t0:
            continue
        sl = w.slots(b, t0, L)
        kb = spread_rows(w, "k", b, t0, L, spread, zero_rows)
        vb = spread_rows(w, "v", b, t0, L, spread, zero_rows)
        if gran == oracle.SCALE_TOKEN:
            oracle.kv_append_token(kb, kc, ks, sl, w.P)
            oracle.kv_append_token(vb, vc, vs, sl, w.P)
        elif gran == oracle.SCALE_HEAD:
            oracle.kv_append_head(kb, kc, sl, w.P, ks)
            oracle.kv_append_head(vb, vc, sl, w.P, vs)
        else:
            oracle.kv_append(kb, kc, sl, w.P, float(ks[0]))
            oracle.kv_append(vb, vc, sl, w.P, float(vs[0]))
    return kc, vc, ks, vs


# ------------------------------------------------------------- dense reference
def torch_dequant_fp8(x_bits, scale):
    """fp32(x) / scale (IEEE fp32) cast by torch to float8_e4m3fn, back to float64 x scale."""
    x = gen.bf16_bits_to_f32(x_bits)
    y = (x / np.float32(scale)).astype(np.float32)
    # amax / (amax / 448) can land a few fp32 ulps above 448; below 464 the
    # nearest e4m3 value is still 448, where torch's cast and saturation agree.
    assert np.all(np.abs(y) < 464.0)
    f8 = torch.from_numpy(y).to(torch.float8_e4m3fn)
    return f8.to(torch.float64) * float(scale)


def sdpa_dense(q_bits, k_dense, v_dense, softmax_scale, G):
    """q [Hq][D] bf16 bits, k/v [L][Hkv][D] float64 -> out [Hq][Dv], lse [Hq]."""
    q = torch.from_numpy(gen.bf16_bits_to_f32(q_bits).astype(np.float64))
    k = k_dense.permute(1, 0, 2).repeat_interleave(G, dim=0)  # [Hq][L][D]
    v = v_dense.permute(1, 0, 2).repeat_interleave(G, dim=0)
    out = torch.nn.functional.scaled_dot_product_attention(
        q[:, None, :], k, v, scale=float(softmax_scale))[:, 0, :]
    s = torch.einsum("hd,hld->hl", q, k) * float(softmax_scale)
    lse = torch.logsumexp(s, dim=1)
    return out.numpy(), lse.numpy()


def dense_reference_paged(w, b):
    """Dense (unpaged) reference for request b, built from the token-ordered
    inputs -- no block table, no cache layout involved."""
    L = int(w.context_lens[b])
    kd = torch_dequant_fp8(w.kv_bits("k", b, 0, L), w.k_scale)
    vd = torch_dequant_fp8(w.kv_bits("v", b, 0, L), w.v_scale)
    return sdpa_dense(w.q_bits()[b], kd, vd, w.softmax_scale, w.G)
