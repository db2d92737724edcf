"""Pins for the oracle's per-head and per-token scale granularities (CPU only).

Explainer page, section "FP8 KV のエンジニアリング上の制約": the scaling factor
of an FP8 KV cache can be per tensor, per head or per token, and finer
granularity is more precise.  Pinned here against things other than the
functions themselves:
  - exact round trips: rows made of e4m3 grid values times a power of two
    quantise back to the very same codes, with the power of two as the scale;
  - the per-token rule's defining property: each row's largest magnitude maps
    onto the largest e4m3 value (code 0x7E / 0xFE), and the e4m3 rounding
    error bound holds element by element;
  - reductions to the per-tensor oracle (pinned in its own tests): per-head
    append of one head equals per-tensor append with that head's scale;
    per-token append of rows sharing one amax equals per-tensor append; decode
    with equal scales equals per-tensor decode bit for bit;
  - a dense float64 reference built with torch's float8_e4m3fn decoding and
    scaled_dot_product_attention (no block table, no cache layout);
  - the section's claim itself: on inputs whose magnitudes differ between
    tokens and heads, per-token error < per-head error < per-tensor error.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from synth import gen
from oracle_helpers import oracle_fill_scaled, sdpa_dense

E4M3_MAX_CODE = 0x7E


def _e4m3_codes_no_nan(key, n):
    c = gen.uniform_int(key, np.arange(n, dtype=np.uint64), 0, 253).astype(np.uint8)
    c[c >= 0x7F] += 1  # skip 0x7F (NaN) ; 0xFF is never drawn
    return c


def _torch_e4m3(codes):
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).to(
        torch.float64).numpy()


def _token_rows(T=7, H=3, D=128, spread=20, seed=11):
    """bf16 rows of normal values, each (token, head) row scaled by 2^e."""
    key = gen.make_key(seed, 1)
    x = gen.normal_f32(key, np.arange(T * H * D, dtype=np.uint64)).reshape(T, H, D)
    e = gen.uniform_int(key ^ 7, np.arange(T * H, dtype=np.uint64), -spread, spread).reshape(T, H, 1)
    return gen.f32_to_bf16_bits(np.ldexp(x, e).astype(np.float32))


def test_token_append_grid_round_trip_is_exact():
    # rows = e4m3 grid values x 2^k with one element at +-448 x 2^k: the scale
    # is 2^k exactly and every code comes back unchanged
    T, H, D, P = 6, 2, 64, 16
    codes = _e4m3_codes_no_nan(gen.make_key(5, 2), T * H * D).reshape(T, H, D)
    codes[:, :, 7] = np.where(np.arange(T * H).reshape(T, H) % 2, 0xFE, 0x7E)
    k = gen.uniform_int(gen.make_key(5, 3), np.arange(T * H, dtype=np.uint64), -30, 30).reshape(T, H)
    vals = np.ldexp(_torch_e4m3(codes), k[:, :, None]).astype(np.float32)
    bits = gen.f32_to_bf16_bits(vals)
    assert np.array_equal(gen.bf16_bits_to_f32(bits), vals)  # exact in bf16
    cache = np.zeros((2, H, P, D), np.uint8)
    scales = np.full((2, H, P), np.nan, np.float32)
    slots = np.array([3, 17, 0, 31, 5, 16], np.int64)
    oracle.kv_append_token(bits, cache, scales, slots, P)
    for t, sl in enumerate(slots):
        pg, off = divmod(int(sl), P)
        for h in range(H):
            assert scales[pg, h, off] == np.float32(2.0) ** k[t, h]
            got = cache[pg, h, off]
            want = codes[t, h].copy()
            want[want == 0x80] = 0x80  # -0 stays -0
            assert np.array_equal(got, want), (t, h)


def test_token_append_amax_maps_to_448_and_error_bound():
    T, H, D, P = 9, 3, 128, 16
    bits = _token_rows(T, H, D)
    bits[4, 1, :] = 0  # an all-zero row
    x = gen.bf16_bits_to_f32(bits).astype(np.float64)
    cache = np.zeros((1, H, P, D), np.uint8)
    scales = np.full((1, H, P), np.nan, np.float32)
    slots = np.arange(T, dtype=np.int64) + 2
    oracle.kv_append_token(bits, cache, scales, slots, P)
    for t in range(T):
        for h in range(H):
            s = float(scales[0, h, t + 2])
            c = cache[0, h, t + 2]
            row = x[t, h]
            if not np.any(row):
                assert s == 0.0 and not np.any(c)
                continue
            amax = np.abs(row).max()
            assert s > 0 and abs(s * 448.0 - amax) <= amax * 2.0 ** -23
            i = int(np.argmax(np.abs(row)))
            assert int(c[i]) & 0x7F == E4M3_MAX_CODE
            assert np.all((c & 0x7F) <= E4M3_MAX_CODE)  # never NaN, never above 448
            deq = _torch_e4m3(c) * s
            # e4m3: 3 mantissa bits -> half-ulp 2^-4 relative in the normal range,
            # subnormal step 2^-9 -> absolute 2^-10 (in units of the scale)
            bound = np.maximum(np.abs(row) * 2.0 ** -4, s * 2.0 ** -10) * (1 + 2.0 ** -20)
            assert np.all(np.abs(deq - row) <= bound), (t, h)


def test_token_append_with_shared_amax_equals_per_tensor():
    T, H, D, P = 5, 2, 128, 16
    x = gen.normal_f32(gen.make_key(8, 1), np.arange(T * H * D, dtype=np.uint64)).reshape(T, H, D)
    x = np.clip(x, -3.0, 3.0).astype(np.float32)
    x[:, :, 0] = np.float32(3.5)  # every row's amax is 3.5
    bits = gen.f32_to_bf16_bits(x)
    slots = np.array([0, 1, 2, 20, 21], np.int64)
    ct = np.zeros((2, H, P, D), np.uint8)
    st = np.zeros((2, H, P), np.float32)
    oracle.kv_append_token(bits, ct, st, slots, P)
    cp = np.zeros_like(ct)
    scale = float(np.float32(3.5) / np.float32(448.0))
    oracle.kv_append(bits, cp, slots, P, scale)
    assert np.array_equal(ct, cp)
    for sl in slots:
        pg, off = divmod(int(sl), P)
        assert np.all(st[pg, :, off] == np.float32(scale))


def test_head_append_equals_per_tensor_append_of_each_head():
    T, H, D, P = 6, 4, 128, 16
    bits = _token_rows(T, H, D, spread=3, seed=4)
    hs = np.array([0.01, 0.25, 3.0, 0.0078125], np.float32)
    slots = np.array([5, 6, 40, 7, 41, 0], np.int64)
    ch = np.zeros((3, H, P, D), np.uint8)
    oracle.kv_append_head(bits, ch, slots, P, hs)
    for h in range(H):
        one = np.zeros((3, 1, P, D), np.uint8)
        oracle.kv_append(bits[:, h:h + 1, :], one, slots, P, float(hs[h]))
        assert np.array_equal(ch[:, h], one[:, 0]), h


def _filled(w, gran, spread=6):
    return oracle_fill_scaled(w, gran, spread)


def _workload(**kw):
    base = dict(B=3, Hq=8, Hkv=2, D=128, P=16, context_lens=np.array([5, 40, 77]), seed=3)
    base.update(kw)
    return synth.PagedWorkload("t", **base)


def test_token_decode_with_equal_scales_is_per_tensor_decode():
    w = _workload().set_scales_host()
    shape = (w.num_pages, w.Hkv, w.P, w.D)
    kc = _e4m3_codes_no_nan(gen.make_key(9, 1), int(np.prod(shape))).reshape(shape)
    vc = _e4m3_codes_no_nan(gen.make_key(9, 2), int(np.prod(shape))).reshape(shape)
    ks = np.full(shape[:3], np.float32(w.k_scale), np.float32)
    vs = np.full(shape[:3], np.float32(w.v_scale), np.float32)
    a = oracle.paged_decode_scaled(w.q_bits(), kc, vc, oracle.SCALE_TOKEN, ks, vs, w.block_tables,
                                   w.context_lens, w.P, w.softmax_scale, w.Hkv)
    b = oracle.paged_decode(w.q_bits(), kc, vc, w.block_tables, w.context_lens, w.P, w.k_scale,
                            w.v_scale, w.softmax_scale, w.Hkv)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    t = oracle.paged_decode_scaled(w.q_bits(), kc, vc, oracle.SCALE_TENSOR, ks[:1, 0, 0],
                                   vs[:1, 0, 0], w.block_tables, w.context_lens, w.P,
                                   w.softmax_scale, w.Hkv)
    assert np.array_equal(t[0], b[0]) and np.array_equal(t[1], b[1])


def test_head_decode_is_per_tensor_decode_of_each_head_group():
    w = _workload(Hq=8, Hkv=4)
    kc, vc, ks, vs = _filled(w, oracle.SCALE_HEAD, spread=2)
    out, lse = oracle.paged_decode_scaled(w.q_bits(), kc, vc, oracle.SCALE_HEAD, ks, vs,
                                          w.block_tables, w.context_lens, w.P, w.softmax_scale, w.Hkv)
    for kvh in range(w.Hkv):
        ref, rlse = oracle.paged_decode(w.q_bits(), kc, vc, w.block_tables, w.context_lens, w.P,
                                        float(ks[kvh]), float(vs[kvh]), w.softmax_scale, w.Hkv)
        hs = slice(kvh * w.G, (kvh + 1) * w.G)
        assert np.array_equal(out[:, hs], ref[:, hs]) and np.array_equal(lse[:, hs], rlse[:, hs])


@pytest.mark.parametrize("gran", [1, 2])
def test_scaled_decode_matches_dense_sdpa(gran):
    w = _workload(Hq=8, Hkv=2, context_lens=np.array([1, 33, 120]), shared_requests=2,
                  shared_tokens=0)
    kc, vc, ks, vs = _filled(w, gran)
    out, lse = oracle.paged_decode_scaled(w.q_bits(), kc, vc, gran, ks, vs, w.block_tables,
                                          w.context_lens, w.P, w.softmax_scale, w.Hkv)
    for b in range(w.B):
        L = int(w.context_lens[b])
        t = np.arange(L)
        pages = w.block_tables[b, t // w.P]
        off = t % w.P
        kcodes = kc[pages, :, off]  # [L][Hkv][D]
        vcodes = vc[pages, :, off]
        if gran == oracle.SCALE_TOKEN:
            ksc = ks[pages, :, off].astype(np.float64)[:, :, None]
            vsc = vs[pages, :, off].astype(np.float64)[:, :, None]
        else:
            ksc = ks.astype(np.float64)[None, :, None]
            vsc = vs.astype(np.float64)[None, :, None]
        kd = torch.from_numpy(_torch_e4m3(kcodes) * ksc)
        vd = torch.from_numpy(_torch_e4m3(vcodes) * vsc)
        ref, rlse = sdpa_dense(w.q_bits()[b], kd, vd, w.softmax_scale, w.G)
        np.testing.assert_allclose(out[b], ref, rtol=1e-10, atol=1e-13)
        np.testing.assert_allclose(lse[b], rlse, rtol=1e-10, atol=1e-12)


def test_finer_granularity_is_more_precise():
    # the section's claim, on rows whose magnitudes differ by token and head
    T, H, D, P = 64, 4, 128, 16
    w = _workload(B=1, Hq=4, Hkv=H, context_lens=np.array([T]))
    bits = w.kv_spread_bits("k", 0, 0, T, spread=5)
    x = gen.bf16_bits_to_f32(bits).astype(np.float64)
    sl = w.slots(0, 0, T)
    pg, off = sl // P, sl % P

    def rel_err(codes, scale_tok):  # scale_tok [T][H]
        deq = _torch_e4m3(codes[pg, :, off]) * scale_tok[:, :, None]
        return np.sqrt(np.sum((deq - x) ** 2) / np.sum(x ** 2))

    c = np.zeros((w.num_pages, H, P, D), np.uint8)
    amax = float(gen.bf16_bits_to_f32(bits).__abs__().max())
    s_tensor = float(np.float32(amax) / np.float32(448.0))
    oracle.kv_append(bits, c, sl, P, s_tensor)
    e_tensor = rel_err(c, np.full((T, H), s_tensor))
    hs = (np.abs(gen.bf16_bits_to_f32(bits)).max(axis=(0, 2)) / np.float32(448.0)).astype(np.float32)
    c = np.zeros_like(c)
    oracle.kv_append_head(bits, c, sl, P, hs)
    e_head = rel_err(c, np.broadcast_to(hs.astype(np.float64), (T, H)))
    c = np.zeros_like(c)
    st = np.zeros((w.num_pages, H, P), np.float32)
    oracle.kv_append_token(bits, c, st, sl, P)
    e_token = rel_err(c, st[pg, :, off].astype(np.float64))
    assert e_token < e_head < e_tensor
    assert e_token < 0.05  # about 2^-5 relative for a 3-bit mantissa
