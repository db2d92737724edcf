"""Pins for the oracle's paged attention, split-KV merge and MLA (CPU only).

Independent references: torch.nn.functional.scaled_dot_product_attention in
float64 over dense K/V rebuilt from the token-ordered inputs with torch's
float8_e4m3fn cast (no block table, no cache layout); closed forms; and the
invariants the pages state -- paging is an indirection that does not change
the result, shared prefix pages are the same data as private copies, and
blockwise attention with the (m, l, O) state equals full attention.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from synth import gen
from oracle_helpers import (dense_reference_paged, oracle_fill_mla, oracle_fill_paged,
                            oracle_fill_paged_bf16, sdpa_dense, torch_dequant_fp8)


def _small(B=3, Hq=8, Hkv=2, P=16, lens=(5, 40, 77), num_pages=None, seed=3, **kw):
    w = synth.PagedWorkload("t", B=B, Hq=Hq, Hkv=Hkv, D=128, P=P, context_lens=np.array(lens),
                            num_pages=num_pages, seed=seed, **kw)
    return w.set_scales_host()


@pytest.mark.parametrize("case", [
    dict(),                                                     # GQA G=4, P=16
    dict(Hq=4, Hkv=4, lens=(1, 17, 33)),                        # MHA
    dict(Hq=16, Hkv=2, P=64, lens=(64, 65, 130), seed=5),       # G=8, P=64
    dict(B=2, Hq=2, Hkv=1, lens=(16, 300), num_pages=64),       # spare pool pages
])
def test_paged_decode_matches_dense_sdpa(case):
    w = _small(**case)
    kc, vc = oracle_fill_paged(w)
    out, lse = oracle.paged_decode(w.q_bits(), kc, vc, w.block_tables, w.context_lens, w.P,
                                   w.k_scale, w.v_scale, w.softmax_scale, w.Hkv)
    for b in range(w.B):
        ref, ref_lse = dense_reference_paged(w, b)
        np.testing.assert_allclose(out[b], ref, rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(lse[b], ref_lse, rtol=1e-10, atol=1e-12)


def test_tiny_gqa_workload_matches_dense_sdpa():
    w = synth.workload(synth.TINY_GQA).set_scales_host()
    kc, vc = oracle_fill_paged(w)
    out, lse = oracle.paged_decode(w.q_bits(), kc, vc, w.block_tables, w.context_lens, w.P,
                                   w.k_scale, w.v_scale, w.softmax_scale, w.Hkv)
    for b in range(w.B):
        ref, ref_lse = dense_reference_paged(w, b)
        np.testing.assert_allclose(out[b], ref, rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(lse[b], ref_lse, rtol=1e-10, atol=1e-12)


def _cache_from_codes(kcodes, vcodes, P, perm):
    """kcodes [L][Hkv][D] u8 -> cache pages placed at perm[logical page]."""
    L, Hkv, D = kcodes.shape
    npg = (L + P - 1) // P
    kc = np.zeros((len(perm), Hkv, P, D), np.uint8)
    vc = np.zeros_like(kc)
    for t in range(L):
        kc[perm[t // P], :, t % P, :] = kcodes[t]
        vc[perm[t // P], :, t % P, :] = vcodes[t]
    bt = np.array([perm[:npg]], np.int32)
    return kc, vc, bt


def test_closed_form_single_token_returns_v0():
    D = 128
    rng = np.random.default_rng(1)
    kcodes = rng.integers(0, 0x7E, size=(1, 1, D), dtype=np.uint8)
    vcodes = rng.integers(0, 0x7E, size=(1, 1, D), dtype=np.uint8) | (rng.integers(0, 2, size=(1, 1, D)) << 7).astype(np.uint8)
    kc, vc, bt = _cache_from_codes(kcodes, vcodes, 16, [3, 0, 1, 2])
    q = gen.f32_to_bf16_bits(rng.standard_normal((1, 1, D)).astype(np.float32))
    out, lse = oracle.paged_decode(q, kc, vc, bt, [1], 16, 0.5, 0.25, 0.1, 1)
    tab = oracle.e4m3_table()
    np.testing.assert_array_equal(out[0, 0], tab[vcodes[0, 0]] * 0.25)
    s = float(np.float32(0.1)) * float(np.dot(gen.bf16_bits_to_f32(q[0, 0]).astype(np.float64), tab[kcodes[0, 0]] * 0.5))
    assert lse[0, 0] == pytest.approx(s, rel=1e-14, abs=1e-14)


def test_closed_form_identical_keys_give_mean_of_values():
    D, L = 128, 37
    rng = np.random.default_rng(2)
    krow = rng.integers(0, 0x7E, size=(1, D), dtype=np.uint8)
    kcodes = np.repeat(krow[None], L, axis=0)
    vcodes = rng.integers(0, 0x7E, size=(L, 1, D), dtype=np.uint8)
    kc, vc, bt = _cache_from_codes(kcodes, vcodes, 16, [2, 0, 1])
    q = gen.f32_to_bf16_bits(rng.standard_normal((1, 1, D)).astype(np.float32))
    out, _ = oracle.paged_decode(q, kc, vc, bt, [L], 16, 1.0, 1.0, 0.3, 1)
    tab = oracle.e4m3_table()
    np.testing.assert_allclose(out[0, 0], tab[vcodes[:, 0, :]].mean(axis=0), rtol=1e-13)


def test_closed_form_two_tokens_logistic_weights():
    D = 128
    kcodes = np.zeros((2, 1, D), np.uint8)
    kcodes[0, 0, 0] = 0x40  # 2.0
    kcodes[1, 0, 0] = 0x38  # 1.0
    vcodes = np.zeros((2, 1, D), np.uint8)
    vcodes[0] = 0x38  # 1.0 everywhere
    vcodes[1] = 0x40  # 2.0 everywhere
    kc, vc, bt = _cache_from_codes(kcodes, vcodes, 16, [0])
    q = np.zeros((1, 1, D), np.uint16)
    q[0, 0, 0] = 0x3F80  # bf16 1.0
    out, lse = oracle.paged_decode(q, kc, vc, bt, [2], 16, 1.0, 1.0, 0.5, 1)
    # s0 = 0.5 * 2 = 1.0, s1 = 0.5 * 1 = 0.5
    w1 = 1.0 / (1.0 + math.exp(0.5))
    expect = (1 - w1) * 1.0 + w1 * 2.0
    np.testing.assert_allclose(out[0, 0], expect, rtol=1e-14)
    assert lse[0, 0] == pytest.approx(math.log(math.e + math.exp(0.5)), rel=1e-14)


def test_closed_form_dominant_score_selects_its_row():
    D, L = 128, 50
    rng = np.random.default_rng(4)
    kcodes = np.zeros((L, 1, D), np.uint8)
    kcodes[17, 0, :] = 0x7E  # 448 everywhere: overwhelmingly largest score
    vcodes = rng.integers(0, 0x7E, size=(L, 1, D), dtype=np.uint8)
    kc, vc, bt = _cache_from_codes(kcodes, vcodes, 16, [1, 3, 0, 2])
    q = np.full((1, 1, D), 0x3F80, np.uint16)
    out, _ = oracle.paged_decode(q, kc, vc, bt, [L], 16, 1.0, 1.0, 1.0, 1)
    tab = oracle.e4m3_table()
    np.testing.assert_allclose(out[0, 0], tab[vcodes[17, 0]], rtol=1e-12)


def test_output_invariant_under_physical_page_permutation():
    w1 = _small(lens=(45, 100, 3), seed=11)
    w2 = _small(lens=(45, 100, 3), seed=11, num_pages=40)  # bigger pool, other permutation
    assert not np.array_equal(w1.block_tables[:, :2], w2.block_tables[:, :2])
    outs = []
    for w in (w1, w2):
        kc, vc = oracle_fill_paged(w)
        outs.append(oracle.paged_decode(w.q_bits(), kc, vc, w.block_tables, w.context_lens, w.P,
                                        w.k_scale, w.v_scale, w.softmax_scale, w.Hkv))
    np.testing.assert_array_equal(outs[0][0], outs[1][0])
    np.testing.assert_array_equal(outs[0][1], outs[1][1])


def test_shared_prefix_pages_equal_private_copies():
    lens = (70, 90, 51)
    shared = _small(lens=lens, shared_requests=3, shared_tokens=48, seed=9)
    assert np.all(shared.block_tables[1:, :3] == shared.block_tables[0, :3])
    kc, vc = oracle_fill_paged(shared)
    out_s, lse_s = oracle.paged_decode(shared.q_bits(), kc, vc, shared.block_tables, shared.context_lens,
                                       shared.P, shared.k_scale, shared.v_scale, shared.softmax_scale,
                                       shared.Hkv)
    # private copies: same token values, every request owning its own pages
    priv = _small(lens=lens, seed=9)
    priv.kv_bits = shared.kv_bits
    priv.k_scale, priv.v_scale = shared.k_scale, shared.v_scale
    assert len(set(priv.block_tables[:, :3].ravel().tolist())) == 9
    kc2, vc2 = oracle_fill_paged(priv)
    out_p, lse_p = oracle.paged_decode(priv.q_bits(), kc2, vc2, priv.block_tables, priv.context_lens,
                                       priv.P, priv.k_scale, priv.v_scale, priv.softmax_scale, priv.Hkv)
    np.testing.assert_array_equal(out_s, out_p)
    np.testing.assert_array_equal(lse_s, lse_p)


@pytest.mark.parametrize("chunk", [1, 7, 16, 64, 4096])
def test_split_kv_merge_equals_full_attention(chunk):
    w = _small(lens=(1, 130, 300), seed=12)
    kc, vc = oracle_fill_paged(w)
    q = w.q_bits()
    for b in range(w.B):
        L = int(w.context_lens[b])
        for h in (0, 5):
            full, lf = oracle.paged_decode_one(q[b, h], kc, vc, w.block_tables[b], L, h // w.G, w.P,
                                               w.k_scale, w.v_scale, w.softmax_scale)
            split, ls = oracle.paged_decode_one(q[b, h], kc, vc, w.block_tables[b], L, h // w.G, w.P,
                                                w.k_scale, w.v_scale, w.softmax_scale, chunk=chunk)
            np.testing.assert_allclose(split, full, rtol=1e-12, atol=1e-14)
            assert ls == pytest.approx(lf, rel=1e-12, abs=1e-13)


def test_empty_context_gives_zeros_and_minus_inf():
    w = _small(lens=(0, 20, 0))
    kc, vc = oracle_fill_paged(w)
    out, lse = oracle.paged_decode(w.q_bits(), kc, vc, w.block_tables, w.context_lens, w.P,
                                   w.k_scale, w.v_scale, w.softmax_scale, w.Hkv)
    assert np.all(out[0] == 0) and np.all(out[2] == 0)
    assert np.all(np.isneginf(lse[0])) and np.all(np.isneginf(lse[2]))
    assert np.all(np.isfinite(lse[1]))


def test_bad_page_id_is_an_error_not_a_read():
    w = _small()
    kc, vc = oracle_fill_paged(w)
    bt = w.block_tables.copy()
    bt[1, 1] = w.num_pages + 5
    with pytest.raises(oracle.OracleError):
        oracle.paged_decode(w.q_bits(), kc, vc, bt, w.context_lens, w.P, w.k_scale, w.v_scale,
                            w.softmax_scale, w.Hkv)


def test_bf16_cache_matches_dense_sdpa():
    w = _small(lens=(9, 33, 64), seed=21)
    kc, vc = oracle_fill_paged_bf16(w)
    out, lse = oracle.paged_decode(w.q_bits(), kc, vc, w.block_tables, w.context_lens, w.P,
                                   1.0, 1.0, w.softmax_scale, w.Hkv)
    for b in range(w.B):
        L = int(w.context_lens[b])
        kd = torch.from_numpy(gen.bf16_bits_to_f32(w.kv_bits("k", b, 0, L)).astype(np.float64))
        vd = torch.from_numpy(gen.bf16_bits_to_f32(w.kv_bits("v", b, 0, L)).astype(np.float64))
        ref, ref_lse = sdpa_dense(w.q_bits()[b], kd, vd, w.softmax_scale, w.G)
        np.testing.assert_allclose(out[b], ref, rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(lse[b], ref_lse, rtol=1e-10, atol=1e-12)


# ------------------------------------------------------------------------ MLA
def _mla_small(topk_n=0, lens=(70, 130), H=4, seed=2):
    m = synth.MlaWorkload("m", B=len(lens), H=H, context_lens=np.array(lens), topk_n=topk_n, P=64,
                          seed=seed)
    return m.set_scales_host()


def _mla_dense_ref(m, b, tokens):
    rows = m.ckv_rows_bits(b, tokens)  # [n][576]
    cd = torch_dequant_fp8(rows, m.ckv_scale)  # float64 [n][576]
    q = torch.from_numpy(gen.bf16_bits_to_f32(m.q_bits()[b]).astype(np.float64))  # [H][576]
    out = torch.nn.functional.scaled_dot_product_attention(
        q[:, None, :], cd[None].expand(m.H, -1, -1), cd[None, :, : m.Dv].expand(m.H, -1, -1),
        scale=m.softmax_scale)[:, 0, :]
    lse = torch.logsumexp((q @ cd.T) * m.softmax_scale, dim=1)
    return out.numpy(), lse.numpy()


def test_mla_all_tokens_matches_dense_sdpa():
    m = _mla_small()
    cache = oracle_fill_mla(m)
    out, lse = oracle.mla_decode(m.q_bits(), cache, m.block_tables, m.context_lens, None, m.P, m.Dv,
                                 m.ckv_scale, m.softmax_scale)
    for b in range(m.B):
        ref, ref_lse = _mla_dense_ref(m, b, np.arange(int(m.context_lens[b])))
        np.testing.assert_allclose(out[b], ref, rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(lse[b], ref_lse, rtol=1e-10, atol=1e-12)


def test_mla_topk_matches_dense_sdpa_over_selected_rows():
    m = _mla_small(topk_n=32, lens=(100, 257))
    cache = oracle_fill_mla(m)
    out, lse = oracle.mla_decode(m.q_bits(), cache, m.block_tables, m.context_lens, m.topk, m.P, m.Dv,
                                 m.ckv_scale, m.softmax_scale)
    for b in range(m.B):
        assert len(np.unique(m.topk[b])) == 32 and np.all(np.diff(m.topk[b]) > 0)
        ref, ref_lse = _mla_dense_ref(m, b, m.topk[b])
        np.testing.assert_allclose(out[b], ref, rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(lse[b], ref_lse, rtol=1e-10, atol=1e-12)


def test_mla_topk_of_every_position_equals_no_topk_and_padding_is_skipped():
    m = _mla_small(lens=(64, 90))
    cache = oracle_fill_mla(m)
    full, _ = oracle.mla_decode(m.q_bits(), cache, m.block_tables, m.context_lens, None, m.P, m.Dv,
                                m.ckv_scale, m.softmax_scale)
    tk = np.full((2, 100), -1, np.int32)
    tk[0, :64] = np.arange(64)
    tk[1, 10:100] = np.arange(90)
    listed, _ = oracle.mla_decode(m.q_bits(), cache, m.block_tables, m.context_lens, tk, m.P, m.Dv,
                                  m.ckv_scale, m.softmax_scale)
    np.testing.assert_array_equal(full, listed)


def test_mla_topk_beyond_context_is_an_error():
    m = _mla_small(lens=(64, 90))
    cache = oracle_fill_mla(m)
    tk = np.array([[0, 64], [1, 2]], np.int32)
    with pytest.raises(oracle.OracleError):
        oracle.mla_decode(m.q_bits(), cache, m.block_tables, m.context_lens, tk, m.P, m.Dv,
                          m.ckv_scale, m.softmax_scale)
