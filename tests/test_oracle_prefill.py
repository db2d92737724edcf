"""Pins for the oracle's multi-query (chunked prefill / verification) attention.

Explainer page: chunked prefill ("チャンク分割と、その大きさの決め方") processes
a prompt in chunks whose tokens attend the cached prefix and, causally, each
other; speculative decoding's verification checks gamma+1 drafted positions in
one forward pass.  Pinned against:
  - float64 scaled_dot_product_attention with an explicit causal mask over
    dense K/V rebuilt from the token-ordered inputs with torch's fp8 cast (no
    block table, no cache layout);
  - the decode oracle (pinned in its own tests): one new token is decode, and
    the last new token attends exactly the whole context;
  - causality: changing the newest token's K/V changes no earlier query's row.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from oracle_helpers import oracle_fill_paged, torch_dequant_fp8
from synth import gen


def _w(Hq=8, Hkv=2, lens=(9, 40, 77), n_new=5, P=16, seed=4):
    w = synth.PagedWorkload("pf", B=len(lens), Hq=Hq, Hkv=Hkv, D=128, P=P, context_lens=np.array(lens),
                            n_new=n_new, seed=seed)
    return w.set_scales_host()


def _prefill(w, kc, vc, q_lens=None):
    return oracle.paged_prefill(w.q_new_bits(q_lens), kc, vc, w.block_tables, w.context_lens,
                                w.q_start(q_lens), w.P, w.k_scale, w.v_scale, w.softmax_scale, w.Hkv)


@pytest.mark.parametrize("case", [dict(), dict(Hq=4, Hkv=4, lens=(16, 17, 64), n_new=16),
                                  dict(Hq=16, Hkv=1, lens=(8, 100), n_new=8, P=64)])
def test_prefill_matches_dense_causal_sdpa(case):
    w = _w(**case)
    kc, vc = oracle_fill_paged(w)
    out, lse = _prefill(w, kc, vc)
    q = w.q_new_bits()
    for b in range(w.B):
        L = int(w.context_lens[b])
        n = w.n_new
        kd = torch_dequant_fp8(w.kv_bits("k", b, 0, L), w.k_scale)  # [L][Hkv][D]
        vd = torch_dequant_fp8(w.kv_bits("v", b, 0, L), w.v_scale)
        k = kd.permute(1, 0, 2).repeat_interleave(w.G, dim=0)  # [Hq][L][D]
        v = vd.permute(1, 0, 2).repeat_interleave(w.G, dim=0)
        qb = torch.from_numpy(gen.bf16_bits_to_f32(q[b * n:(b + 1) * n]).astype(np.float64))
        qb = qb.permute(1, 0, 2)  # [Hq][n][D]
        pos = torch.arange(L - n, L)[:, None]
        mask = torch.arange(L)[None, :] <= pos  # [n][L], True = attend
        ref = torch.nn.functional.scaled_dot_product_attention(qb, k, v, attn_mask=mask,
                                                               scale=float(w.softmax_scale))
        s = torch.einsum("hnd,hld->hnl", qb, k) * float(w.softmax_scale)
        ref_lse = torch.logsumexp(s.masked_fill(~mask, -float("inf")), dim=2)
        np.testing.assert_allclose(out[b * n:(b + 1) * n], ref.permute(1, 0, 2).numpy(), rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(lse[b * n:(b + 1) * n], ref_lse.permute(1, 0).numpy(), rtol=1e-10, atol=1e-12)


def test_one_new_token_is_decode_and_last_token_sees_everything():
    w = _w(n_new=6)
    kc, vc = oracle_fill_paged(w)
    out, lse = _prefill(w, kc, vc)
    q = w.q_new_bits()
    last = q[w.n_new - 1::w.n_new]  # [B][Hq][D]: each request's newest query
    ref, ref_lse = oracle.paged_decode(last, kc, vc, w.block_tables, w.context_lens, w.P, w.k_scale,
                                       w.v_scale, w.softmax_scale, w.Hkv)
    assert np.array_equal(out[w.n_new - 1::w.n_new], ref)
    assert np.array_equal(lse[w.n_new - 1::w.n_new], ref_lse)
    ones = np.ones(w.B, np.int64)
    o1, l1 = _prefill(w, kc, vc, ones)
    d1, dl1 = oracle.paged_decode(w.q_new_bits(ones), kc, vc, w.block_tables, w.context_lens, w.P,
                                  w.k_scale, w.v_scale, w.softmax_scale, w.Hkv)
    assert np.array_equal(o1, d1) and np.array_equal(l1, dl1)


def test_newest_token_does_not_reach_earlier_queries():
    w = _w(n_new=4)
    kc, vc = oracle_fill_paged(w)
    out, lse = _prefill(w, kc, vc)
    kc2, vc2 = kc.copy(), vc.copy()
    for b in range(w.B):
        sl = int(w.slots(b, int(w.context_lens[b]) - 1, int(w.context_lens[b]))[0])
        kc2[sl // w.P, :, sl % w.P] ^= 0x21
        vc2[sl // w.P, :, sl % w.P] ^= 0x12
    out2, lse2 = _prefill(w, kc2, vc2)
    n = w.n_new
    for b in range(w.B):
        assert np.array_equal(out[b * n:b * n + n - 1], out2[b * n:b * n + n - 1])
        assert not np.array_equal(out[b * n + n - 1], out2[b * n + n - 1])


def test_varlen_queries_and_errors():
    w = _w(n_new=8, lens=(8, 40, 77))
    kc, vc = oracle_fill_paged(w)
    ql = np.array([8, 0, 3])
    out, lse = _prefill(w, kc, vc, ql)
    assert out.shape[0] == 11
    full, flse = _prefill(w, kc, vc)
    # request 2's 3 newest queries are the last 3 of its 8
    assert np.array_equal(out[8:11], full[16 + 5:24])
    with pytest.raises(oracle.OracleError):  # more queries than context (request 0 holds 8)
        oracle.paged_prefill(np.zeros((9, 8, 128), np.uint16), kc, vc, w.block_tables, w.context_lens,
                             np.array([0, 9, 9, 9]), w.P, w.k_scale, w.v_scale, w.softmax_scale, w.Hkv)
