"""paged_prefill_attn (several new query tokens per request, causal among them)
on the GPU against the oracle.

Small cases: caches encoded by the oracle from the host generator are
uploaded and every output row is compared with the oracle (tolerance
|err| <= 2e-3 * max|ref| + 1e-3 + half a bf16 ulp; lse to 2e-5 relative).
Full size: the long split-KV workload's cache is filled through the product's append from the
device generator, its 8 appended tokens per request are the queries, and
sampled (request, query, head) rows are recomputed by the oracle from the
host generator in a private cache whose bytes are checked against the GPU's."""
import numpy as np
import pytest

import oracle
import synth

from gpu_helpers import (append_fp8_fn, assert_within_tolerance, gpu_pages_of, oracle_one_head, pf,
                         to_np_bf16)
from oracle_helpers import oracle_fill_paged

pytestmark = pytest.mark.gpu


def _dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda")


def _dev_bits(bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to("cuda").view(torch.bfloat16)


def _run(p, w, kc, vc, q_lens=None, split=0, max_q=None, max_ctx=None, bt=None, ctx=None):
    import torch
    qs = w.q_start(q_lens)
    q = _dev_bits(w.q_new_bits(q_lens))
    out = torch.zeros_like(q)
    lse = torch.full((q.shape[0], w.Hq), float("nan"), dtype=torch.float32, device="cuda")
    max_q = max_q or max(int(np.diff(qs).max(initial=1)), 1)
    max_ctx = max_ctx or int(w.context_lens.max())
    ws = p.paged_prefill_attn(out, q, kc, vc, _dev(w.block_tables if bt is None else bt),
                              _dev(w.context_lens if ctx is None else ctx), _dev(qs), max_q, max_ctx,
                              w.k_scale, w.v_scale, w.softmax_scale, kv_split_tokens=split, lse_out=lse)
    torch.cuda.synchronize()
    return to_np_bf16(out), lse.cpu().numpy(), p.workspace_status(ws)


def _check_small(w, q_lens=None, split=0, **kw):
    p = pf()
    w.set_scales_host()
    kc, vc = oracle_fill_paged(w)
    out, lse, status = _run(p, w, _dev(kc), _dev(vc), q_lens, split, **kw)
    assert status == 0
    ref, ref_lse = oracle.paged_prefill(w.q_new_bits(q_lens), kc, vc, w.block_tables, w.context_lens,
                                        w.q_start(q_lens), w.P, w.k_scale, w.v_scale, w.softmax_scale, w.Hkv)
    if ref.shape[0]:
        assert_within_tolerance(out, ref, f"{w.name} split {split}")
        np.testing.assert_allclose(lse, ref_lse, rtol=2e-5, atol=2e-4)


def _w(name, Hq, Hkv, lens, n_new, P=16, seed=31):
    return synth.PagedWorkload(name, B=len(lens), Hq=Hq, Hkv=Hkv, D=128, P=P, context_lens=np.array(lens),
                               n_new=n_new, seed=seed)


@pytest.mark.parametrize("split", [0, 64, 192])
def test_gqa_verification_sized(split):
    _check_small(_w("g8", 16, 2, (9, 40, 77, 300), n_new=5), split=split)


@pytest.mark.parametrize("split", [0, 128])
def test_mha_two_row_blocks(split):
    # G = 1: 128 query tokens per row block, 200 new tokens -> two blocks
    _check_small(_w("mha", 4, 4, (200, 250, 333), n_new=200), split=split)


def test_group16_page64_long():
    _check_small(_w("g16", 16, 1, (8, 100, 700), n_new=8, P=64), split=128)


def test_whole_prompt_is_new():
    # prefill from an empty cache: n_b = L_b
    w = _w("fresh", 8, 2, (1, 65, 130), n_new=1)
    _check_small(w, q_lens=np.array([1, 65, 130]))


def test_varlen_queries_including_none():
    w = _w("varlen", 8, 2, (40, 16, 77, 5), n_new=1)
    _check_small(w, q_lens=np.array([5, 0, 33, 1]), max_q=40)
    _check_small(w, q_lens=np.array([5, 0, 33, 1]), split=64, max_q=40)


def test_group4_many_requests():
    lens = synth.gen.uniform_int(77, np.arange(40, dtype=np.uint64), 8, 400)
    _check_small(_w("many", 16, 4, tuple(lens.tolist()), n_new=8), split=64)


@pytest.mark.parametrize("split", [0, 128])
def test_few_rows_varlen_with_an_empty_request(split):
    # at most 8 queries x G 8 = 64 rows per block: 128-token tiles with
    # half-height products; request 1 has no queries, contexts end mid-tile
    w = _w("wide", 16, 2, (40, 16, 200, 129), n_new=1)
    _check_small(w, q_lens=np.array([5, 0, 8, 1]), split=split, max_q=8)


def test_few_rows_whole_prompt_is_new():
    w = _w("wide_fresh", 16, 2, (1, 7, 64), n_new=1)
    _check_small(w, q_lens=np.array([1, 7, 8]), max_q=8)


@pytest.mark.parametrize("Hq,Hkv,n_new", [(4, 4, 64), (8, 4, 32), (32, 2, 4), (64, 1, 1)])
def test_few_rows_across_group_sizes(Hq, Hkv, n_new):
    # G x n_new = 64 rows per block for G = 1, 2, 16, 64; contexts end mid-tile
    w = _w(f"wide_g{Hq // Hkv}", Hq, Hkv, (70, 129, 300), n_new=n_new)
    _check_small(w)
    _check_small(w, split=128)


def test_partly_padded_128_row_blocks():
    # G 16 x 8 queries = 128 rows per block, but requests 1 and 2 have 48 and
    # 16 rows: their blocks are mostly padding rows
    w = _w("g16_varlen", 16, 1, (100, 50, 300), n_new=1)
    _check_small(w, q_lens=np.array([8, 3, 1]), max_q=8)
    _check_small(w, q_lens=np.array([8, 3, 1]), split=64, max_q=8)


@pytest.mark.parametrize("P", [32, 128])
def test_pages_of_32_and_128_tokens(P):
    # boxes as tall as the page allows: 32 rows at page 32, two 64-row boxes per
    # page at page 128; both kernels, contexts ending mid-page and mid-tile
    w = _w(f"p{P}_wide", 16, 2, (40, 130, 300, 517), n_new=6, P=P)  # 48 rows: the even split
    _check_small(w)
    w = _w(f"p{P}_rows", 16, 2, (300, 517, 1000), n_new=40, P=P)  # 320 rows: 128-row blocks
    _check_small(w)
    _check_small(w, split=192)


def test_128_row_blocks_page64_mha_and_varlen():
    # G = 1 with 300 new tokens (three blocks, the last one partial) at page 64,
    # and varlen requests whose blocks are partly padding
    _check_small(_w("mha_p64", 4, 4, (300, 700, 1301), n_new=300, P=64))
    w = _w("g8_varlen_p64", 16, 2, (600, 257, 129, 1500), n_new=1, P=64)
    _check_small(w, q_lens=np.array([100, 17, 0, 64]), max_q=100)


def test_128_row_blocks_bad_page_sets_status():
    p = pf()
    w = _w("bad_rows", 8, 2, (200, 300), n_new=32).set_scales_host()  # 128 rows per block
    kc, vc = oracle_fill_paged(w)
    bt = w.block_tables.copy()
    bt[1, 3] = w.num_pages + 7
    out, _, status = _run(p, w, _dev(kc), _dev(vc), bt=bt)
    assert status & p.DEVERR["BAD_PAGE"]
    assert np.all(np.isfinite(out))


def test_bad_page_and_clamped_context_set_status():
    p = pf()
    w = _w("bad", 8, 2, (40, 90), n_new=4).set_scales_host()
    kc, vc = oracle_fill_paged(w)
    bt = w.block_tables.copy()
    bt[1, 2] = w.num_pages + 5
    out, _, status = _run(p, w, _dev(kc), _dev(vc), bt=bt)
    assert status & p.DEVERR["BAD_PAGE"]
    assert np.all(np.isfinite(out))
    _, _, status = _run(p, w, _dev(kc), _dev(vc), max_ctx=64)  # request 1 holds 90 tokens
    assert status & p.DEVERR["BAD_CONTEXT"]


def test_bad_arguments_are_rejected():
    import torch
    p = pf()
    w = _w("arg", 12, 2, (40,), n_new=4).set_scales_host()  # G = 6 does not divide 128
    kc = torch.zeros((w.num_pages, 2, 16, 128), dtype=torch.uint8, device="cuda")
    q = torch.zeros((4, 12, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(p.PfkvError) as e:
        p.paged_prefill_attn(torch.empty_like(q), q, kc, kc, _dev(w.block_tables), _dev(w.context_lens),
                             _dev(w.q_start()), 4, 40, 1.0, 1.0, 0.1)
    assert e.value.code == -2
    w = _w("arg2", 8, 2, (40,), n_new=4).set_scales_host()
    q = torch.zeros((4, 8, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(p.PfkvError) as e:  # split not a multiple of 64
        p.paged_prefill_attn(torch.empty_like(q), q, kc, kc, _dev(w.block_tables), _dev(w.context_lens),
                             _dev(w.q_start()), 4, 40, 1.0, 1.0, 0.1, kv_split_tokens=48)
    assert e.value.code == -1


def _prefill_group(w, st, qbits, out, lse, b, kvh, rows):
    """One (request, KV head): the GPU's K/V rows of that head bit for bit
    against the oracle's encoding, then each listed (query token, head)
    against the oracle's decode over the context up to and including that token."""
    L = int(w.context_lens[b])
    kc, vc, bt_row = oracle_one_head(w, b, kvh)
    assert np.array_equal(gpu_pages_of(st.k_cache, w.block_tables[b], kvh, L, w.P), kc.reshape(-1, w.D)[:L])
    assert np.array_equal(gpu_pages_of(st.v_cache, w.block_tables[b], kvh, L, w.P), vc.reshape(-1, w.D)[:L])
    qs = w.q_start()
    res = []
    for i, h in rows:
        row = qs[b] + i
        ref, ref_lse = oracle.paged_decode_one(qbits[row, h], kc, vc, bt_row, L - w.n_new + i + 1, 0, w.P,
                                               w.k_scale, w.v_scale, w.softmax_scale)
        assert abs(lse[row, h] - ref_lse) <= 2e-4 + 2e-5 * abs(ref_lse), ("lse", b, i, h)
        res.append((out[row, h], ref))
    return res


def test_long_splitkv_appended_tokens_full_size_sampled():
    """Long split-KV B 8 (256K-1M tokens), the 8 appended tokens of each
    request as causal queries: for every request, two KV heads (the last KV
    head among them), on each the first, a middle and the last appended token
    with two query heads each."""
    import torch
    from concurrent.futures import ThreadPoolExecutor
    from synth import device as sdev
    p = pf()
    w = synth.workload(synth.LONG_SPLITKV)
    st = sdev.setup_paged(w, append_fp8_fn(p, w))
    p.kv_append_fp8(st.k_new, st.v_new, st.k_cache, st.v_cache, st.step_slots, w.k_scale, w.v_scale)
    qbits = w.q_new_bits()
    q = _dev_bits(qbits)
    out = torch.empty_like(q)
    lse = torch.empty((q.shape[0], w.Hq), dtype=torch.float32, device="cuda")
    ws = p.paged_prefill_attn(out, q, st.k_cache, st.v_cache, st.block_tables, st.context_lens,
                              _dev(w.q_start()), w.n_new, int(w.context_lens.max()), w.k_scale, w.v_scale,
                              w.softmax_scale, kv_split_tokens=w.kv_split_tokens, lse_out=lse)
    torch.cuda.synchronize()
    assert p.workspace_status(ws) == 0
    out, lse = to_np_bf16(out), lse.cpu().numpy()
    groups = {}
    for b in range(w.B):
        for j, kvh in enumerate((b % w.Hkv, (b + 4) % w.Hkv)):
            rows = []
            for i in (0, (b + j) % w.n_new, w.n_new - 1):
                rows += [(i, kvh * w.G + (3 * b + i) % w.G), (i, kvh * w.G + (5 * b + 2 * i + 1) % w.G)]
            groups[(b, kvh)] = sorted(set(rows))
    assert {kvh for _, kvh in groups} == set(range(w.Hkv))
    keys = sorted(groups, key=lambda k: -int(w.context_lens[k[0]]))
    with ThreadPoolExecutor(max_workers=8) as ex:
        futs = [ex.submit(_prefill_group, w, st, qbits, out, lse, b, kvh, groups[(b, kvh)]) for b, kvh in keys]
        pairs = [r for f in futs for r in f.result()]
    assert_within_tolerance(np.stack([g for g, _ in pairs]), np.stack([r for _, r in pairs]),
                            f"long split-KV appended tokens, {len(pairs)} sampled rows")
