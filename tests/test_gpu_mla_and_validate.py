"""mla_decode_attn and validate_tables on the GPU against the oracle."""
import numpy as np
import pytest

import oracle
import synth
from synth import gen

from gpu_helpers import assert_within_tolerance, pf, to_np_bf16

pytestmark = pytest.mark.gpu


def _setup_mla(p, m):
    from synth import device as sdev
    if m.ckv_scale is None and int(m.context_lens.sum()) * m.Dqk <= (1 << 24):
        m.set_scales_host()
    st = sdev.setup_mla(m, lambda c, c4, s: p.kv_append_fp8(c, None, c4, None, s, m.ckv_scale))
    p.kv_append_fp8(st.c_new, None, st.ckv_cache.view(m.num_pages, 1, m.P, m.Dqk), None, st.step_slots,
                    m.ckv_scale)
    return st


def _run_mla(p, m, st, topk=True):
    import torch
    out = torch.empty((m.B, m.H, m.Dv), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((m.B, m.H), dtype=torch.float32, device="cuda")
    ws = p.mla_decode_attn(out, st.q, st.ckv_cache, st.block_tables, st.context_lens,
                           st.topk if topk else None, m.ckv_scale, m.softmax_scale, lse_out=lse)
    torch.cuda.synchronize()
    return to_np_bf16(out), lse.cpu().numpy(), p.workspace_status(ws)


def _oracle_cache(m, rows_of=None):
    c = np.zeros((m.num_pages, 1, m.P, m.Dqk), np.uint8)
    for b in range(m.B):
        L = int(m.context_lens[b])
        oracle.kv_append(m.ckv_bits(b, 0, L), c, m.slots(b, 0, L), m.P, m.ckv_scale)
    return c.reshape(m.num_pages, m.P, m.Dqk)


@pytest.mark.parametrize("case", [
    dict(H=128, lens=(300, 129), topk=64),
    dict(H=128, lens=(64, 1000, 17), topk=0),
    dict(H=16, lens=(2048, 70), topk=50),
    dict(H=64, lens=(1, 65), topk=1),
])
def test_mla_small_cases_match_oracle(case):
    p = pf()
    m = synth.MlaWorkload("mla", B=len(case["lens"]), H=case["H"], context_lens=np.array(case["lens"]),
                          topk_n=case["topk"], P=64, seed=8)
    st = _setup_mla(p, m)
    out, lse, status = _run_mla(p, m, st)
    assert status == 0
    c = _oracle_cache(m)
    assert np.array_equal(st.ckv_cache.cpu().numpy(), c)
    ref, ref_lse = oracle.mla_decode(m.q_bits(), c, m.block_tables, m.context_lens, m.topk, m.P, m.Dv,
                                     m.ckv_scale, m.softmax_scale)
    assert_within_tolerance(out, ref, "mla")
    np.testing.assert_allclose(lse, ref_lse, rtol=2e-5, atol=2e-4)


def _mla_check(p, m, st, topk=None, ws=None, what="mla"):
    import torch
    out = torch.empty((m.B, m.H, m.Dv), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((m.B, m.H), dtype=torch.float32, device="cuda")
    tk = st.topk if topk is None else torch.from_numpy(topk).cuda()
    ws = p.mla_decode_attn(out, st.q, st.ckv_cache, st.block_tables, st.context_lens,
                           tk if (m.topk is not None or topk is not None) else None, m.ckv_scale, m.softmax_scale,
                           lse_out=lse, workspace=ws)
    torch.cuda.synchronize()
    assert p.workspace_status(ws) == 0
    c = _oracle_cache(m)
    ref, ref_lse = oracle.mla_decode(m.q_bits(), c, m.block_tables, m.context_lens,
                                     m.topk if topk is None else topk, m.P, m.Dv, m.ckv_scale, m.softmax_scale)
    assert_within_tolerance(to_np_bf16(out), ref, what)
    fin = np.isfinite(ref_lse)
    np.testing.assert_allclose(lse.cpu().numpy()[fin], ref_lse[fin], rtol=2e-5, atol=2e-4)
    assert np.all(np.isneginf(lse.cpu().numpy()[~fin]))
    return to_np_bf16(out)


def test_mla_small_batch_splits_lists_across_sm_pairs():
    """Three requests leave most SM pairs idle, so each list (every token here)
    is split into runs on separate pairs and folded by log-sum-exp; the short
    request's later runs are empty."""
    p = pf()
    m = synth.MlaWorkload("mla_split", B=3, H=128, context_lens=np.array([4000, 2500, 70]), topk_n=0, P=64, seed=12)
    assert p.mla_decode_workspace_size(3, 128, 512, 0) > 256  # room for the split states
    st = _setup_mla(p, m)
    full = _mla_check(p, m, st, what="mla split across pairs")
    import torch
    one = torch.empty(256, dtype=torch.uint8, device="cuda")  # room for no split: one pair per request
    single = _mla_check(p, m, st, ws=one, what="mla unsplit")
    assert np.abs(full - single).max() < 0.05


def test_mla_split_with_padded_and_partial_lists():
    """Top-k lists split across pairs where one request's second half is all
    padding (a run with no token at all)."""
    p = pf()
    m = synth.MlaWorkload("mla_split_pad", B=2, H=64, context_lens=np.array([3000, 2000]), topk_n=600, P=64,
                          seed=14)
    st = _setup_mla(p, m)
    tk = m.topk.copy()
    tk[1, 300:] = -1
    _mla_check(p, m, st, topk=tk, what="mla split, padded list")


def test_mla_topk_padding_and_out_of_range_indices():
    import torch
    p = pf()
    m = synth.MlaWorkload("mla", B=2, H=16, context_lens=np.array([100, 300]), topk_n=0, P=64, seed=5)
    st = _setup_mla(p, m)
    tk = np.full((2, 40), -1, np.int32)
    tk[0, :10] = np.arange(0, 100, 10)
    tk[1, 5:35] = np.arange(0, 300, 10)
    st.topk = torch.from_numpy(tk).cuda()
    out, _, status = _run_mla(p, m, st)
    assert status == 0
    c = _oracle_cache(m)
    ref, _ = oracle.mla_decode(m.q_bits(), c, m.block_tables, m.context_lens, tk, m.P, m.Dv, m.ckv_scale,
                               m.softmax_scale)
    assert_within_tolerance(out, ref, "mla padding")
    tk[1, 0] = 300  # == context length: skipped and flagged
    st.topk = torch.from_numpy(tk).cuda()
    out2, _, status = _run_mla(p, m, st)
    assert status & p.DEVERR["BAD_TOPK"]
    assert_within_tolerance(out2, ref, "mla bad index skipped")


def _mla_request_check(m, st, q, out, lse, b, heads):
    """One request: its selected latent rows on the GPU bit for bit against
    the oracle's encoding of the host generator's rows, then each listed head
    against the oracle's decode over those rows."""
    import torch
    tok = m.topk[b]
    rows = m.ckv_rows_bits(b, tok)  # [k][576] bf16 bits of the selected tokens
    mini = np.zeros((len(tok), 1, 1, m.Dqk), np.uint8)
    oracle.kv_append(rows[:, None, :], mini, np.arange(len(tok), dtype=np.int64), 1, m.ckv_scale)
    mini = mini.reshape(len(tok), 1, m.Dqk)
    pages = torch.as_tensor(m.block_tables[b, tok // m.P].astype(np.int64), device="cuda")
    offs = torch.as_tensor((tok % m.P).astype(np.int64), device="cuda")
    assert np.array_equal(st.ckv_cache[pages, offs].cpu().numpy(), mini[:, 0, :]), ("latent rows", b)
    res = []
    for h in heads:
        ref, ref_lse = oracle.mla_decode_one(q[b, h], mini, np.arange(len(tok), dtype=np.int32),
                                             len(tok), None, 1, m.Dv, m.ckv_scale, m.softmax_scale)
        assert abs(lse[b, h] - ref_lse) <= 2e-4 + 2e-5 * abs(ref_lse), ("lse", b, h)
        res.append((out[b, h], ref))
    return res


def _mla_sampled(m, st, out, lse, whole, what):
    """Every request's latent rows bit for bit; every head of the requests in
    `whole`, and 8 heads (a different stride phase per request) of the rest."""
    from concurrent.futures import ThreadPoolExecutor
    q = m.q_bits()
    plan = [(b, list(range(m.H)) if b in whole else list(range(b % 16, m.H, 16))) for b in range(m.B)]
    with ThreadPoolExecutor(max_workers=8) as ex:
        futs = [ex.submit(_mla_request_check, m, st, q, out, lse, b, hs) for b, hs in plan]
        pairs = [r for f in futs for r in f.result()]
    assert_within_tolerance(np.stack([g for g, _ in pairs]), np.stack([r for _, r in pairs]),
                            f"{what}, {len(pairs)} sampled rows")


def test_mla_topk2048_full_size_sampled():
    """MLA B 64 x 128 heads, top-k 2048 of 65536: every request's selected
    latent rows bit for bit; every head of requests 0, 21, 42 and 63 (the
    first and last clusters of the grid among them) and 8 heads of each
    other request against the oracle."""
    p = pf()
    m = synth.workload(synth.MLA_TOPK)
    st = _setup_mla(p, m)
    out, lse, status = _run_mla(p, m, st)
    assert status == 0
    _mla_sampled(m, st, out, lse, (0, 21, 42, m.B - 1), "MLA 64 x 128 heads, top-k 2048")


def test_mla_topk2048_batch16_split_full_size_sampled():
    """16 requests x 128 heads, top-k 2048 of 65536: the lists are split over
    idle SM pairs and folded; every request's selected latent rows bit for
    bit, every head of requests 0 and 15 and 8 heads of each other request
    against the oracle."""
    p = pf()
    m = synth.MlaWorkload("mla_b16", B=16, H=128, context_lens=np.full(16, 65536), topk_n=2048, P=64)
    assert p.mla_decode_workspace_size(16, 128, 512, 2048) > 256  # the split states fit
    st = _setup_mla(p, m)
    out, lse, status = _run_mla(p, m, st)
    assert status == 0
    _mla_sampled(m, st, out, lse, (0, m.B - 1), "MLA 16 x 128 heads, top-k 2048, split")


def test_validate_tables_flags_each_error_kind():
    import torch
    p = pf()
    B, maxp, P, pages = 3, 4, 16, 10
    bt = torch.tensor([[0, 1, 2, -1], [3, 4, -1, -1], [5, 6, 7, 8]], dtype=torch.int32, device="cuda")
    cl = torch.tensor([40, 20, 64], dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    p.validate_tables(bt, cl, P, pages, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    bt[2, 3] = 10
    p.validate_tables(bt, cl, P, pages, err)
    torch.cuda.synchronize()
    assert err.item() == p.DEVERR["BAD_PAGE"]
    bt[2, 3] = 8
    cl[1] = 70
    p.validate_tables(bt, cl, P, pages, err)
    torch.cuda.synchronize()
    assert err.item() & p.DEVERR["BAD_CONTEXT"]
    cl[1] = 20
    tk = torch.tensor([[0, 39], [19, 20], [1, -1]], dtype=torch.int32, device="cuda")
    p.validate_tables(bt, cl, P, pages, err, topk_idx=tk)
    torch.cuda.synchronize()
    assert err.item() == p.DEVERR["BAD_TOPK"]
    sl = torch.tensor([0, 159, 160], dtype=torch.int64, device="cuda")
    p.validate_tables(bt, cl, P, pages, err, slot_mapping=sl)
    torch.cuda.synchronize()
    assert err.item() == p.DEVERR["BAD_SLOT"]


def test_device_generator_matches_host_generator():
    import torch
    from synth import device as sdev
    key = gen.make_key(0, gen.TENSOR_V)
    base = (5 << 21) * 1024 + 12345
    n = 1_000_003
    t = torch.empty(n, dtype=torch.int16, device="cuda")
    word = torch.zeros(1, dtype=torch.int32, device="cuda")
    sdev.fill_normal_bf16(t, key, base, word)
    host = gen.normal_bf16(key, np.arange(base, base + n, dtype=np.uint64))
    assert np.array_equal(t.cpu().numpy().view(np.uint16), host)
    assert word.item() == int((host & 0x7FFF).max())


def test_bounded_barrier_wait_times_out_with_a_status():
    """A wait on a barrier that nothing completes gives up (about one second)
    and reports the timeout bit; the context stays usable afterwards."""
    import torch
    p = pf()
    st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    p.selftest_barrier_timeout(st)
    torch.cuda.synchronize()
    assert st.item() == p.DEVERR["WAIT_TIMEOUT"]
    x = torch.arange(10, device="cuda").sum()  # the context still works
    assert x.item() == 45
