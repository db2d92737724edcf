"""paged_decode_attn on the GPU against the oracle.

Small cases are compared element by element over every output; the full-size
workloads are compared on sampled (request, head) rows, each recomputed by the
oracle from the host generator in a private cache, with the GPU's cache bytes
for that row checked bit for bit as well."""
import numpy as np
import pytest

import oracle
import synth

from gpu_helpers import (append_bf16_fn, append_fp8_fn, assert_within_tolerance, gpu_pages_of,
                         oracle_caches, oracle_one_head, pf, to_np_bf16)

pytestmark = pytest.mark.gpu


def _run(p, w, st, split=0, ws=None):
    import torch
    out = torch.empty_like(st.q)
    lse = torch.empty(w.B, w.Hq, dtype=torch.float32, device="cuda")
    k_scale = 1.0 if st.k_cache.dtype == torch.bfloat16 else w.k_scale
    v_scale = 1.0 if st.k_cache.dtype == torch.bfloat16 else w.v_scale
    maxc = int(sum((int(L) + split - 1) // split for L in w.context_lens)) if split else 0
    ws = p.paged_decode_attn(out, st.q, st.k_cache, st.v_cache, st.block_tables, st.context_lens, k_scale,
                             v_scale, w.softmax_scale, kv_split_tokens=split, lse_out=lse, workspace=ws,
                             max_total_chunks=maxc)
    torch.cuda.synchronize()
    return to_np_bf16(out), lse.cpu().numpy(), p.workspace_status(ws)


def _setup(p, w, bf16=False):
    from synth import device as sdev
    if bf16:
        st = sdev.setup_paged(w, append_bf16_fn(p), bf16_cache=True, scales_on_device=False)
        p.kv_append_bf16(st.k_new, st.v_new, st.k_cache, st.v_cache, st.step_slots)
    else:
        # small workloads: scales from the host generator; full-size ones: the
        # same amax reduced on the device by the (bit-identical) device generator
        if w.k_scale is None and w.unique_tokens * w.Hkv * w.D <= (1 << 24):
            w.set_scales_host()
        st = sdev.setup_paged(w, append_fp8_fn(p, w))
        p.kv_append_fp8(st.k_new, st.v_new, st.k_cache, st.v_cache, st.step_slots, w.k_scale, w.v_scale)
    return st


def _full_check(p, w, split=0, bf16=False):
    st = _setup(p, w, bf16)
    out, lse, status = _run(p, w, st, split)
    assert status == 0
    kc, vc = oracle_caches(w, bf16=bf16)
    got_k = st.k_cache.cpu().numpy() if not bf16 else st.k_cache.view(__import__("torch").int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got_k, kc)
    ks, vs = (1.0, 1.0) if bf16 else (w.k_scale, w.v_scale)
    ref, ref_lse = oracle.paged_decode(w.q_bits(), kc, vc, w.block_tables, w.context_lens, w.P, ks, vs,
                                       w.softmax_scale, w.Hkv)
    assert_within_tolerance(out, ref, w.name)
    fin = np.isfinite(ref_lse)
    np.testing.assert_allclose(lse[fin], ref_lse[fin], rtol=2e-5, atol=2e-4)
    assert np.all(np.isneginf(lse[~fin]))
    return out


def test_tiny_gqa_workload():
    _full_check(pf(), synth.workload(synth.TINY_GQA))


@pytest.mark.parametrize("case", [
    dict(Hq=4, Hkv=4, P=16, lens=(1, 15, 17, 300)),            # MHA, ragged tails
    dict(Hq=8, Hkv=2, P=16, lens=(16, 33, 250, 2)),            # G = 4
    dict(Hq=16, Hkv=2, P=64, lens=(64, 65, 700, 129)),         # G = 8, page 64
    dict(Hq=32, Hkv=2, P=16, lens=(40, 500, 3, 77)),           # G = 16 (two head tiles)
    dict(Hq=10, Hkv=2, P=32, lens=(31, 96, 1, 200)),           # G = 5, page 32
    dict(Hq=8, Hkv=8, P=16, lens=(0, 50, 0, 7)),               # empty contexts
])
@pytest.mark.parametrize("split", [0, 16, 64])
def test_small_cases_match_oracle(case, split):
    w = synth.PagedWorkload("small", B=len(case["lens"]), Hq=case["Hq"], Hkv=case["Hkv"], D=128,
                            P=case["P"], context_lens=np.array(case["lens"]), seed=13,
                            n_new=1 if min(case["lens"]) > 0 else 0)
    _full_check(pf(), w, split=split)


def test_many_requests_cross_scan_chunks():
    rng_lens = synth.gen.uniform_int(99, np.arange(1500, dtype=np.uint64), 1, 40)
    w = synth.PagedWorkload("many", B=1500, Hq=4, Hkv=1, D=128, P=16, context_lens=rng_lens, seed=3)
    _full_check(pf(), w)


def test_shared_prefix_requests():
    lens = np.array([70, 90, 51, 200, 33])
    w = synth.PagedWorkload("prefix", B=5, Hq=16, Hkv=2, D=128, P=16, context_lens=lens,
                            shared_requests=3, shared_tokens=48, seed=9)
    _full_check(pf(), w)


@pytest.mark.parametrize("lens", [(5, 40, 77, 300), (1, 16, 17, 1000)])
def test_bf16_cache_matches_oracle(lens):
    w = synth.PagedWorkload("bf16", B=4, Hq=8, Hkv=2, D=128, P=16, context_lens=np.array(lens), seed=21)
    _full_check(pf(), w, bf16=True)


def test_bad_page_sets_status_and_reads_zeros():
    import torch
    p = pf()
    w = synth.PagedWorkload("bad", B=2, Hq=4, Hkv=1, D=128, P=16, context_lens=np.array([40, 40]), seed=2)
    st = _setup(p, w)
    bt = st.block_tables.clone()
    bt[1, 1] = w.num_pages + 100  # outside the pool
    st.block_tables = bt
    out, lse, status = _run(p, w, st)
    assert status & p.DEVERR["BAD_PAGE"]
    assert np.all(np.isfinite(out))


def test_context_beyond_block_table_sets_status():
    import torch
    p = pf()
    w = synth.PagedWorkload("ctx", B=2, Hq=4, Hkv=1, D=128, P=16, context_lens=np.array([40, 40]), seed=2)
    st = _setup(p, w)
    st.context_lens = torch.tensor([40, 10_000], dtype=torch.int32, device="cuda")
    _, _, status = _run(p, w, st)
    assert status & p.DEVERR["BAD_CONTEXT"]


def test_workspace_too_small_is_rejected_on_host():
    import torch
    p = pf()
    w = synth.PagedWorkload("ws", B=2, Hq=4, Hkv=1, D=128, P=16, context_lens=np.array([40, 40]), seed=2)
    st = _setup(p, w)
    ws = torch.empty(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(p.PfkvError) as e:
        _run(p, w, st, ws=ws)
    assert e.value.code == -5


# ------------------------------------------------------------ full-size, sampled
def _check_group(w, st, q, out, lse, b, kvh, heads, bf16):
    """One (request, KV head): the GPU's K/V rows of that head bit for bit
    against the oracle's encoding of the host generator's rows, then every
    listed query head of the group against the oracle's decode."""
    L = int(w.context_lens[b])
    kc, vc, bt_row = oracle_one_head(w, b, kvh, bf16=bf16)
    got_k = gpu_pages_of(st.k_cache, w.block_tables[b], kvh, L, w.P)
    got_v = gpu_pages_of(st.v_cache, w.block_tables[b], kvh, L, w.P)
    if bf16:
        got_k, got_v = got_k.view(np.uint16), got_v.view(np.uint16)
    assert np.array_equal(got_k, kc.reshape(-1, w.D)[:L]), ("K rows", b, kvh)
    assert np.array_equal(got_v, vc.reshape(-1, w.D)[:L]), ("V rows", b, kvh)
    ks, vs = (1.0, 1.0) if bf16 else (w.k_scale, w.v_scale)
    res = []
    for h in heads:
        ref, ref_lse = oracle.paged_decode_one(q[b, h], kc, vc, bt_row, L, 0, w.P, ks, vs, w.softmax_scale)
        assert abs(lse[b, h] - ref_lse) <= 2e-4 + 2e-5 * abs(ref_lse), ("lse", b, h, lse[b, h], ref_lse)
        res.append((out[b, h], ref))
    return res


def _sampled_check(p, w, st, out, lse, samples, bf16=False, threads=8):
    """Every sampled (request, query head) against the oracle; the samples are
    grouped by (request, KV head) so each group's rows are encoded once, and
    the groups run on host threads (the oracle's ctypes calls release the GIL)."""
    from concurrent.futures import ThreadPoolExecutor
    q = w.q_bits()
    groups = {}
    for (b, h) in samples:
        groups.setdefault((int(b), int(h) // w.G), set()).add(int(h))
    # longest contexts first, so the pool's tail is short
    keys = sorted(groups, key=lambda k: -int(w.context_lens[k[0]]))
    with ThreadPoolExecutor(max_workers=threads) as ex:
        futs = [ex.submit(_check_group, w, st, q, out, lse, b, kvh, sorted(groups[(b, kvh)]), bf16)
                for (b, kvh) in keys]
        pairs = [r for f in futs for r in f.result()]
    gots = np.stack([g for g, _ in pairs])
    refs = np.stack([r for _, r in pairs])
    assert_within_tolerance(gots, refs, f"{w.name} sampled {len(pairs)} (request, head) rows")


def _appended_rows_check(w, st):
    """The step's appended rows (every request, every KV head) bit for bit:
    read back through the slot mapping and compared with the oracle's encoding
    of the same bf16 rows."""
    import torch
    slots = w.step_slots()
    if slots.size == 0:
        return
    T = slots.size
    sl = torch.as_tensor(slots, device=st.k_cache.device)
    for which, cache, scale in (("k", st.k_cache, w.k_scale), ("v", st.v_cache, w.v_scale)):
        rows = cache.permute(0, 2, 1, 3).reshape(-1, w.Hkv, w.D)  # [page*P + off][Hkv][D]
        got = rows.index_select(0, sl).cpu().numpy()
        mini = np.zeros((T, w.Hkv, 1, w.D), np.uint8)
        oracle.kv_append(w.step_kv_bits(which), mini, np.arange(T, dtype=np.int64), 1, scale)
        assert np.array_equal(got, mini[:, :, 0, :]), f"appended {which} rows differ"


def _samples(w, n, seed):
    b = synth.gen.uniform_int(seed, np.arange(n, dtype=np.uint64), 0, w.B - 1)
    h = synth.gen.uniform_int(seed + 1, np.arange(n, dtype=np.uint64), 0, w.Hq - 1)
    return list(zip(b.tolist(), h.tolist()))


@pytest.mark.parametrize("bf16", [False, True])
def test_mha_b32_full_size_sampled(bf16):
    """MHA B 32 x 48 heads x 8192: every head of request 7 and of the last
    request, plus seeded samples."""
    p = pf()
    w = synth.workload(synth.MHA_B32)
    st = _setup(p, w, bf16=bf16)
    out, lse, status = _run(p, w, st)
    assert status == 0
    whole = [(7, h) for h in range(w.Hq)] + [(w.B - 1, h) for h in range(w.Hq)]
    _sampled_check(p, w, st, out, lse, _samples(w, 6, 41) + [(0, 0)] + whole, bf16=bf16)
    if not bf16:
        _appended_rows_check(w, st)


def test_gqa_shared_prefix_full_size_sampled():
    """GQA 64/8 with a 2048-token prefix shared by requests 0-15: two query
    heads (on different KV heads) of every sharer and of 16 private requests,
    including the last."""
    p = pf()
    w = synth.workload(synth.GQA_PREFIX)
    st = _setup(p, w)
    out, lse, status = _run(p, w, st)
    assert status == 0
    privs = list(range(w.shared_requests, w.B, 3))[:15] + [w.B - 1]
    samples = []
    for i, b in enumerate(list(range(w.shared_requests)) + privs):
        samples += [(b, (5 * i) % w.Hq), (b, (5 * i + 4 * w.G + 3) % w.Hq)]
    samples += [(0, 0), (5, 63)]
    _sampled_check(p, w, st, out, lse, samples)
    _appended_rows_check(w, st)


def test_long_split_kv_full_size_sampled():
    """Long split-KV B 8, contexts 256K-1M, 4096-token chunks: two query heads
    on different KV heads of every request (both 1,048,576-token requests
    included, the last KV head among them), and every request's eight appended
    rows on every KV head."""
    p = pf()
    w = synth.workload(synth.LONG_SPLITKV)
    st = _setup(p, w)
    out, lse, status = _run(p, w, st, split=w.kv_split_tokens)
    assert status == 0
    samples = []
    for b in range(w.B):
        kv_a, kv_b = b % w.Hkv, (b + 4) % w.Hkv
        samples += [(b, kv_a * w.G + (3 * b) % w.G), (b, kv_b * w.G + (5 * b + 1) % w.G)]
    samples += [(0, 0), (w.B - 1, w.Hq - 1)]
    assert {b for b, _ in samples} == set(range(w.B))
    assert (w.Hq - 1) // w.G == w.Hkv - 1
    _sampled_check(p, w, st, out, lse, samples)
    _appended_rows_check(w, st)
