"""Per-tensor (device), per-head and per-token scales on the GPU against the oracle.

kv_append_fp8_scaled: codes and per-token scales bit for bit.  Decode: caches
and scales built by the oracle from the host generator are uploaded, the GPU
decodes them and every output is compared with the oracle's decode of the
same bytes (tolerance |err| <= 2e-3 * max|ref| + 1e-3 + half a bf16 ulp).
The full-size workload fills its cache through the product's per-token append
on device-generated rows; sampled (request, head) rows are recomputed by the
oracle from the host generator, their codes and scales checked bit for bit,
and decoded by the oracle."""
import numpy as np
import pytest

import oracle
import synth

from gpu_helpers import (assert_within_tolerance, gpu_pages_of, gpu_scales_of, oracle_one_head_token,
                         pf, to_np_bf16)
from oracle_helpers import oracle_fill_scaled, spread_rows, spread_scales

pytestmark = pytest.mark.gpu

GRANS = [oracle.SCALE_TENSOR, oracle.SCALE_HEAD, oracle.SCALE_TOKEN]


def _dev_bits(bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to("cuda").view(torch.bfloat16)


def _dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda")


def _gpu_fill(p, w, gran, spread=6, zero_rows=False):
    """Device caches and scales written by the product's scaled append from
    the same host rows the oracle encodes."""
    import torch
    shape = (w.num_pages, w.Hkv, w.P, w.D)
    kc = torch.zeros(shape, dtype=torch.uint8, device="cuda")
    vc = torch.zeros_like(kc)
    if gran == oracle.SCALE_TOKEN:
        ks = torch.full(shape[:3], float("nan"), dtype=torch.float32, device="cuda")
        vs = torch.full_like(ks, float("nan"))
    else:
        hk, hv = spread_scales(w, gran, spread, zero_rows)
        ks, vs = _dev(hk), _dev(hv)
    for b in range(w.B):
        L = int(w.context_lens[b])
        t0 = w.shared_tokens if 0 < b < w.shared_requests else 0
        if L <= t0:
            continue
        kb = _dev_bits(spread_rows(w, "k", b, t0, L, spread, zero_rows))
        vb = _dev_bits(spread_rows(w, "v", b, t0, L, spread, zero_rows))
        p.kv_append_fp8_scaled(kb, vb, kc, vc, _dev(w.slots(b, t0, L)), gran, ks, vs)
    torch.cuda.synchronize()
    return kc, vc, ks, vs


def _decode(p, w, kc, vc, gran, ks, vs, split=0):
    import torch
    q = _dev_bits(w.q_bits())
    out = torch.empty_like(q)
    lse = torch.empty(w.B, w.Hq, dtype=torch.float32, device="cuda")
    maxc = int(sum((int(L) + split - 1) // split for L in w.context_lens)) if split else 0
    ws = p.paged_decode_attn_scaled(out, q, kc, vc, gran, ks, vs, _dev(w.block_tables),
                                    _dev(w.context_lens), w.softmax_scale, kv_split_tokens=split,
                                    lse_out=lse, max_total_chunks=maxc)
    torch.cuda.synchronize()
    return to_np_bf16(out), lse.cpu().numpy(), p.workspace_status(ws)


def _scale_rows_used(w, scales):
    """Per-token scales at every attended slot (others are never read)."""
    rows = []
    for b in range(w.B):
        L = int(w.context_lens[b])
        sl = w.slots(b, 0, L)
        rows.append(scales[sl // w.P, :, sl % w.P])
    return np.concatenate(rows)


# ------------------------------------------------------------------ append
@pytest.mark.parametrize("gran", GRANS)
@pytest.mark.parametrize("D", [64, 128, 512])
def test_scaled_append_is_bit_exact(gran, D):
    p = pf()
    w = synth.PagedWorkload("app", B=3, Hq=4, Hkv=2, D=D, P=16, context_lens=np.array([1, 31, 70]),
                            seed=17)
    kc, vc, ks, vs = _gpu_fill(p, w, gran, zero_rows=True)
    okc, ovc, oks, ovs = oracle_fill_scaled(w, gran, zero_rows=True)
    assert np.array_equal(kc.cpu().numpy(), okc)
    assert np.array_equal(vc.cpu().numpy(), ovc)
    if gran == oracle.SCALE_TOKEN:
        a, b = _scale_rows_used(w, ks.cpu().numpy()), _scale_rows_used(w, oks)
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
        a, b = _scale_rows_used(w, vs.cpu().numpy()), _scale_rows_used(w, ovs)
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_token_append_k_only_and_skipped_slots():
    import torch
    p = pf()
    T, H, D, P, pages = 40, 3, 128, 16, 8
    w = synth.PagedWorkload("konly", B=1, Hq=H, Hkv=H, D=D, P=P, context_lens=np.array([T]), seed=5)
    bits = spread_rows(w, "k", 0, 0, T, spread=10, zero_rows=True)
    slots = ((np.arange(T) * 5) % (pages * P)).astype(np.int64)
    slots[3] = -1  # skipped
    slots[7] = pages * P + 2  # outside the cache: skipped
    kc = torch.zeros((pages, H, P, D), dtype=torch.uint8, device="cuda")
    ks = torch.full((pages, H, P), -1.0, dtype=torch.float32, device="cuda")
    p.kv_append_fp8_scaled(_dev_bits(bits), None, kc, None, _dev(slots), oracle.SCALE_TOKEN, ks, None)
    torch.cuda.synchronize()
    okc = np.zeros((pages, H, P, D), np.uint8)
    oks = np.full((pages, H, P), -1.0, np.float32)
    keep = (slots >= 0) & (slots < pages * P)
    oracle.kv_append_token(bits[keep], okc, oks, slots[keep], P)
    assert np.array_equal(kc.cpu().numpy(), okc)
    assert np.array_equal(ks.cpu().numpy().view(np.uint32), oks.view(np.uint32))


def test_scaled_append_rejects_bad_arguments():
    import torch
    p = pf()
    kb = torch.zeros((2, 1, 128), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((1, 1, 16, 128), dtype=torch.uint8, device="cuda")
    sl = torch.zeros(2, dtype=torch.int64, device="cuda")
    ks = torch.zeros((1, 1, 16), dtype=torch.float32, device="cuda")
    with pytest.raises(p.PfkvError) as e:
        p.kv_append_fp8_scaled(kb, None, kc, None, sl, 7, ks, None)
    assert e.value.code == -1
    with pytest.raises(p.PfkvError) as e:
        p.kv_append_fp8_scaled(kb, None, kc, None, sl, oracle.SCALE_TOKEN, None, None)
    assert e.value.code == -1
    wide = torch.zeros((2, 1, 576), dtype=torch.bfloat16, device="cuda")
    wc = torch.zeros((1, 1, 16, 576), dtype=torch.uint8, device="cuda")
    with pytest.raises(p.PfkvError) as e:
        p.kv_append_fp8_scaled(wide, None, wc, None, sl, oracle.SCALE_TOKEN, ks, None)
    assert e.value.code == -2


# ------------------------------------------------------------------ decode
CASES = [
    dict(Hq=8, Hkv=2, lens=(5, 40, 77)),                       # G=4
    dict(Hq=16, Hkv=1, lens=(1, 16, 17, 300)),                 # G=16 (two head tiles)
    dict(Hq=4, Hkv=4, lens=(33, 64, 100)),                     # MHA
    dict(Hq=8, Hkv=1, lens=(0, 130, 64, 200), P=64),           # empty request, P=64
]


@pytest.mark.parametrize("gran", GRANS)
@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("split", [0, 32])
def test_scaled_decode_matches_oracle(gran, case, split):
    p = pf()
    case = dict(case)
    lens = case.pop("lens")
    w = synth.PagedWorkload("dec", B=len(lens), D=128, P=case.pop("P", 16),
                            context_lens=np.array(lens), seed=23, **case)
    okc, ovc, oks, ovs = oracle_fill_scaled(w, gran, zero_rows=True)
    out, lse, status = _decode(p, w, _dev(okc), _dev(ovc), gran, _dev(oks), _dev(ovs), split)
    assert status == 0
    ref, ref_lse = oracle.paged_decode_scaled(w.q_bits(), okc, ovc, gran, oks, ovs, w.block_tables,
                                              w.context_lens, w.P, w.softmax_scale, w.Hkv)
    assert_within_tolerance(out, ref, f"gran {gran} {lens} split {split}")
    fin = np.isfinite(ref_lse)
    assert np.all(~np.isfinite(lse[~fin]))
    np.testing.assert_allclose(lse[fin], ref_lse[fin], rtol=2e-5, atol=2e-4)


def test_token_decode_shared_prefix_and_wide_spread():
    p = pf()
    lens = np.array([70, 90, 51, 200, 33])
    w = synth.PagedWorkload("prefix", B=5, Hq=16, Hkv=2, D=128, P=16, context_lens=lens,
                            shared_requests=3, shared_tokens=48, seed=9)
    gran = oracle.SCALE_TOKEN
    okc, ovc, oks, ovs = oracle_fill_scaled(w, gran, spread=12)
    out, lse, status = _decode(p, w, _dev(okc), _dev(ovc), gran, _dev(oks), _dev(ovs))
    assert status == 0
    ref, _ = oracle.paged_decode_scaled(w.q_bits(), okc, ovc, gran, oks, ovs, w.block_tables,
                                        w.context_lens, w.P, w.softmax_scale, w.Hkv)
    assert_within_tolerance(out, ref, "shared prefix, spread 12")


def test_token_decode_bad_page_sets_status_and_stays_finite():
    import torch
    p = pf()
    w = synth.PagedWorkload("bad", B=2, Hq=4, Hkv=1, D=128, P=16, context_lens=np.array([40, 40]), seed=2)
    gran = oracle.SCALE_TOKEN
    okc, ovc, oks, ovs = oracle_fill_scaled(w, gran)
    bt = w.block_tables.copy()
    bt[1, 1] = w.num_pages + 100
    q = _dev_bits(w.q_bits())
    out = torch.empty_like(q)
    ws = p.paged_decode_attn_scaled(out, q, _dev(okc), _dev(ovc), gran, _dev(oks), _dev(ovs), _dev(bt),
                                    _dev(w.context_lens), w.softmax_scale)
    torch.cuda.synchronize()
    assert p.workspace_status(ws) & p.DEVERR["BAD_PAGE"]
    assert np.all(np.isfinite(to_np_bf16(out)))


def test_scaled_decode_rejects_bad_arguments():
    import torch
    p = pf()
    w = synth.PagedWorkload("arg", B=1, Hq=4, Hkv=1, D=128, P=16, context_lens=np.array([16]), seed=2)
    q = torch.zeros((1, 4, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    kc = torch.zeros((w.num_pages, 1, 16, 128), dtype=torch.uint8, device="cuda")
    ks = torch.ones((w.num_pages, 1, 16), dtype=torch.float32, device="cuda")
    bt, cl = _dev(w.block_tables), _dev(w.context_lens)
    with pytest.raises(p.PfkvError) as e:
        p.paged_decode_attn_scaled(out, q, kc, kc, 5, ks, ks, bt, cl, 0.1)
    assert e.value.code == -1
    with pytest.raises(p.PfkvError) as e:  # misaligned scale array (not 16-byte aligned)
        p.paged_decode_attn_scaled(out, q, kc, kc, oracle.SCALE_TOKEN, ks.view(-1)[1:], ks, bt, cl, 0.1)
    assert e.value.code == -1


# ------------------------------------------------------- full size, sampled
def _token_group(w, st, ks, vs, q, out, lse, b, kvh, heads):
    """One (request, KV head) under per-token scales: codes and scales bit for
    bit against the oracle's encoding, then each listed query head against
    the oracle's decode of those bytes."""
    L = int(w.context_lens[b])
    kc, vc, oks, ovs, bt_row = oracle_one_head_token(w, b, kvh)
    assert np.array_equal(gpu_pages_of(st.k_cache, w.block_tables[b], kvh, L, w.P), kc.reshape(-1, w.D)[:L])
    assert np.array_equal(gpu_pages_of(st.v_cache, w.block_tables[b], kvh, L, w.P), vc.reshape(-1, w.D)[:L])
    assert np.array_equal(gpu_scales_of(ks, w.block_tables[b], kvh, L, w.P).view(np.uint32),
                          oks.reshape(-1)[:L].view(np.uint32))
    assert np.array_equal(gpu_scales_of(vs, w.block_tables[b], kvh, L, w.P).view(np.uint32),
                          ovs.reshape(-1)[:L].view(np.uint32))
    res = []
    for h in heads:
        ref, ref_lse = oracle.paged_decode_scaled_one(q[b, h], kc, vc, oracle.SCALE_TOKEN, oks, ovs, bt_row,
                                                      L, 0, w.P, w.softmax_scale)
        assert abs(lse[b, h] - ref_lse) <= 2e-4 + 2e-5 * abs(ref_lse), ("lse", b, h)
        res.append((out[b, h], ref))
    return res


def test_mha_b32_token_scales_full_size_sampled():
    """MHA B 32 x 48 heads x 8192 under per-token scales: two heads of every
    request (the first and last head among them), codes, scales and output."""
    import torch
    from concurrent.futures import ThreadPoolExecutor
    from synth import device as sdev
    p = pf()
    w = synth.workload(synth.MHA_B32)
    shape = (w.num_pages, w.Hkv, w.P)
    ks = torch.zeros(shape, dtype=torch.float32, device="cuda")
    vs = torch.zeros_like(ks)
    append = lambda k, v, kc, vc, s: p.kv_append_fp8_scaled(k, v, kc, vc, s, oracle.SCALE_TOKEN, ks, vs)
    w.k_scale = w.v_scale = 1.0  # unused: the per-token scales replace them
    st = sdev.setup_paged(w, append)
    append(st.k_new, st.v_new, st.k_cache, st.v_cache, st.step_slots)
    out = torch.empty_like(st.q)
    lse = torch.empty(w.B, w.Hq, dtype=torch.float32, device="cuda")
    ws = p.paged_decode_attn_scaled(out, st.q, st.k_cache, st.v_cache, oracle.SCALE_TOKEN, ks, vs,
                                    st.block_tables, st.context_lens, w.softmax_scale, lse_out=lse)
    torch.cuda.synchronize()
    assert p.workspace_status(ws) == 0
    out, lse = to_np_bf16(out), lse.cpu().numpy()
    q = w.q_bits()
    groups = {}
    for b in range(w.B):
        for h in ((7 * b) % w.Hq, (7 * b + w.Hq // 2 + 1) % w.Hq):
            groups.setdefault((b, h // w.G), set()).add(h)
    groups.setdefault((0, 0), set()).add(0)
    groups.setdefault((w.B - 1, (w.Hq - 1) // w.G), set()).add(w.Hq - 1)
    with ThreadPoolExecutor(max_workers=8) as ex:
        futs = [ex.submit(_token_group, w, st, ks, vs, q, out, lse, b, kvh, sorted(hs))
                for (b, kvh), hs in groups.items()]
        pairs = [r for f in futs for r in f.result()]
    assert_within_tolerance(np.stack([g for g, _ in pairs]), np.stack([r for _, r in pairs]),
                            f"MHA 32 x 48 x 8192 per-token, {len(pairs)} sampled rows")
