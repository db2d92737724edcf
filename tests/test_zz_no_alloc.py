"""The allocation-free decode entry point, for callers that cannot allocate
device memory on their decode path (an engine that reserves all device memory
up front and hands it out from its own pool, or a per-token path that cannot
pay for cudaMalloc's synchronisation and latency).

It is called through the C ABI and must agree with pfkv_paged_decode_attn (the
entry point that takes a caller-allocated workspace) on the same inputs, on two
calls in a row, since all calls share the library's one fixed scratch array.
This file is collected last so that a run stopping at its first failure has
already run every other test; it builds its inputs on the host, so it also
passes alone in a fresh process."""
import numpy as np
import pytest

import oracle
import synth
from gpu_helpers import assert_within_tolerance, oracle_caches, pf

pytestmark = pytest.mark.gpu


def _host_state(w, bf16=False):
    """Caches filled through the product's append from host-generated rows."""
    import torch
    p = pf()
    if bf16:
        kc = torch.zeros((w.num_pages, w.Hkv, w.P, w.D), dtype=torch.bfloat16, device="cuda")
        w.k_scale = w.v_scale = 1.0
    else:
        w.set_scales_host()
        kc = torch.zeros((w.num_pages, w.Hkv, w.P, w.D), dtype=torch.uint8, device="cuda")
    vc = torch.zeros_like(kc)
    for b in range(w.B):
        t1 = int(w.context_lens[b])
        k = torch.from_numpy(w.kv_bits("k", b, 0, t1).view(np.int16)).cuda().view(torch.bfloat16)
        v = torch.from_numpy(w.kv_bits("v", b, 0, t1).view(np.int16)).cuda().view(torch.bfloat16)
        sl = torch.from_numpy(w.slots(b, 0, t1)).cuda()
        if bf16:
            p.kv_append_bf16(k, v, kc, vc, sl)
        else:
            p.kv_append_fp8(k, v, kc, vc, sl, w.k_scale, w.v_scale)
    q = torch.from_numpy(w.q_bits().view(np.int16)).cuda().view(torch.bfloat16)
    bt = torch.from_numpy(w.block_tables).cuda()
    cl = torch.from_numpy(w.context_lens).cuda()
    return p, kc, vc, q, bt, cl


def _chunks(w, split):
    return int(sum((int(L) + split - 1) // split for L in w.context_lens)) if split else 0


def _workspace_call(p, w, st, split):
    import torch
    _, kc, vc, q, bt, cl = st
    out = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq), dtype=torch.float32, device="cuda")
    p.paged_decode_attn(out, q, kc, vc, bt, cl, w.k_scale, w.v_scale, w.softmax_scale, kv_split_tokens=split,
                        lse_out=lse, max_total_chunks=_chunks(w, split))
    torch.cuda.synchronize()
    return out.view(torch.int16).cpu().numpy(), lse.cpu().numpy()


def _noalloc_call(p, w, st, split):
    import torch
    _, kc, vc, q, bt, cl = st
    out = torch.full_like(q, float("nan"))
    lse = torch.full((w.B, w.Hq), float("nan"), dtype=torch.float32, device="cuda")
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    p.paged_decode_attn_noalloc(out, q, kc, vc, bt, cl, w.k_scale, w.v_scale, w.softmax_scale,
                                kv_split_tokens=split, max_total_chunks=_chunks(w, split), lse_out=lse,
                                status_out=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    return out.view(torch.int16).cpu().numpy(), lse.cpu().numpy()


@pytest.mark.parametrize("split", [0, 64])
def test_noalloc_matches_workspace_entry_point_on_two_calls(split):
    """Same kernels, same grid, same inputs: the output and lse bits must be
    identical to the workspace entry point's, on two calls in a row."""
    w = synth.PagedWorkload("noalloc", B=3, Hq=32, Hkv=4, D=128, P=16, context_lens=np.array([700, 33, 1500]),
                            seed=31, n_new=0)
    st = _host_state(w)
    p = st[0]
    ref, ref_lse = _workspace_call(p, w, st, split)
    for _ in range(2):  # the shared scratch keeps the previous call's bytes
        out, lse = _noalloc_call(p, w, st, split)
        assert np.array_equal(out, ref)
        assert np.array_equal(lse.view(np.uint32), ref_lse.view(np.uint32))


def test_noalloc_smaller_call_after_a_larger_one_matches_the_oracle():
    """A larger call (more requests, 64-token chunks) leaves its tile starts,
    unit starts and partial states in the shared scratch; a smaller call with
    another batch and split that follows must not read any of them: its output
    equals the workspace entry point's bit for bit and the oracle's within the
    stated tolerance."""
    big = synth.PagedWorkload("noalloc_big", B=7, Hq=16, Hkv=2, D=128, P=16,
                              context_lens=np.array([900, 3000, 17, 2500, 640, 1, 1999]), seed=33, n_new=0)
    small = synth.PagedWorkload("noalloc_small", B=2, Hq=16, Hkv=2, D=128, P=16, context_lens=np.array([450, 61]),
                                seed=34, n_new=0)
    st_big = _host_state(big)
    st_small = _host_state(small)
    p = st_big[0]
    ref, ref_lse = _workspace_call(p, small, st_small, 16)
    _noalloc_call(p, big, st_big, 64)
    out, lse = _noalloc_call(p, small, st_small, 16)
    assert np.array_equal(out, ref)
    assert np.array_equal(lse.view(np.uint32), ref_lse.view(np.uint32))
    kc, vc = oracle_caches(small)
    oref, olse = oracle.paged_decode(small.q_bits(), kc, vc, small.block_tables, small.context_lens, small.P,
                                     small.k_scale, small.v_scale, small.softmax_scale, small.Hkv)
    got = out.view(np.uint16).astype(np.uint32) << 16
    assert_within_tolerance(got.view(np.float32).astype(np.float64), oref, "noalloc after a larger call")
    np.testing.assert_allclose(lse, olse, rtol=2e-5, atol=2e-4)


def test_noalloc_bf16_cache_matches_workspace_entry_point():
    w = synth.PagedWorkload("noalloc_bf16", B=2, Hq=8, Hkv=2, D=128, P=16, context_lens=np.array([333, 90]),
                            seed=35, n_new=0)
    st = _host_state(w, bf16=True)
    p = st[0]
    ref, ref_lse = _workspace_call(p, w, st, 0)
    for _ in range(2):
        out, lse = _noalloc_call(p, w, st, 0)
        assert np.array_equal(out, ref)
        assert np.array_equal(lse.view(np.uint32), ref_lse.view(np.uint32))


def test_noalloc_empty_batch_clears_the_status_word():
    import torch
    p = pf()
    q = torch.zeros((0, 8, 128), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((1, 2, 16, 128), dtype=torch.uint8, device="cuda")
    bt = torch.zeros((0, 1), dtype=torch.int32, device="cuda")
    cl = torch.zeros((0,), dtype=torch.int32, device="cuda")
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    p.paged_decode_attn_noalloc(q, q, kc, kc, bt, cl, 1.0, 1.0, 0.1, status_out=status)
    torch.cuda.synchronize()
    assert status.item() == 0


def test_noalloc_rejects_calls_beyond_its_scratch():
    import torch
    p = pf()
    B, Hq, Hkv, P = 4000, 64, 4, 16  # needs well over 64 MiB of partial-state slots
    q = torch.zeros((B, Hq, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    kc = torch.zeros((4, Hkv, P, 128), dtype=torch.uint8, device="cuda")
    bt = torch.zeros((B, 1), dtype=torch.int32, device="cuda")
    cl = torch.ones((B,), dtype=torch.int32, device="cuda")
    assert p.paged_decode_workspace_size(B, Hq, Hkv, 128) > (64 << 20)
    with pytest.raises(p.PfkvError) as e:
        p.paged_decode_attn_noalloc(out, q, kc, kc, bt, cl, 1.0, 1.0, 0.1)
    assert e.value.code == -5
    assert "64 MiB" in str(e.value)
