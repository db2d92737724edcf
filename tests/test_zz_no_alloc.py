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

import synth
from gpu_helpers import assert_within_tolerance, pf, to_np_bf16

pytestmark = pytest.mark.gpu


def _host_state(w):
    """Caches filled through the product's append from host-generated rows."""
    import torch
    p = pf()
    w.set_scales_host()
    kc = torch.zeros((w.num_pages, w.Hkv, w.P, w.D), dtype=torch.uint8, device="cuda")
    vc = torch.zeros_like(kc)
    for b in range(w.B):
        t1 = int(w.context_lens[b])
        k = torch.from_numpy(w.kv_bits("k", b, 0, t1).view(np.int16)).cuda().view(torch.bfloat16)
        v = torch.from_numpy(w.kv_bits("v", b, 0, t1).view(np.int16)).cuda().view(torch.bfloat16)
        p.kv_append_fp8(k, v, kc, vc, torch.from_numpy(w.slots(b, 0, t1)).cuda(), w.k_scale, w.v_scale)
    q = torch.from_numpy(w.q_bits().view(np.int16)).cuda().view(torch.bfloat16)
    bt = torch.from_numpy(w.block_tables).cuda()
    cl = torch.from_numpy(w.context_lens).cuda()
    return p, kc, vc, q, bt, cl


@pytest.mark.parametrize("split", [0, 64])
def test_noalloc_matches_workspace_entry_point_on_two_calls(split):
    import torch
    w = synth.PagedWorkload("noalloc", B=3, Hq=32, Hkv=4, D=128, P=16, context_lens=np.array([700, 33, 1500]),
                            seed=31, n_new=0)
    p, kc, vc, q, bt, cl = _host_state(w)
    maxc = int(sum((int(L) + split - 1) // split for L in w.context_lens)) if split else 0
    ref = torch.empty_like(q)
    ref_lse = torch.empty((w.B, w.Hq), dtype=torch.float32, device="cuda")
    p.paged_decode_attn(ref, q, kc, vc, bt, cl, w.k_scale, w.v_scale, w.softmax_scale, kv_split_tokens=split,
                        lse_out=ref_lse, max_total_chunks=maxc)
    torch.cuda.synchronize()
    ref_np = to_np_bf16(ref)
    for _ in range(2):  # the shared scratch keeps the previous call's bytes
        out = torch.full_like(q, float("nan"))
        lse = torch.full((w.B, w.Hq), float("nan"), dtype=torch.float32, device="cuda")
        status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        p.paged_decode_attn_noalloc(out, q, kc, vc, bt, cl, w.k_scale, w.v_scale, w.softmax_scale,
                                    kv_split_tokens=split, max_total_chunks=maxc, lse_out=lse,
                                    status_out=status)
        torch.cuda.synchronize()
        assert status.item() == 0
        assert_within_tolerance(to_np_bf16(out), ref_np, "noalloc vs workspace entry point")
        np.testing.assert_allclose(lse.cpu().numpy(), ref_lse.cpu().numpy(), rtol=1e-6, atol=1e-6)


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
