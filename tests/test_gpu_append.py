"""kv_append_fp8 / kv_append_bf16 on the GPU against the oracle: cache bytes
and page/slot indexing must match bit for bit."""
import numpy as np
import pytest

import oracle
import synth
from synth import gen

from gpu_helpers import append_fp8_fn, oracle_caches, pf

pytestmark = pytest.mark.gpu


def _torch():
    import torch
    return torch


@pytest.mark.parametrize("scale", [1.0, 0.125, 0.37, 3.0, 1.0e-30, 7.0e30, 0.0096261156])
def test_every_bf16_pattern_encodes_like_the_oracle(scale):
    """All 65536 bf16 inputs (normals, subnormals, ties, +-inf, NaN) divided by
    the scale and rounded to e4m3, through the real append path."""
    torch = _torch()
    p = pf()
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    T, H, D, P = 4096, 1, 16, 16
    x = bits.reshape(T, H, D)
    perm = gen.permutation(gen.make_key(3, gen.TENSOR_PERM), T)  # one token per page-row, shuffled
    slots = perm.astype(np.int64)
    pages = T // P
    kc = torch.full((pages, H, P, D), 0xAB, dtype=torch.uint8, device="cuda")
    xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    p.kv_append_fp8(xd, None, kc, None, torch.from_numpy(slots).cuda(), scale)
    got = kc.cpu().numpy()
    ref = np.full((pages, H, P, D), 0xAB, np.uint8)
    oracle.kv_append(x, ref, slots, P, scale)
    f = gen.bf16_bits_to_f32(bits).reshape(T, H, D)
    is_nan_in = np.isnan(f)
    nan_pos = np.zeros_like(got, dtype=bool)
    nan_pos.reshape(-1, D)[slots] = is_nan_in.reshape(T, D)
    same = got == ref
    assert np.all(same | nan_pos), f"{int((~same & ~nan_pos).sum())} codes differ"
    # NaN inputs: any e4m3 NaN code is a valid result
    assert np.all(np.isin(got[nan_pos], [0x7F, 0xFF]))


def _wide_scales(n):
    """n seeded positive fp32 scales: exponent fields uniform over every
    normal binade (1 .. 254) with random mantissas, so x / s spans subnormal,
    normal and saturating e4m3 results for every bf16 input, plus the
    smallest subnormal and the largest finite scale."""
    key = gen.make_key(17, gen.TENSOR_PERM)
    idx = np.arange(n, dtype=np.uint64)
    e = gen.uniform_int(key, idx, 1, 254).astype(np.uint32)
    m = (gen.uniform_u64(key ^ 0x9E3779B97F4A7C15, idx) & np.uint64(0x7FFFFF)).astype(np.uint32)
    bits = (e << np.uint32(23)) | m
    bits[0] = 0x00000001  # 2^-149
    bits[1] = 0x7F7FFFFF  # largest finite fp32
    return bits.view(np.float32)


def test_every_bf16_pattern_over_512_scales_encodes_like_the_oracle():
    """All 65536 bf16 patterns against 512 seeded scales (256 calls, K and V
    each with its own scale) through the host-scalar append path: bit-exact
    codes, NaN inputs excepted (any NaN code)."""
    torch = _torch()
    p = pf()
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    T, H, D, P = 4096, 1, 16, 16
    x = bits.reshape(T, H, D)
    slots = np.arange(T, dtype=np.int64)
    pages = T // P
    scales = _wide_scales(512)
    xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    sl = torch.from_numpy(slots).cuda()
    nan_in = np.isnan(gen.bf16_bits_to_f32(bits)).reshape(pages, H, P, D)
    kcs = torch.empty((256, pages, H, P, D), dtype=torch.uint8, device="cuda")
    vcs = torch.empty_like(kcs)
    for i in range(256):
        p.kv_append_fp8(xd, xd, kcs[i], vcs[i], sl, float(scales[2 * i]), float(scales[2 * i + 1]))
    got_k, got_v = kcs.cpu().numpy(), vcs.cpu().numpy()
    bad = 0
    for i in range(512):
        ref = np.zeros((pages, H, P, D), np.uint8)
        oracle.kv_append(x, ref, slots, P, float(scales[i]))
        got = (got_k if i % 2 == 0 else got_v)[i // 2]
        same = got == ref
        bad += int((~same & ~nan_in).sum())
        assert np.all(np.isin(got[nan_in], [0x7F, 0xFF]))
    assert bad == 0, f"{bad} codes differ"


def test_tiny_gqa_cache_bytes_bit_exact():
    torch = _torch()
    p = pf()
    from synth import device as sdev
    w = synth.workload(synth.TINY_GQA).set_scales_host()
    st = sdev.setup_paged(w, append_fp8_fn(p, w))
    p.kv_append_fp8(st.k_new, st.v_new, st.k_cache, st.v_cache, st.step_slots, w.k_scale, w.v_scale)
    torch.cuda.synchronize()
    kc, vc = oracle_caches(w)
    assert np.array_equal(st.k_cache.cpu().numpy(), kc)
    assert np.array_equal(st.v_cache.cpu().numpy(), vc)


def test_negative_and_out_of_range_slots_write_nothing():
    torch = _torch()
    p = pf()
    T, H, D, P, pages = 6, 2, 32, 16, 4
    x = gen.normal_bf16(77, np.arange(T * H * D, dtype=np.uint64)).reshape(T, H, D)
    slots = np.array([5, -1, 63, 64, 1 << 40, 17], np.int64)  # 64 and 2^40 are beyond the cache
    kc = torch.full((pages, H, P, D), 0x5A, dtype=torch.uint8, device="cuda")
    vc = torch.full((pages, H, P, D), 0x5A, dtype=torch.uint8, device="cuda")
    xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    p.kv_append_fp8(xd, xd, kc, vc, torch.from_numpy(slots).cuda(), 0.01, 0.02)
    ref_k = np.full((pages, H, P, D), 0x5A, np.uint8)
    ref_v = ref_k.copy()
    keep = np.array([0, 2, 5])
    oracle.kv_append(x[keep], ref_k, slots[keep], P, 0.01)
    oracle.kv_append(x[keep], ref_v, slots[keep], P, 0.02)
    assert np.array_equal(kc.cpu().numpy(), ref_k)
    assert np.array_equal(vc.cpu().numpy(), ref_v)


def test_latent_rows_576_wide():
    torch = _torch()
    p = pf()
    T, D, P, pages = 70, 576, 64, 3
    x = gen.normal_bf16(91, np.arange(T * D, dtype=np.uint64)).reshape(T, 1, D)
    slots = gen.permutation(5, pages * P)[:T].astype(np.int64)
    c = torch.zeros((pages, 1, P, D), dtype=torch.uint8, device="cuda")
    p.kv_append_fp8(torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16), None, c, None,
                    torch.from_numpy(slots).cuda(), 0.0123)
    ref = np.zeros((pages, 1, P, D), np.uint8)
    oracle.kv_append(x, ref, slots, P, 0.0123)
    assert np.array_equal(c.cpu().numpy(), ref)


def test_bf16_cache_append_is_a_scatter_copy():
    torch = _torch()
    p = pf()
    w = synth.PagedWorkload("b", B=3, Hq=4, Hkv=2, D=128, P=16, context_lens=np.array([5, 40, 33]), seed=4)
    from synth import device as sdev
    st = sdev.setup_paged(w, lambda k, v, kc, vc, s: p.kv_append_bf16(k, v, kc, vc, s), bf16_cache=True,
                          scales_on_device=False)
    p.kv_append_bf16(st.k_new, st.v_new, st.k_cache, st.v_cache, st.step_slots)
    torch.cuda.synchronize()
    kc, vc = oracle_caches(w, bf16=True)
    assert np.array_equal(st.k_cache.view(torch.int16).cpu().numpy().view(np.uint16), kc)
    assert np.array_equal(st.v_cache.view(torch.int16).cpu().numpy().view(np.uint16), vc)


def test_host_side_argument_errors():
    torch = _torch()
    p = pf()
    x = torch.zeros((2, 1, 24), dtype=torch.bfloat16, device="cuda")
    c = torch.zeros((2, 1, 16, 24), dtype=torch.uint8, device="cuda")
    s = torch.zeros(2, dtype=torch.int64, device="cuda")
    with pytest.raises(p.PfkvError) as e:
        p.kv_append_fp8(x, None, c, None, s, 1.0)  # head_dim 24 is not a multiple of 16
    assert e.value.code == -2
    x = torch.zeros((2, 1, 32), dtype=torch.bfloat16, device="cuda")
    c = torch.zeros((2, 1, 16, 32), dtype=torch.uint8, device="cuda")
    with pytest.raises(p.PfkvError) as e:
        p.kv_append_fp8(x, None, c, None, s, 0.0)  # scale must be > 0
    assert e.value.code == -1
