"""KV-bytes formula against the pages' worked example; allocated cache bytes of
every workload against that formula; byte halving of FP8; and the seeded input
generator (CPU only)."""
import json
import math
import os

import numpy as np
import torch

import oracle
import synth
from synth import gen

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_kv_bytes_worked_example_from_the_page():
    g = json.load(open(os.path.join(GOLDEN, "kv_bytes_worked_example.json")))
    per_tok = oracle.kv_bytes(g["layers"], g["kv_heads"], g["head_dim"], 1, g["bytes_per_elem"])
    assert per_tok == 1_474_560
    assert round(per_tok / 1e6, 2) == g["per_token_MB_approx"]
    gb8 = oracle.kv_bytes(g["layers"], g["kv_heads"], g["head_dim"], g["seq_8k_tokens"], g["bytes_per_elem"]) / 1e9
    gb16 = oracle.kv_bytes(g["layers"], g["kv_heads"], g["head_dim"], g["seq_16k_tokens"], g["bytes_per_elem"]) / 1e9
    assert abs(gb8 - g["seq_8k_GB_approx"]) < 0.5
    assert abs(gb16 - g["seq_16k_GB_approx"]) < 1.0


def test_fp8_halves_bytes_and_doubles_capacity():
    g = json.load(open(os.path.join(GOLDEN, "fp8_capacity_doubling.json")))
    bf16 = oracle.kv_bytes(1, 48, 128, 8192, g["bytes_per_elem_bf16"])
    fp8 = oracle.kv_bytes(1, 48, 128, 8192, g["bytes_per_elem_fp8"])
    assert bf16 == 2 * fp8
    # the page's capacity figures double within their rounding
    assert abs(g["fp8_tokens_approx"] / g["bf16_tokens_approx"] - 2.0) < 0.01


def test_allocated_cache_bytes_equal_formula_for_every_paged_workload():
    for name in (synth.TINY_GQA, synth.MHA_B32, synth.GQA_PREFIX, synth.LONG_SPLITKV):
        w = synth.workload(name)
        # a cache holding exactly the workload's pages, one layer
        pages_needed = int(w.pages_per_req.sum()) - max(w.shared_requests - 1, 0) * (w.shared_tokens // w.P)
        alloc = 2 * pages_needed * w.Hkv * w.P * w.D  # K + V, e4m3
        padded_tokens = pages_needed * w.P
        assert alloc == oracle.kv_bytes(1, w.Hkv, w.D, padded_tokens, 1)
        if all(int(L) % w.P == 0 for L in w.context_lens) and w.shared_requests == 0:
            assert alloc == w.kv_bytes(1)
    w2 = synth.workload(synth.MHA_B32)
    assert w2.kv_bytes(1) == 3_221_225_472
    assert w2.kv_bytes(2) == 2 * w2.kv_bytes(1)
    assert synth.workload(synth.LONG_SPLITKV).kv_bytes(1) == 11_542_724_608


def test_generator_is_deterministic_and_roughly_standard_normal():
    key = gen.make_key(0, gen.TENSOR_K)
    idx = np.arange(2_000_000, dtype=np.uint64)
    a = gen.normal_f32(key, idx)
    b = gen.normal_f32(key, idx)
    assert np.array_equal(a, b)
    assert abs(a.mean()) < 3e-3 and abs(a.std() - 1.0) < 3e-3
    assert a.min() >= -6.0 and a.max() <= 6.0
    # values are multiples of 2^-16 (exact construction)
    assert np.all(a * 65536 == np.round(a * 65536))
    assert gen.make_key(0, gen.TENSOR_K) != gen.make_key(1, gen.TENSOR_K)


def test_bf16_rounding_matches_torch_cast():
    x = gen.normal_f32(12345, np.arange(500_000, dtype=np.uint64)) * np.float32(37.25)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(gen.f32_to_bf16_bits(x), ref)


def test_workload_tables_are_valid():
    for name in (synth.TINY_GQA, synth.MHA_B32, synth.GQA_PREFIX, synth.LONG_SPLITKV):
        w = synth.workload(name)
        used = []
        for b in range(w.B):
            npg = int(w.pages_per_req[b])
            row = w.block_tables[b, :npg]
            assert np.all((row >= 0) & (row < w.num_pages))
            assert np.all(w.block_tables[b, npg:] == -1)
            used.append(row)
        u = np.concatenate(used)
        shared_dups = max(w.shared_requests - 1, 0) * (w.shared_tokens // w.P)
        assert len(np.unique(u)) == len(u) - shared_dups
    w3 = synth.workload(synth.GQA_PREFIX)
    assert np.all(w3.context_lens >= 256) and np.all(w3.context_lens <= 32768)
    assert np.all(w3.context_lens[:16] >= 2048 + 16)
    assert np.all(w3.block_tables[1:16, :128] == w3.block_tables[0, :128])
    assert 2000 < np.median(w3.context_lens) < 8000
    w1 = synth.workload(synth.TINY_GQA)
    assert np.all((w1.context_lens >= 16) & (w1.context_lens <= 300)) and w1.num_pages == 128


def test_mla_topk_lists_are_unique_sorted_in_range():
    m = synth.workload(synth.MLA_TOPK)
    assert m.topk.shape == (64, 2048)
    assert np.all(np.diff(m.topk, axis=1) > 0)
    assert m.topk.min() >= 0 and m.topk.max() < 65536
    assert m.algorithmic_bytes()["kv"] == 64 * 2048 * 576
    assert m.flops() == 64 * 2048 * (2 * 128 * 576 + 2 * 128 * 512)


def test_slots_follow_block_tables_and_shared_tokens_map_to_request_0():
    w = synth.workload(synth.GQA_PREFIX)
    sl = w.slots(5, 100, 140)
    t = np.arange(100, 140)
    assert np.array_equal(sl, w.block_tables[5, t // 16].astype(np.int64) * 16 + t % 16)
    assert np.array_equal(w.kv_bits("k", 7, 0, 4), w.kv_bits("k", 0, 0, 4))
    assert not np.array_equal(w.kv_bits("k", 7, 2048, 2050), w.kv_bits("k", 0, 2048, 2050))
    runs = list(w.kv_runs(3, 2040, 2060))
    assert len(runs) == 2 and runs[0][1] == 2048


def test_host_c_generator_twin_matches_numpy_definition():
    key = gen.make_key(3, gen.TENSOR_V)
    idx = (np.arange(200_000, dtype=np.uint64) * np.uint64(977)) + np.uint64(1 << 40)
    assert np.array_equal(gen.normal_bf16(key, idx), gen.normal_bf16_numpy(key, idx))
    assert np.array_equal(gen.normal_bf16_range(key, 5, 3000),
                          gen.normal_bf16_numpy(key, np.arange(5, 3005, dtype=np.uint64)))
    rows = gen.normal_bf16_rows(key, 11, 40, 16, 1000)
    ref = gen.normal_bf16_numpy(key, (np.uint64(11) + np.arange(40, dtype=np.uint64)[:, None] * np.uint64(1000)
                                      + np.arange(16, dtype=np.uint64)[None, :]).reshape(-1)).reshape(40, 16)
    assert np.array_equal(rows, ref)


def test_workload_rows_follow_the_documented_counter_layout():
    w = synth.workload(synth.GQA_PREFIX)
    b, t0, t1 = 20, 100, 131
    idx = (((np.int64(b) << 21) + np.arange(t0, t1))[:, None] * (w.Hkv * w.D)
           + np.arange(w.Hkv * w.D)[None, :]).astype(np.uint64)
    ref = gen.normal_bf16_numpy(w.key_k, idx.reshape(-1)).reshape(t1 - t0, w.Hkv, w.D)
    assert np.array_equal(w.kv_bits("k", b, t0, t1), ref)
    assert np.array_equal(w.kv_head_bits("k", b, 5, t0, t1), ref[:, 5, :])
    # shared prefix tokens of request 3 are request 0's
    assert np.array_equal(w.kv_head_bits("v", 3, 2, 2040, 2056)[:8], w.kv_head_bits("v", 0, 2, 2040, 2048))
