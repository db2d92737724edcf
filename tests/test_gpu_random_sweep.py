"""Seeded random configurations of the decode and multi-query paths, each
compared element by element with the oracle.

The hand-picked cases in test_gpu_paged_decode.py and test_gpu_prefill.py
cover each branch once; here every parameter the entry points accept is drawn
at random within the documented limits (head groups 1-16, pages of 16 to 128
tokens including sizes that are not powers of two, empty and one-token
contexts, contexts ending on and next to page and tile boundaries, explicit
chunking), so that combinations nobody picked are exercised too.  The draws
are fixed by the case number, so a failure names a reproducible case."""
import numpy as np
import pytest

import synth

from gpu_helpers import pf
from test_gpu_paged_decode import _full_check
from test_gpu_prefill import _check_small

pytestmark = pytest.mark.gpu


def _edge_len(r, P):
    return int(r.choice([1, 15, 16, 17, P - 1, P, P + 1, 2 * P, 127, 128, 129]))


def _decode_case(case):
    r = np.random.default_rng(1000 + case)
    Hkv = int(r.choice([1, 2, 4]))
    G = int(r.integers(1, 17))
    P = int(r.choice([16, 32, 48, 64, 96, 128]))
    B = int(r.integers(1, 10))
    lens = r.integers(1, 900, size=B)
    for i in range(B):
        u = r.random()
        if u < 0.15:
            lens[i] = 0
        elif u < 0.35:
            lens[i] = _edge_len(r, P)
    if lens.max() == 0:  # a cache holds at least one page
        lens[0] = _edge_len(r, P)
    split = int(r.choice([0, 0, 16, 32, 80, 256]))
    return Hkv, G, P, lens, split


@pytest.mark.parametrize("case", range(40))
def test_decode_random_configuration(case):
    Hkv, G, P, lens, split = _decode_case(case)
    w = synth.PagedWorkload(f"sweep{case}", B=len(lens), Hq=G * Hkv, Hkv=Hkv, D=128, P=P, context_lens=lens,
                            n_new=1 if lens.min() > 0 else 0, seed=case)
    _full_check(pf(), w, split=split)


def _prefill_case(case):
    r = np.random.default_rng(2000 + case)
    Hkv = int(r.choice([1, 2]))
    G = int(r.choice([1, 2, 4, 8, 16]))
    P = int(r.choice([16, 32, 48, 64, 96, 128]))
    B = int(r.integers(1, 6))
    lens = r.integers(1, 700, size=B)
    for i in range(B):
        if r.random() < 0.3:
            lens[i] = max(1, _edge_len(r, P))
    q_lens = np.array([int(r.integers(0, min(int(L), 48) + 1)) for L in lens])
    if q_lens.max() == 0:
        q_lens[0] = 1
    split = int(r.choice([0, 0, 64, 128, 192]))
    return Hkv, G, P, lens, q_lens, split


@pytest.mark.parametrize("case", range(30))
def test_prefill_random_configuration(case):
    Hkv, G, P, lens, q_lens, split = _prefill_case(case)
    w = synth.PagedWorkload(f"psweep{case}", B=len(lens), Hq=G * Hkv, Hkv=Hkv, D=128, P=P,
                            context_lens=lens, n_new=1, seed=50 + case)
    _check_small(w, q_lens=q_lens, split=split, max_q=int(q_lens.max()))


def _mla_case(case):
    r = np.random.default_rng(3000 + case)
    H = int(r.choice([16, 32, 64, 96, 128]))
    P = int(r.choice([16, 32, 64, 128]))
    B = int(r.choice([1, 2, 3, 5, 6, 40]))
    lens = r.integers(1, 3000 if B < 40 else 300, size=B)
    for i in range(B):
        if r.random() < 0.3:
            lens[i] = _edge_len(r, P)
    K = 0 if case % 3 == 0 else int(r.choice([1, 31, 32, 33, 256, 700]))  # 0: every token
    topk = None
    if K:
        # distinct positions at random places of each row, the rest padding;
        # every other case lists them out of order
        topk = np.full((B, K), -1, np.int32)
        for b in range(B):
            n = int(r.integers(0, min(K, int(lens[b])) + 1))
            pos = r.choice(int(lens[b]), size=n, replace=False)
            if case % 2 == 0:
                pos = np.sort(pos)
            topk[b, np.sort(r.choice(K, size=n, replace=False))] = pos
    return H, P, lens, topk


@pytest.mark.parametrize("case", range(24))
def test_mla_random_configuration(case):
    from test_gpu_mla_and_validate import _mla_check, _setup_mla
    H, P, lens, topk = _mla_case(case)
    p = pf()
    m = synth.MlaWorkload(f"msweep{case}", B=len(lens), H=H, context_lens=lens, topk_n=0, P=P, seed=70 + case)
    st = _setup_mla(p, m)
    if topk is None:
        _mla_check(p, m, st, what=f"mla sweep {case}")
    else:
        _mla_check(p, m, st, topk=topk, what=f"mla sweep {case}")


def _scaled_case(case):
    r = np.random.default_rng(4000 + case)
    Hkv = int(r.choice([1, 2, 4]))
    G = int(r.integers(1, 17))
    P = int(r.choice([16, 32, 48, 64, 96, 128]))
    B = int(r.integers(1, 8))
    lens = r.integers(1, 600, size=B)
    for i in range(B):
        u = r.random()
        if u < 0.15:
            lens[i] = 0
        elif u < 0.35:
            lens[i] = _edge_len(r, P)
    if lens.max() == 0:
        lens[0] = _edge_len(r, P)
    split = int(r.choice([0, 0, 16, 48, 128]))
    spread = int(r.choice([0, 3, 6, 12]))
    zero_rows = bool(r.random() < 0.4)
    return Hkv, G, P, lens, split, spread, zero_rows


@pytest.mark.parametrize("case", range(24))
def test_scaled_append_and_decode_random_configuration(case):
    """The scaled append writes the oracle's codes and scales bit for bit; the
    decode over those bytes matches the oracle's decode."""
    import oracle
    from oracle_helpers import oracle_fill_scaled
    from test_gpu_scales import GRANS, _decode, _gpu_fill, _scale_rows_used
    from gpu_helpers import assert_within_tolerance
    gran = GRANS[case % 3]
    Hkv, G, P, lens, split, spread, zero_rows = _scaled_case(case)
    p = pf()
    w = synth.PagedWorkload(f"ssweep{case}", B=len(lens), Hq=G * Hkv, Hkv=Hkv, D=128, P=P, context_lens=lens,
                            seed=90 + case)
    kc, vc, ks, vs = _gpu_fill(p, w, gran, spread, zero_rows)
    okc, ovc, oks, ovs = oracle_fill_scaled(w, gran, spread, zero_rows)
    assert np.array_equal(kc.cpu().numpy(), okc)
    assert np.array_equal(vc.cpu().numpy(), ovc)
    if gran == oracle.SCALE_TOKEN:
        for got, ref in ((ks, oks), (vs, ovs)):
            assert np.array_equal(_scale_rows_used(w, got.cpu().numpy()).view(np.uint32),
                                  _scale_rows_used(w, ref).view(np.uint32))
    out, lse, status = _decode(p, w, kc, vc, gran, ks, vs, split)
    assert status == 0
    ref, ref_lse = oracle.paged_decode_scaled(w.q_bits(), okc, ovc, gran, oks, ovs, w.block_tables,
                                              w.context_lens, w.P, w.softmax_scale, w.Hkv)
    assert_within_tolerance(out, ref, f"scaled sweep {case} gran {gran}")
    fin = np.isfinite(ref_lse)
    assert np.all(~np.isfinite(lse[~fin]))
    np.testing.assert_allclose(lse[fin], ref_lse[fin], rtol=2e-5, atol=2e-4)
