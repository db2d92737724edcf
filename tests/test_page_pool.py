"""The library's host page pool (pfkv_pool_*, pfkv_block_hash,
pfkv_slots_from_table) against the oracle on seeded random scenarios: block
tables, tags, cached lengths, reference counts and the free list agree
exactly (CPU only; no CUDA call)."""
import numpy as np
import pytest

from oracle import page_pool as op


@pytest.fixture(scope="module")
def pf():
    import paged_fp8_kv_02_gb300 as pf
    from paged_fp8_kv_02_gb300 import _build
    _build.build_pfkv()
    return pf


def test_block_hash_matches_the_oracle(pf):
    rng = np.random.default_rng(5)
    for n in (0, 1, 16, 64):
        toks = rng.integers(-2**31, 2**31, n).astype(np.int32)
        parent = int(rng.integers(0, 2**63))
        assert pf.block_hash(parent, toks) == op.block_hash(parent, toks.tolist())


@pytest.mark.parametrize("seed,P", [(0, 16), (1, 64), (2, 4)])
def test_random_map_and_release_sequences_match_the_oracle(pf, seed, P):
    rng = np.random.default_rng(seed)
    num_pages, max_pages = 300, 40
    lib, ref = pf.PagePool(num_pages, P), op.PagePool(num_pages, P)
    prefixes = [rng.integers(0, 50000, int(rng.integers(0, 6 * P))).tolist() for _ in range(4)]
    live = []
    for step in range(120):
        if live and (rng.random() < 0.35 or lib.num_free() < 3 * max_pages // 2):
            k = int(rng.integers(0, len(live)))
            row, n = live.pop(k)
            lib.release(row, n)
            ref.release(row.tolist(), n)
        else:
            pre = prefixes[int(rng.integers(0, len(prefixes)))]
            toks = pre + rng.integers(0, 50000, int(rng.integers(0, 5 * P))).tolist()
            toks = toks[: max_pages * P]
            try:
                exp = ref.map_request(toks, max_pages)
            except op.NoPages:
                with pytest.raises(pf.PfkvError):
                    lib.map_request(np.array(toks, np.int32), max_pages)
                continue
            row, tags, cached = lib.map_request(np.array(toks, np.int32), max_pages)
            assert row.tolist() == exp[0] and tags.tolist() == exp[1] and cached == exp[2], step
            live.append((row, -(-len(toks) // P)))
        assert lib.num_free() == len(ref.free)
        assert all(lib.refcount(p) == ref.ref[p] for p in range(num_pages))
        assert lib.page_tags().tolist() == ref.tag


def test_release_of_a_page_not_held_changes_nothing(pf):
    pool = pf.PagePool(16, 4)
    row, _, _ = pool.map_request(np.arange(6, dtype=np.int32), 4)
    bad = row.copy()
    bad[1] = 9  # never handed out
    with pytest.raises(pf.PfkvError):
        pool.release(bad, 2)
    assert pool.refcount(int(row[0])) == 1 and pool.num_free() == 14


def test_slots_follow_the_table(pf):
    row = np.array([7, 2, 11, -1], np.int32)
    sl = pf.slots_from_table(row, 16, 5, 40)
    t = np.arange(5, 45)
    assert np.array_equal(sl, row[t // 16].astype(np.int64) * 16 + t % 16)
    with pytest.raises(pf.PfkvError):
        pf.slots_from_table(row, 16, 40, 10)  # tokens 48.. fall in the unmapped 4th entry


def test_a_page_listed_twice_needs_two_holders(pf):
    """Each entry of a released row drops one holder.  A page held once but
    listed twice is an error that changes nothing (it would otherwise return
    to the free list while still counted); a shared page held by two requests
    may be listed twice and is then freed once."""
    from oracle.page_pool import PagePool as OraclePool
    P = 4
    lib, ref = pf.PagePool(16, P), OraclePool(16, P)
    toks = np.arange(8, dtype=np.int32)              # two full blocks
    row, _, _ = lib.map_request(toks, 4)
    rrow, _, _ = ref.map_request(toks, 4)
    assert list(row[:2]) == list(rrow[:2])
    dup = np.array([row[0], row[0]], np.int32)
    with pytest.raises(pf.PfkvError):
        lib.release(dup, 2)
    with pytest.raises(ValueError):
        ref.release(list(dup), 2)
    assert lib.refcount(int(row[0])) == 1 and lib.num_free() == 14
    assert ref.ref[int(row[0])] == 1 and len(ref.free) == 14
    # a second request shares both blocks: each page now has two holders
    row2, _, cached = lib.map_request(toks, 4)
    rrow2, _, rcached = ref.map_request(toks, 4)
    assert cached == rcached == 8 and list(row2[:2]) == list(row[:2]) == list(rrow2[:2])
    lib.release(dup, 2)
    ref.release(list(dup), 2)
    assert lib.refcount(int(row[0])) == 0 and ref.ref[int(row[0])] == 0
    assert lib.num_free() == len(ref.free) == 15
    assert lib.refcount(int(row[1])) == 2
    with pytest.raises(ValueError):
        lib.release(row, 5)                           # more entries than the row holds
