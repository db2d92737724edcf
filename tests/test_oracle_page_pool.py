"""The page-pool / prefix-cache oracle against the pages and published values
(CPU only): FNV-1a test vectors, the explainer's worked example (100 shared
tokens with 16-token blocks reuse 96), the chaining property of block hashes,
and the free-list / reference-count / tag behaviour the pages describe."""
import numpy as np
import pytest

from oracle import page_pool as op


def test_fnv1a64_published_test_vectors():
    # the FNV-1a 64-bit reference values for "", "a" and "foobar"
    assert op.fnv1a64(b"") == 0xCBF29CE484222325
    assert op.fnv1a64(b"a") == 0xAF63DC4C8601EC8C
    assert op.fnv1a64(b"foobar") == 0x85944171F73967E8


def test_block_hash_covers_tokens_and_parent():
    t = list(range(16))
    assert op.block_hash(0, t) == op.fnv1a64(bytes(8) + b"".join(x.to_bytes(4, "little") for x in t))
    assert op.block_hash(1, t) != op.block_hash(0, t)
    assert op.block_hash(0, t[:15] + [99]) != op.block_hash(0, t)


def test_changing_a_token_changes_its_block_and_every_later_one():
    rng = np.random.default_rng(3)
    toks = rng.integers(0, 32000, 160).tolist()
    h = op.chain_hashes(toks, 16)
    assert len(h) == 10
    for pos in (0, 37, 100, 159):
        t2 = list(toks)
        t2[pos] += 1
        h2 = op.chain_hashes(t2, 16)
        blk = pos // 16
        assert h2[:blk] == h[:blk] and all(a != b for a, b in zip(h2[blk:], h[blk:]))


def test_explainer_example_100_shared_tokens_reuse_96():
    pool = op.PagePool(64, 16)
    shared = list(range(1000, 1100))
    _, _, c0 = pool.map_request(shared + [1, 2, 3], 16)
    _, _, c1 = pool.map_request(shared + [7, 8, 9, 10], 16)
    assert c0 == 0 and c1 == 96


@pytest.mark.parametrize("shared,expect", [(0, 0), (15, 0), (16, 16), (31, 16), (32, 32), (33, 32)])
def test_hits_floor_to_whole_blocks(shared, expect):
    pool = op.PagePool(64, 16)
    base = list(range(500, 600))
    pool.map_request(base, 8)
    _, _, cached = pool.map_request(base[:shared] + list(range(9000, 9050)), 8)
    assert cached == expect


def test_free_list_refcounts_and_tags():
    pool = op.PagePool(8, 4)
    a_row, a_tags, _ = pool.map_request(list(range(10)), 4)       # 3 pages: 2 full blocks + a tail
    assert a_row == [0, 1, 2, -1] and a_tags == [1, 1, 1, 0] and len(pool.free) == 5
    b_row, _, cached = pool.map_request(list(range(8)) + [77], 4)  # shares the 2 full blocks
    assert cached == 8 and b_row[:2] == [0, 1] and b_row[2] == 3
    assert pool.ref[:4] == [2, 2, 1, 1]
    pool.release(a_row, 3)
    assert pool.ref[:4] == [1, 1, 0, 1] and 2 in pool.free
    pool.release(b_row, 3)
    assert sorted(pool.free) == list(range(8)) and pool.prefix == {}
    # the last page freed (3) comes back first, and its tag moves on
    c_row, c_tags, cached = pool.map_request(list(range(100, 104)), 4)
    assert cached == 0 and c_row[0] == 3 and c_tags[0] == 2 == pool.tag[3]
    with pytest.raises(op.NoPages):
        pool.map_request(list(range(200, 240)), 16)
