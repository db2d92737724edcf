"""The oracle's page-tag integrity check against hand-worked cases (CPU only).

Workers AI post, §3 "共用 KV キャッシュの保護" (動作原理): every physical page
carries a tag that changes each time the page is handed out again; before
decode reads the cache, the pages a request uses are checked against the tags
it recorded when it mapped them, and a request that fails is aborted instead
of reading another request's data.  Each expected status below is worked out
by hand from that rule."""
import numpy as np

import oracle

OK, MISMATCH, BAD = 0, oracle.REQ_TAG_MISMATCH, oracle.REQ_BAD_INDEX


def _run(bt, tt, lens, tags, P=16):
    return oracle.verify_page_tags(np.array(bt, np.int32), np.array(tt, np.uint32), np.array(lens, np.int32), P,
                                   np.array(tags, np.uint32)).tolist()


def test_matching_tags_pass_and_a_reassigned_page_aborts_its_old_holder():
    # pool of 6 pages; request 0 holds pages 4, 1 (tags 9, 3); request 1 holds 0, 2, 5
    tags = [5, 3, 8, 0, 9, 2]
    bt = [[4, 1, -1], [0, 2, 5]]
    tt = [[9, 3, 0], [5, 8, 2]]
    assert _run(bt, tt, [32, 40], tags) == [OK, OK]
    # page 1 is freed and handed to another owner: its tag moves on (3 -> 4);
    # request 0 still holds the old mapping and must be aborted, request 1 is untouched
    tags[1] = 4
    assert _run(bt, tt, [32, 40], tags) == [MISMATCH, OK]
    # the new owner recorded the new tag
    assert _run([[1, -1, -1]], [[4, 0, 0]], [1], tags) == [OK]


def test_only_the_pages_a_request_reads_are_checked():
    tags = [1, 1, 1, 1]
    # L = 16 reads exactly one page (entry 0); entry 1 is stale but unread
    assert _run([[0, 1]], [[1, 7]], [16], tags) == [OK]
    # L = 17 reads two pages: the stale entry is now read
    assert _run([[0, 1]], [[1, 7]], [17], tags) == [MISMATCH]
    # an empty context reads nothing, whatever its row holds
    assert _run([[-5, 99]], [[0, 0]], [0], tags) == [OK]


def test_out_of_range_ids_and_lengths_are_index_errors():
    tags = [2, 2, 2]
    assert _run([[0, 3]], [[2, 2]], [20], tags) == [BAD]            # page 3 is outside the 3-page pool
    assert _run([[-1, 0]], [[2, 2]], [1], tags) == [BAD]             # negative id in a read entry
    assert _run([[0, 1]], [[2, 2]], [33], tags) == [BAD]             # 33 tokens need 3 pages of a 2-page row
    assert _run([[0, 1]], [[2, 2]], [-4], tags) == [BAD]             # negative length
    assert _run([[0, 1]], [[2, 5]], [33], tags) == [BAD | MISMATCH]  # both: clamped row still has a stale tag


def test_page_size_changes_which_entries_are_read():
    tags = [0, 0, 0, 0]
    bt, tt = [[0, 1, 2, 3]], [[0, 0, 0, 1]]
    assert _run(bt, tt, [48], tags, P=16) == [OK]        # pages 0-2
    assert _run(bt, tt, [49], tags, P=16) == [MISMATCH]  # page 3 now read
    assert _run(bt, tt, [192], tags, P=64) == [OK]       # 3 pages of 64
