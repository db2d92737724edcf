"""verify_page_tags on the GPU against the oracle: planted tag mismatches and
bad indices over random and full-size block tables (statuses bit-exact)."""
import numpy as np
import pytest

import oracle
import synth

from gpu_helpers import pf

pytestmark = pytest.mark.gpu


def _gpu(p, bt, tt, lens, P, tags):
    import torch
    d = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a).astype(dt)).cuda()
    st = torch.full((bt.shape[0],), -7, dtype=torch.int32, device="cuda")
    p.verify_page_tags(d(bt, np.int32), d(tt.view(np.int32), np.int32), d(lens, np.int32), P,
                       d(tags.view(np.int32), np.int32), st)
    torch.cuda.synchronize()
    return st.cpu().numpy()


def test_random_tables_with_planted_faults_match_oracle():
    p = pf()
    rng = np.random.default_rng(11)
    B, maxp, P, pages = 300, 96, 16, 5000
    bt = rng.integers(0, pages, (B, maxp)).astype(np.int32)
    tags = rng.integers(0, 2**32, pages, dtype=np.uint64).astype(np.uint32)
    tt = tags[bt]
    lens = rng.integers(0, maxp * P + 1, B).astype(np.int32)
    lens[:5] = [0, 1, maxp * P, maxp * P + 1, -3]
    # stale tags and bad ids, some inside and some past each request's context
    for _ in range(120):
        b, i = rng.integers(0, B), rng.integers(0, maxp)
        if rng.random() < 0.7:
            tt[b, i] ^= np.uint32(1 + rng.integers(0, 1000))
        else:
            bt[b, i] = pages + rng.integers(0, 10) if rng.random() < 0.5 else -1 - rng.integers(0, 10)
    ref = oracle.verify_page_tags(bt, tt, lens, P, tags)
    got = _gpu(p, bt, tt, lens, P, tags)
    assert np.array_equal(got, ref)
    assert (ref == 0).sum() > 50 and (ref & oracle.REQ_TAG_MISMATCH).sum() > 20 and (ref & oracle.REQ_BAD_INDEX).sum() > 5


@pytest.mark.parametrize("name", ["mha_b32_h48_l8192_p16", "long_splitkv_b8_h64kv8_p64"])
def test_full_size_tables_flag_exactly_the_planted_request(name):
    p = pf()
    w = synth.workload(name)
    tags = np.arange(w.num_pages, dtype=np.uint32) * np.uint32(2654435761)
    bt = w.block_tables.astype(np.int32)
    tt = np.where(bt >= 0, tags[np.clip(bt, 0, None)], 0).astype(np.uint32)
    lens = w.context_lens.astype(np.int32)
    assert not _gpu(p, bt, tt, lens, w.P, tags).any()
    b = w.B // 2
    last = (int(lens[b]) - 1) // w.P        # the last page request b reads
    tags[bt[b, last]] += np.uint32(1)       # that page is handed out again
    got = _gpu(p, bt, tt, lens, w.P, tags)
    ref = oracle.verify_page_tags(bt, tt, lens, w.P, tags)
    assert np.array_equal(got, ref)
    assert got[b] == oracle.REQ_TAG_MISMATCH and got.sum() == got[b]
