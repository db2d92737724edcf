"""End to end through the host page pool: the shared-prefix GQA workload's block tables and slot
mappings are produced from token streams by the prefix cache (requests 0-15
share a 2048-token prompt prefix), the cache is filled through those slots
(the shared prefix written once), decode runs over the pool's tables, and
sampled outputs match the oracle; the pool's page tags pass the integrity
check, and a released-then-reassigned page flags only its old holder."""
import numpy as np
import pytest

import oracle
import synth

from gpu_helpers import pf
from test_gpu_paged_decode import _run, _sampled_check, _setup

pytestmark = pytest.mark.gpu


def _streams(w, seed=23):
    """Seeded token ids: requests sharing the prefix share its first tokens."""
    rng = np.random.default_rng(seed)
    shared = rng.integers(0, 32000, w.shared_tokens)
    out = []
    for b in range(w.B):
        L = int(w.context_lens[b])
        if b < w.shared_requests:
            out.append(np.concatenate([shared, rng.integers(0, 32000, L - w.shared_tokens)]).astype(np.int32))
        else:
            out.append(rng.integers(0, 32000, L).astype(np.int32))
    return out


def test_shared_prefix_workload_from_token_streams_through_the_prefix_cache():
    import torch
    p = pf()
    w = synth.workload(synth.GQA_PREFIX)
    maxp = w.block_tables.shape[1]
    pool = p.PagePool(w.num_pages, w.P)
    rows = np.full((w.B, maxp), -1, np.int32)
    tags = np.zeros((w.B, maxp), np.uint32)
    cached = []
    for b, toks in enumerate(_streams(w)):
        rows[b], tags[b], c = pool.map_request(toks, maxp)
        cached.append(c)
    n_shared = w.shared_tokens // w.P
    assert cached[0] == 0 and cached[1:w.shared_requests] == [w.shared_tokens] * (w.shared_requests - 1)
    assert not any(cached[w.shared_requests:])
    assert np.array_equal(rows[1:w.shared_requests, :n_shared], np.broadcast_to(rows[0, :n_shared], (w.shared_requests - 1, n_shared)))
    used = np.concatenate([rows[b, :(int(w.context_lens[b]) + w.P - 1) // w.P] for b in range(w.B)])
    assert len(np.unique(used)) == w.num_pages and pool.num_free() == 0   # every page used, shared ones once
    assert all(pool.refcount(int(pg)) == w.shared_requests for pg in rows[0, :n_shared])

    # the workload now lives in the pool's pages: its slots and the oracle follow these tables
    w.block_tables = rows
    st = _setup(p, w)
    out, lse, status = _run(p, w, st)
    assert status == 0
    _sampled_check(p, w, st, out, lse, [(0, 0), (3, 17), (15, 63), (16, 5), (40, 30), (63, 63)])

    # page tags: all current; then request 40 finishes, its pages go to a new request, and only
    # request 40's (now stale) row fails the check
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int32)).cuda()
    status_dev = torch.empty(w.B, dtype=torch.int32, device="cuda")
    p.verify_page_tags(st.block_tables, d(tags), st.context_lens, w.P, d(pool.page_tags()), status_dev)
    assert not status_dev.cpu().numpy().any()
    n40 = (int(w.context_lens[40]) + w.P - 1) // w.P
    pool.release(rows[40], n40)
    pool.map_request(np.arange(int(w.context_lens[40]), dtype=np.int32) + 50000, maxp)
    p.verify_page_tags(st.block_tables, d(tags), st.context_lens, w.P, d(pool.page_tags()), status_dev)
    got = status_dev.cpu().numpy()
    ref = oracle.verify_page_tags(rows, tags, w.context_lens, w.P, pool.page_tags())
    assert np.array_equal(got, ref) and got[40] == oracle.REQ_TAG_MISMATCH and got.sum() == got[40]
