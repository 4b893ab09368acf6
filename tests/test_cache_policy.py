"""Device expert cache, host logic: slot assignment, hits, misses and the two
eviction policies, through the library's cache in planning mode (no upload
streams, so no CUDA call is made and these tests run without a GPU).

The expected behaviour is a small independent model of the policies written
here: plain LRU, and "keep the experts used by two rows or more" (the least
recently used single-row slot, else the most recently used slot); a request
never evicts one of its own experts."""

import numpy as np
import pytest

from mxfp4_mixture_experts_router_gb300 import binding as B
from mxfp4_mixture_experts_router_gb300 import build as build_mod

TINY = B.desc(256, 64, 32, 4)


@pytest.fixture(scope="module", autouse=True)
def built():
    build_mod.build()


class Model:
    """Reference model: slots, LRU order (most recent last), last rows per slot."""

    def __init__(self, n_slots, keep_multi_row):
        self.n = n_slots
        self.keep = keep_multi_row
        self.free = list(range(n_slots))
        self.key = {}           # slot -> (layer, expert)
        self.where = {}         # (layer, expert) -> slot
        self.rows = {}
        self.order = []         # least recent first
        self.hits = self.misses = self.evictions = 0

    def _touch(self, s):
        if s in self.order:
            self.order.remove(s)
        self.order.append(s)

    def request(self, layer, experts, rows):
        out = [None] * len(experts)
        mine = set()
        for i, e in enumerate(experts):
            k = (layer, e)
            if k in self.where:
                s = self.where[k]
                self._touch(s)
                self.rows[s] = rows[i]
                mine.add(s)
                out[i] = (s, 0)
                self.hits += 1
        for i, e in enumerate(experts):
            if out[i] is not None:
                continue
            if self.free:
                s = self.free.pop(0)
            else:
                cands = [s for s in self.order if s not in mine]
                if self.keep:
                    few = [s for s in cands if self.rows[s] < 2]
                    s = few[0] if few else cands[-1]
                else:
                    s = cands[0]
                del self.where[self.key[s]]
                self.evictions += 1
            self.key[s] = (layer, e)
            self.where[(layer, e)] = s
            self.rows[s] = rows[i]
            self._touch(s)
            mine.add(s)
            out[i] = (s, 1)
            self.misses += 1
        return out


def run_both(n_slots, policy, requests):
    h = B.moe_cache_create(TINY, None, B.moe_slab_bytes(TINY, B.MOE_FMT_MXFP4), n_slots, None, 0, policy)
    m = Model(n_slots, policy == B.MOE_CACHE_KEEP_MULTI_ROW)
    try:
        for layer, experts, rows in requests:
            slots, miss = B.moe_cache_request(h, layer, experts, rows, None, 0)
            want = m.request(layer, list(experts), list(rows))
            got_miss = [int(v) for v in miss]
            assert got_miss == [w[1] for w in want], (layer, experts)
            # slots: the same occupancy (which key lives where may differ only through
            # the free-slot order, which both take lowest-first here)
            assert [int(v) for v in slots] == [w[0] for w in want], (layer, experts)
            assert len(set(int(v) for v in slots)) == len(experts)
        st = B.moe_cache_stats(h)
        assert st["hits"] == m.hits and st["misses"] == m.misses and st["evictions"] == m.evictions
        assert st["bytes_uploaded"] == m.misses * B.moe_slab_bytes(TINY, B.MOE_FMT_MXFP4)
        return st
    finally:
        B.moe_cache_destroy(h)


def test_hits_misses_and_lru_order():
    reqs = [(0, [1, 2, 3], [1, 1, 1]),
            (0, [1, 4], [1, 1]),          # 1 hits; 4 evicts the LRU slot (expert 2)
            (0, [2, 3], [1, 1]),          # 2 misses again (was evicted), 3 hits
            (1, [1], [1])]                # same expert id, other layer: a different slab
    st = run_both(3, B.MOE_CACHE_LRU, reqs)
    assert st["hits"] == 2 and st["misses"] == 6


def test_keep_multi_row_protects_experts_shared_by_rows():
    # expert 7 was used by 3 rows; expert 8 by one row; under LRU the older (7) goes,
    # under the multi-row policy 8 goes first
    reqs = [(0, [7], [3]), (0, [8], [1]), (0, [9], [1])]
    lru = run_both(2, B.MOE_CACHE_LRU, reqs + [(0, [7], [1])])
    keep = run_both(2, B.MOE_CACHE_KEEP_MULTI_ROW, reqs + [(0, [7], [1])])
    assert lru["hits"] == 0 and keep["hits"] == 1


def test_a_request_never_evicts_its_own_experts():
    reqs = [(0, [0, 1, 2, 3], [2, 2, 2, 2]), (0, [3, 4, 5, 6], [1, 1, 1, 1])]
    for pol in (B.MOE_CACHE_LRU, B.MOE_CACHE_KEEP_MULTI_ROW):
        run_both(4, pol, reqs)


def test_random_traffic_matches_the_model():
    rng = np.random.default_rng(3)
    reqs = []
    for t in range(300):
        layer = int(rng.integers(0, 4))
        n = int(rng.integers(1, 7))
        experts = sorted(rng.choice(24, size=n, replace=False).tolist())
        rows = rng.integers(1, 4, size=n).tolist()
        reqs.append((layer, experts, rows))
    for pol in (B.MOE_CACHE_LRU, B.MOE_CACHE_KEEP_MULTI_ROW):
        run_both(10, pol, reqs)


def test_keep_multi_row_holds_a_working_set_larger_than_the_cache():
    # a cyclic scan over 3 layers x 4 multi-row experts with 8 slots: LRU never hits,
    # keeping the longer-held experts does
    reqs = [(t % 3, [0, 1, 2, 3], [2, 2, 2, 2]) for t in range(30)]
    lru = run_both(8, B.MOE_CACHE_LRU, reqs)
    keep = run_both(8, B.MOE_CACHE_KEEP_MULTI_ROW, reqs)
    assert lru["hits"] == 0 and keep["hits"] > 30


def test_more_experts_than_slots_is_refused():
    h = B.moe_cache_create(TINY, None, B.moe_slab_bytes(TINY, B.MOE_FMT_MXFP4), 2, None, 0, B.MOE_CACHE_LRU)
    try:
        with pytest.raises(B.MoeError):
            B.moe_cache_request(h, 0, [1, 2, 3], None, None, 0)
    finally:
        B.moe_cache_destroy(h)


def test_bad_arguments():
    slab = B.moe_slab_bytes(TINY, B.MOE_FMT_MXFP4)
    with pytest.raises(B.MoeError):
        B.moe_cache_create(TINY, None, slab - 1, 4, None, 0, B.MOE_CACHE_LRU)   # slot too small
    with pytest.raises(B.MoeError):
        B.moe_cache_create(TINY, None, slab, 4, None, 0, 7)                     # unknown policy
    with pytest.raises(B.MoeError):
        B.moe_cache_create(TINY, None, slab, 4, None, 2, B.MOE_CACHE_LRU)      # uploads need a pool
