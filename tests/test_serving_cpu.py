"""Host logic of the synthetic serving loop (bit_kv_cache_int2_gb300.serving),
with a fake device: page accounting, first-come-first-served admission under
the page budget, dense batch slots and retirement."""
import random

import pytest

from bit_kv_cache_int2_gb300.serving import PagePool, Request, Scheduler, pages_needed


class FakeBackend:
    """Mirrors the device state the real backend keeps per slot."""

    def __init__(self, pool_pages):
        self.slots = {}
        self.owner = {}  # page id -> rid
        self.pool_pages = pool_pages
        self.batches = []

    def admit(self, slot, req):
        for p in req.pages:
            assert 0 <= p < self.pool_pages
            assert p not in self.owner, "page handed out twice"
            self.owner[p] = req.rid
        self.slots[slot] = req.rid

    def move(self, src, dst):
        self.slots[dst] = self.slots.pop(src)

    def step(self, active):
        # slots 0..n-1 hold the active requests in order (rows beyond n are stale and unused)
        assert [self.slots[i] for i in range(len(active))] == [r.rid for r in active]
        self.batches.append(len(active))
        for r in active:
            assert r.done < r.gen

    def release_check(self, finished):
        for r in finished:
            for p in r.pages:
                if self.owner.get(p) == r.rid:
                    del self.owner[p]


def test_pages_needed():
    assert pages_needed(100, 10) == 0           # all inside sink + recent
    assert pages_needed(320, 1) == 1            # first history token
    assert pages_needed(320 + 64, 0) == 1
    assert pages_needed(320 + 65, 0) == 2


def test_page_pool_alloc_release():
    pool = PagePool(10)
    a = pool.alloc(4)
    b = pool.alloc(6)
    assert pool.alloc(1) is None and pool.available == 0
    assert sorted(a + b) == list(range(10))
    pool.release(a)
    assert pool.available == 4 and sorted(pool.alloc(4)) == sorted(a)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_scheduler_budget_slots_and_retirement(seed):
    rng = random.Random(seed)
    pool_pages, max_batch = 60, 6
    reqs = [Request(rid=i, prefix=rng.randint(0, 1500), gen=rng.randint(1, 40)) for i in range(25)]
    be = FakeBackend(pool_pages)
    sched = Scheduler(PagePool(pool_pages), max_batch, be, max_pages_per_req=64)

    class Checking:
        def admit(self, slot, req):
            # pages in use never exceed the pool
            in_use = sum(len(r.pages) for r in sched.active)
            assert in_use <= pool_pages
            be.admit(slot, req)

        def move(self, src, dst):
            be.move(src, dst)

        def step(self, active):
            be.step(active)

    sched.backend = Checking()
    for r in reqs:
        sched.submit(r)

    released = []
    orig_release = sched.pool.release

    def release(ids):
        for p in ids:
            be.owner.pop(p, None)
        released.extend(ids)
        orig_release(ids)

    sched.pool.release = release
    done = sched.run()
    assert sorted(r.rid for r in done) == list(range(25))
    assert all(r.done == r.gen for r in done)
    assert sched.pool.available == pool_pages          # every page came back
    assert max(be.batches) <= max_batch
    # first come, first served: admission order is submission order
    order = sorted(reqs, key=lambda r: (r.admitted_step, r.rid))
    assert [r.rid for r in order] == list(range(25))
    # a request runs exactly gen steps once admitted
    assert all(r.finished_step - r.admitted_step == r.gen for r in done)


def test_scheduler_rejects_a_request_that_never_fits():
    sched = Scheduler(PagePool(4), 2, FakeBackend(4), max_pages_per_req=64)
    with pytest.raises(ValueError):
        sched.submit(Request(rid=0, prefix=320 + 64 * 5, gen=1))
