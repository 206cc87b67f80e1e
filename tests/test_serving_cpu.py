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


def test_device_backend_feeds_each_slot_its_own_next_token(monkeypatch):
    """DeviceBackend's slot buffers on CPU tensors, with the library calls
    replaced by recorders: every step's k, v and q rows are the active
    requests' own tokens at position prefix + done, through admissions, slot
    moves and retirements."""
    import ctypes
    import types

    import numpy as np
    import torch

    from bit_kv_cache_int2_gb300 import serving

    Hq, Hkv, B = 4, 2, 3
    cfg = types.SimpleNamespace(max_batch=B, num_q_heads=Hq, num_kv_heads=Hkv)
    cache = {"page_table": torch.full((B, 8), -1, dtype=torch.int32),
             "sink_k": torch.zeros(B, 1), "sink_v": torch.zeros(B, 1), "ring_k": torch.zeros(B, 1),
             "ring_v": torch.zeros(B, 1), "seq_lens": torch.zeros(B, dtype=torch.int32),
             "hist_lens": torch.zeros(B, dtype=torch.int32)}
    seen = []

    def bind(ctx, layer, cache_, out, lse, scratch, bf16_history=False):
        def call(k_ptr, v_ptr, q_ptr, n):
            grab = lambda p, heads: np.frombuffer(ctypes.string_at(p, n * heads * 128 * 2), dtype=np.uint16
                                                  ).reshape(n, heads, 128).copy()
            seen.append((grab(k_ptr, Hkv), grab(v_ptr, Hkv), grab(q_ptr, Hq)))
        return call

    fake = types.SimpleNamespace(alloc_scratch=lambda c, d: torch.zeros(1), bind_step_any_batch=bind,
                                 oscar_import_tokens=lambda *a: None, oscar_import_bf16_history=lambda *a: None)
    monkeypatch.setattr(serving, "oscar", fake)

    def tok(rid, pos, which, h):
        # a distinct value per (request, position, operand, head), exact in bf16:
        # a power of two times a 7-bit mantissa
        i = ((rid * 16 + pos) * 3 + which) * 4 + h
        return 2.0 ** (i // 128 - 4) * (1 + (i % 128) / 128)

    def draw(req):
        n = req.prefix + req.gen
        K = torch.tensor([[[tok(req.rid, p, 0, h)] * 128 for p in range(n)] for h in range(Hkv)]).to(torch.bfloat16)
        V = torch.tensor([[[tok(req.rid, p, 1, h)] * 128 for p in range(n)] for h in range(Hkv)]).to(torch.bfloat16)
        Q = torch.tensor([[[tok(req.rid, req.prefix + t, 2, h)] * 128 for h in range(Hq)]
                          for t in range(req.gen)]).to(torch.bfloat16)
        return K, V, Q

    checks = []

    def on_step(active, q, out):
        k, v, qq = seen[-1]
        as_f = lambda a: (a.astype(np.uint32) << 16).view(np.float32)
        for i, r in enumerate(active):
            p = r.prefix + r.done
            for h in range(Hkv):
                assert as_f(k[i, h, 0]) == np.float32(tok(r.rid, p, 0, h)), (r.rid, p, h)
                assert as_f(v[i, h, 0]) == np.float32(tok(r.rid, p, 1, h)), (r.rid, p, h)
            for h in range(Hq):
                assert as_f(qq[i, h, 0]) == np.float32(tok(r.rid, p, 2, h)), (r.rid, p, h)
        checks.append(len(active))

    backend = serving.DeviceBackend("int2", None, cfg, cache, draw, on_step=on_step, max_gen=4)
    reqs = [Request(rid=0, prefix=3, gen=2), Request(rid=1, prefix=0, gen=5), Request(rid=2, prefix=1, gen=3),
            Request(rid=3, prefix=2, gen=6), Request(rid=4, prefix=0, gen=1)]
    sched = Scheduler(PagePool(40), B, backend, max_pages_per_req=8)
    for r in reqs:
        sched.submit(r)
    done = sched.run()
    assert sorted(r.rid for r in done) == [0, 1, 2, 3, 4]
    assert sum(checks) == sum(r.gen for r in reqs) and max(checks) == B
    assert backend.gen_cap == 6  # grew for the 6-token request
