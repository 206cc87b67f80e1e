"""Memory-budgeted continuous batching over one attention layer (synthetic).

The job-level claim of the pages ([News], "结果": up to 7.83x throughput at
batch 32 against BF16 KV; [Blog], serving paragraphs) comes from memory: at a
fixed KV budget INT2 history holds about 7x more requests than BF16 history, so
more of them decode together.  This module is the loop that turns a page budget
into a batch:

* a request arrives with a cached prefix (a full prefix hit, imported as stored
  KV) and generates ``gen`` tokens; it is admitted, first come first served,
  once the pool holds every history page it will ever need
  (ceil(max(prefix + gen - 320, 0) / 64));
* active requests sit in batch slots 0..n-1; each iteration runs one decode
  step for all of them (append the new token, demote the oldest recent one,
  attend) through the C ABI: ``oscar_decode_step`` for INT2, or
  ``oscar_append_bf16_history`` + ``oscar_decode_bf16_history`` for the BF16
  baseline;
* a finished request returns its pages; the last active request moves into
  its slot so the batch stays dense.

Host bookkeeping only: every step of the attention runs in the library's
kernels.  One layer, synthetic tokens: it measures the memory-bound batching
effect, not a model.
"""
from __future__ import annotations

import dataclasses
import time

from . import oscar

HISTORY_FREE = 320  # sink 64 + recent 256 tokens live outside the history pages


def pages_needed(prefix: int, gen: int, page: int = 64) -> int:
    """History pages a request needs by the end of its generation."""
    hist = max(prefix + gen - HISTORY_FREE, 0)
    return (hist + page - 1) // page


class PagePool:
    """Free list of the pool's page ids."""

    def __init__(self, num_pages: int):
        self.num_pages = num_pages
        self._free = list(range(num_pages - 1, -1, -1))

    @property
    def available(self) -> int:
        return len(self._free)

    def alloc(self, n: int):
        if n > len(self._free):
            return None
        return [self._free.pop() for _ in range(n)]

    def release(self, ids):
        self._free.extend(reversed(ids))


@dataclasses.dataclass
class Request:
    rid: int
    prefix: int
    gen: int
    done: int = 0          # tokens generated so far
    pages: list = None
    admitted_step: int = -1
    finished_step: int = -1


class Scheduler:
    """Admission, slots and retirement, independent of the device (testable on CPU).

    The backend receives: ``admit(slot, req)`` (pages in req.pages),
    ``step(slots)`` (active requests in slot order) and ``move(src, dst)``
    (copy slot src's device state into slot dst)."""

    def __init__(self, pool: PagePool, max_batch: int, backend, max_pages_per_req: int):
        self.pool = pool
        self.max_batch = max_batch
        self.backend = backend
        self.max_pages = max_pages_per_req
        self.active = []   # slot i holds active[i]
        self.waiting = []
        self.finished = []
        self.steps = 0

    def submit(self, req: Request):
        if pages_needed(req.prefix, req.gen) > min(self.max_pages, self.pool.num_pages):
            raise ValueError(f"request {req.rid} can never fit the pool")
        self.waiting.append(req)

    def _admit(self):
        while self.waiting and len(self.active) < self.max_batch:
            req = self.waiting[0]
            ids = self.pool.alloc(pages_needed(req.prefix, req.gen))
            if ids is None:
                break  # first come, first served: later requests wait too
            self.waiting.pop(0)
            req.pages = ids
            req.admitted_step = self.steps
            slot = len(self.active)
            self.active.append(req)
            self.backend.admit(slot, req)

    def _retire(self):
        slot = 0
        while slot < len(self.active):
            req = self.active[slot]
            if req.done < req.gen:
                slot += 1
                continue
            req.finished_step = self.steps
            self.pool.release(req.pages)
            self.finished.append(req)
            last = len(self.active) - 1
            if slot != last:
                self.backend.move(last, slot)
                self.active[slot] = self.active[last]
            self.active.pop()

    def run(self, max_steps: int = 1 << 30):
        self._admit()
        while (self.active or self.waiting) and self.steps < max_steps:
            if not self.active:
                raise RuntimeError("nothing admitted: the pool is too small for the next request")
            self.backend.step(self.active)
            for req in self.active:
                req.done += 1
            self.steps += 1
            self._retire()
            self._admit()
        return self.finished


class DeviceBackend:
    """One layer's cache on the GPU, driven through the C ABI.

    draw(req) -> (K, V, Q): the request's synthetic stream, K and V bf16
    [Hkv][prefix + gen][128] and Q bf16 [gen][Hq][128] device tensors.  At
    admission the prefix is imported and the request's future tokens are
    copied into its batch slot's buffers; a step then gathers every active
    slot's next token with one indexed read per operand and runs one
    pre-marshalled library call.  fmt is "int2" or "bf16"."""

    def __init__(self, fmt, ctx, cfg, cache, draw, on_step=None, time_steps=False, max_gen=64):
        import torch

        self.fmt, self.ctx, self.cfg, self.cache = fmt, ctx, cfg, cache
        self.draw, self.on_step = draw, on_step
        B, Hq, Hkv = cfg.max_batch, cfg.num_q_heads, cfg.num_kv_heads
        dev = cache["seq_lens"].device
        self.dev = dev
        self.out = torch.empty(B, Hq, 128, dtype=torch.bfloat16, device=dev)
        self.scratch = oscar.alloc_scratch(cfg, dev)
        self.gen_cap = 0
        self._grow(max_gen)
        self.pos = torch.zeros(B, dtype=torch.long, device=dev)  # next token of each slot
        self.slots = torch.arange(B, device=dev)
        self.call = oscar.bind_step_any_batch(ctx, 0, cache, self.out, None, self.scratch,
                                              bf16_history=(fmt == "bf16"))
        self.step_events = [] if time_steps else None
        self.import_events = [] if time_steps else None

    def _grow(self, gen):
        """Slot buffers for up to `gen` future tokens per request, keeping the
        tokens already held."""
        import torch

        B, Hq, Hkv = self.cfg.max_batch, self.cfg.num_q_heads, self.cfg.num_kv_heads
        bufs = (torch.zeros(B, gen, Hkv, 128, dtype=torch.bfloat16, device=self.dev),
                torch.zeros(B, gen, Hkv, 128, dtype=torch.bfloat16, device=self.dev),
                torch.zeros(B, gen, Hq, 128, dtype=torch.bfloat16, device=self.dev))
        if self.gen_cap:
            for new, old in zip(bufs, (self.kbuf, self.vbuf, self.qbuf)):
                new[:, :self.gen_cap] = old
        self.kbuf, self.vbuf, self.qbuf = bufs
        self.gen_cap = gen

    def _view(self, slot):
        v = dict(self.cache)
        for key in ("page_table", "sink_k", "sink_v", "ring_k", "ring_v", "seq_lens", "hist_lens"):
            v[key] = self.cache[key][slot:slot + 1]
        return v

    def admit(self, slot, req):
        import torch

        if req.gen > self.gen_cap:
            self._grow(req.gen)
        K, V, Q = self.draw(req)
        P, n = req.prefix, req.gen
        self.kbuf[slot, :n] = K[:, P:P + n].permute(1, 0, 2)
        self.vbuf[slot, :n] = V[:, P:P + n].permute(1, 0, 2)
        self.qbuf[slot, :n] = Q[:n]
        self.pos[slot] = 0
        row = self.cache["page_table"][slot]
        row.fill_(-1)
        if req.pages:
            # pinned and non-blocking: a pageable copy would wait for all queued GPU work
            ids = torch.tensor(req.pages, dtype=torch.int32)
            if row.is_cuda:
                ids = ids.pin_memory()
            row[:len(req.pages)].copy_(ids, non_blocking=row.is_cuda)
        self.cache["seq_lens"][slot] = 0
        self.cache["hist_lens"][slot] = 0
        if P:
            view = self._view(slot)
            Kp = K[:, :P].unsqueeze(0).contiguous()
            Vp = V[:, :P].unsqueeze(0).contiguous()
            if self.import_events is not None:
                ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                ev[0].record()
            if self.fmt == "int2":
                oscar.oscar_import_tokens(self.ctx, 0, view, Kp, Vp, 1, P)
            else:
                oscar.oscar_import_bf16_history(self.ctx, view, Kp, Vp, 1, P)
            if self.import_events is not None:
                ev[1].record()
                self.import_events.append(ev)

    def move(self, src, dst):
        for key in ("page_table", "sink_k", "sink_v", "ring_k", "ring_v", "seq_lens", "hist_lens"):
            self.cache[key][dst].copy_(self.cache[key][src])
        for buf in (self.kbuf, self.vbuf, self.qbuf, self.pos):
            buf[dst].copy_(buf[src])

    def step(self, active):
        import torch

        n = len(active)
        sl, ps = self.slots[:n], self.pos[:n]
        k = self.kbuf[sl, ps]
        v = self.vbuf[sl, ps]
        q = self.qbuf[sl, ps]
        if self.step_events is not None:
            ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            ev[0].record()
        self.call(k.data_ptr(), v.data_ptr(), q.data_ptr(), n)
        if self.step_events is not None:
            ev[1].record()
            self.step_events.append(ev)
        self.pos[:n] += 1
        if self.on_step is not None:
            self.on_step(active, q, self.out[:n])


def step_seconds(backend):
    """Device time of the decode steps (append + attention), summed, when the
    backend was made with time_steps=True."""
    return sum(a.elapsed_time(b) for a, b in backend.step_events) * 1e-3


def import_seconds(backend):
    """Device time of the prefix imports, summed (time_steps=True)."""
    return sum(a.elapsed_time(b) for a, b in backend.import_events) * 1e-3


def run_job(backend, pool_pages, max_batch, max_pages_per_req, requests):
    """Runs the requests to completion; returns (finished, steps, seconds)."""
    import torch

    sched = Scheduler(PagePool(pool_pages), max_batch, backend, max_pages_per_req)
    for r in requests:
        sched.submit(r)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    done = sched.run()
    torch.cuda.synchronize()
    return done, sched.steps, time.perf_counter() - t0
