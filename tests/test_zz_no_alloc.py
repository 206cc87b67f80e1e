"""oscar_decode_noalloc: the decode entry point for callers that must not
allocate device memory on the decode path (engines that reserve all memory for
their KV pools up front, code where an allocation would stall other work on
the device, C callers without an allocator).  Instead of a caller-provided
scratch buffer it uses one buffer the library keeps in device memory.

Its results must equal oscar_decode's bit for bit on the same cache and
queries, on two calls in a row (the second call starts from the first call's
leftovers in the shared buffer): the same kernels run with the same work list,
so any difference would be leftover state of the shared buffer leaking in.
This file is collected last on purpose."""
import pytest
import torch

from bit_kv_cache_int2_gb300 import build as B
from bit_kv_cache_int2_gb300 import oscar

pytestmark = pytest.mark.gpu

import gpu_scenario as GS  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def built():
    B.build()
    oscar.lib()


def test_decode_noalloc_matches_decode_on_two_calls():
    sc = GS.build("noalloc", [70000, 320, 5000, 1], Hq=8, Hkv=2, g=128, calib_n=512)
    try:
        q = GS.queries(sc, seed=11)
        ref, rlse = GS.decode(sc, q)  # the existing entry point, caller-provided scratch
        assert oscar.oscar_get_error(sc.ctx) == 0
        assert bool(torch.isfinite(ref.float()).all())
        for _ in range(2):
            out = torch.full_like(q, float("nan"))
            lse = torch.full((q.shape[0], q.shape[1]), float("nan"), dtype=torch.float32, device=q.device)
            oscar.oscar_decode_noalloc(sc.ctx, 0, sc.cache, q, out, lse, sc.B)
            torch.cuda.synchronize()
            assert oscar.oscar_get_error(sc.ctx) == 0
            assert torch.equal(out, ref)
            assert torch.equal(lse, rlse)
    finally:
        sc.close()


def test_decode_noalloc_rejects_requests_beyond_its_buffer():
    # 4096 requests x 64 query heads need far more working memory than the
    # built-in buffer holds: refused before anything is launched.
    cfg = oscar.make_config(1, 64, 8, 128, max_batch=4096, max_pages_per_req=1, num_pages=1)
    assert oscar.oscar_layout(cfg).decode_scratch_bytes > oscar.NOALLOC_SCRATCH_BYTES
    ctx = oscar.oscar_create(cfg)
    try:
        q = torch.zeros(4096, 64, 128, dtype=torch.bfloat16, device="cuda")
        with pytest.raises(oscar.OscarError) as e:
            oscar.oscar_decode_noalloc(ctx, 0, {}, q, torch.empty_like(q), None, 4096)
        assert e.value.status == oscar.ERR_TOO_LARGE
    finally:
        oscar.oscar_destroy(ctx)
