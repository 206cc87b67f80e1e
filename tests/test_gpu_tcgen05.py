"""The tensor-memory decode kernel (OSCAR_DECODE_TCGEN05) against the oracle:
ragged batches whose even split over the SMs cuts requests' pages and window
chunks at arbitrary places, group sizes with one to four groups per head,
GQA 1 to 8, a decode step bit for bit equal to append then decode, and
missing pages reported without a fault."""
import numpy as np
import pytest
import torch

from bit_kv_cache_int2_gb300 import build as B
from bit_kv_cache_int2_gb300 import oscar

pytestmark = pytest.mark.gpu

import gpu_scenario as GS  # noqa: E402

REL_TOL = 1e-2  # max|out - ref| / max|ref| against the fp64 oracle on the stored codes
LSE_TOL = 1e-2
TC = oscar.DECODE_TCGEN05


@pytest.fixture(scope="module", autouse=True)
def built():
    B.build()
    oscar.lib()


def _rel(got, ref):
    return float(np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-30))


def _check_all(sc, q, out, lse):
    hc = GS.HostCache(sc)
    qn = q.float().cpu().numpy()
    for b, L in enumerate(sc.lengths):
        got = out[b].float().cpu().numpy()
        if L == 0:
            assert np.all(got == 0) and np.all(np.isneginf(lse[b].cpu().numpy()))
            continue
        ref, rlse = GS.oracle_decode(sc, hc, qn, b)
        assert _rel(got, ref) <= REL_TOL, (b, L, _rel(got, ref))
        assert np.abs(lse[b].cpu().numpy() - rlse).max() <= LSE_TOL, (b, L)


def test_small_single_request():
    sc = GS.build("tc1", [1000], Hq=4, Hkv=1, g=128, calib_n=512)
    try:
        q = GS.queries(sc, seed=1)
        out, lse = GS.decode(sc, q, TC)
        assert oscar.oscar_get_error(sc.ctx) == 0
        _check_all(sc, q, out, lse)
    finally:
        sc.close()


@pytest.mark.parametrize("G,g", [(4, 128), (4, 32), (8, 128), (8, 32), (2, 64), (1, 32)])
def test_ragged_batch_split_over_sms(G, g):
    # totals of a few thousand page units spread over the SMs: every CTA's
    # range starts and ends inside some request's pages or window chunks
    lengths = [9000, 320, 14000, 6234, 0, 700, 12500, 64 * 50 + 320 + 3, 1, 385]
    sc = GS.build(f"tcr{G}{g}", lengths, Hq=2 * G, Hkv=2, g=g, interleave=True, calib_n=512)
    try:
        q = GS.queries(sc, seed=2)
        out, lse = GS.decode(sc, q, TC)
        assert oscar.oscar_get_error(sc.ctx) == 0
        _check_all(sc, q, out, lse)
    finally:
        sc.close()


def test_long_request_many_tiles_per_cta():
    # one request of 200K tokens, 4 kv heads: ~80 page pairs per CTA, so the
    # lazy rescale of the running maximum and the buffer rings wrap many times
    sc = GS.build("tclong", [200_000], Hq=16, Hkv=4, g=128, calib_n=512)
    try:
        q = GS.queries(sc, seed=3)
        out, lse = GS.decode(sc, q, TC)
        assert oscar.oscar_get_error(sc.ctx) == 0
        _check_all(sc, q, out, lse)
    finally:
        sc.close()


def test_matches_the_mma_sync_kernel():
    sc = GS.build("tcvs", [5000, 40000, 321], Hq=8, Hkv=2, g=64, calib_n=512)
    try:
        q = GS.queries(sc, seed=4)
        ref, rlse = GS.decode(sc, q, oscar.DECODE_TENSOR)
        out, lse = GS.decode(sc, q, TC)
        assert oscar.oscar_get_error(sc.ctx) == 0
        r = ref.float().cpu().numpy()
        o = out.float().cpu().numpy()
        assert np.abs(o - r).max() <= REL_TOL * np.abs(r).max()
        np.testing.assert_allclose(lse.cpu().numpy(), rlse.cpu().numpy(), atol=LSE_TOL)
    finally:
        sc.close()


def test_decode_step_equals_append_then_decode():
    lengths = [300, 64, 1500, 20000]
    scs = [GS.build("tcstep", lengths, Hq=8, Hkv=2, g=128, extra_tokens=40, calib_n=512) for _ in range(2)]
    try:
        for s_ in scs:
            oscar.oscar_set_option(s_.ctx, oscar.OPT_DECODE_IMPL, TC)
        scratch = [oscar.alloc_scratch(s_.cfg) for s_ in scs]
        for t in range(40):
            k = torch.stack([scs[0].K[i][:, lengths[i] + t] for i in range(4)]).contiguous()
            v = torch.stack([scs[0].V[i][:, lengths[i] + t] for i in range(4)]).contiguous()
            q = GS.queries(scs[0], seed=300 + t)
            outs = []
            for j, s_ in enumerate(scs):
                out = torch.empty_like(q)
                lse = torch.empty(q.shape[0], q.shape[1], dtype=torch.float32, device=q.device)
                if j == 0:
                    oscar.oscar_decode_step(s_.ctx, 0, s_.cache, k, v, q, out, lse, scratch[j], 4)
                else:
                    oscar.oscar_append(s_.ctx, 0, s_.cache, k, v, 4)
                    oscar.oscar_decode(s_.ctx, 0, s_.cache, q, out, lse, scratch[j], 4)
                outs.append((out, lse))
            torch.cuda.synchronize()
            assert torch.equal(outs[0][0], outs[1][0]), t
            assert torch.equal(outs[0][1], outs[1][1]), t
        for s_ in scs:
            assert oscar.oscar_get_error(s_.ctx) == 0
        _check_all(scs[0], q, outs[0][0], outs[0][1])
    finally:
        for s_ in scs:
            s_.close()


def test_missing_page_is_reported_not_faulted():
    sc = GS.build("tcerr", [5000], Hq=4, Hkv=1, calib_n=512)
    try:
        pt = sc.cache["page_table"]
        saved = pt.clone()
        q = GS.queries(sc, seed=7)
        pt[0, 3] = -1
        GS.decode(sc, q, TC)
        assert oscar.oscar_get_error(sc.ctx) == oscar.ERR_NO_PAGE
        pt[0, 3] = 10 ** 6
        GS.decode(sc, q, TC)
        assert oscar.oscar_get_error(sc.ctx) == oscar.ERR_RANGE
        pt.copy_(saved)
        out, lse = GS.decode(sc, q, TC)
        assert oscar.oscar_get_error(sc.ctx) == 0
        _check_all(sc, q, out, lse)
    finally:
        sc.close()
