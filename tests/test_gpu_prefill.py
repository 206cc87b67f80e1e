"""GPU parity of oscar_prefill (chunked prefill over the cache) against the
oracle's chunk_prefill_attention, through the C ABI, on the GPU's own cache
contents: every chunk token and query head at small sizes (several row tiles,
ragged chunks, ragged last pages, empty and partial windows), sampled tokens at
a full 100K-token context."""
import numpy as np
import pytest
import torch

import oracle as O
from bit_kv_cache_int2_gb300 import build as B
from bit_kv_cache_int2_gb300 import oscar, synth

pytestmark = pytest.mark.gpu

import gpu_scenario as GS  # noqa: E402

REL_TOL = 1e-2  # max|gpu - oracle| / max|oracle| per (request, kv head) block
LSE_TOL = 1e-2  # absolute, natural-log units


@pytest.fixture(scope="module", autouse=True)
def built():
    B.build()
    oscar.lib()


def _rel(a, b):
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-30))


def chunk_inputs(sc, T, seed):
    """q [B][T][Hq][128] drawn from each head's query law; k, v [B][T][Hkv][128]
    the next T tokens of each request's own sequence."""
    G = sc.Hq // sc.Hkv
    qs, ks, vs = [], [], []
    for b, L in enumerate(sc.lengths):
        rows = [synth.draw_queries(sc.stats[h], T * G, synth.stream_seed(seed, "PQ", b, h), "cuda").view(T, G, 128)
                for h in range(sc.Hkv)]
        qs.append(torch.cat(rows, dim=1))
        ks.append(sc.K[b][:, L:L + T].permute(1, 0, 2))
        vs.append(sc.V[b][:, L:L + T].permute(1, 0, 2))
    return (torch.stack(qs).contiguous(), torch.stack(ks).contiguous(), torch.stack(vs).contiguous())


def run_prefill(sc, q, k, v, with_lse=True, impl=oscar.PREFILL_TCGEN05):
    Bn, T = q.shape[0], q.shape[1]
    oscar.oscar_set_option(sc.ctx, oscar.OPT_PREFILL_IMPL, impl)
    out = torch.full_like(q, float("nan"))
    lse = torch.full((Bn, T, sc.Hq), float("nan"), dtype=torch.float32, device="cuda") if with_lse else None
    scratch = oscar.alloc_scratch(sc.cfg, prefill=True)
    oscar.oscar_prefill(sc.ctx, 0, sc.cache, q, k, v, T, out, lse, scratch, Bn)
    torch.cuda.synchronize()
    return out, lse


def oracle_prefill(sc, hc, q, k, v, b, h, tokens=None):
    G = sc.Hq // sc.Hkv
    qn = q[b, :, h * G:(h + 1) * G].float().cpu().numpy()
    kc = k[b, :, h].float().cpu().numpy()
    vc = v[b, :, h].float().cpu().numpy()
    wk, wv = hc.window(b, h)
    f = hc.history_int2(b, h, sc.g)
    if f is None:
        hk = hv = np.zeros((0, 128))
    else:
        ck, cv = sc.cb("k", h), sc.cb("v", h)  # Lloyd-Max levels, or None for the uniform ones
        hk = (O.dequantize(f["k_codes"], f["k_s"], f["k_z"], sc.g) if ck is None
              else O.dequantize_codebook(f["k_codes"], f["k_s"], f["k_z"], sc.g, *ck))
        hv = (O.dequantize(f["v_codes"], f["v_s"], f["v_z"], sc.g) if cv is None
              else O.dequantize_codebook(f["v_codes"], f["v_s"], f["v_z"], sc.g, *cv))
    return O.chunk_prefill_attention(qn, kc, vc, wk, wv, hk, hv, O.rotation(sc.U_K[h], sc.mode),
                                     O.rotation(sc.U_V[h], sc.mode), tokens=tokens)


def check_all(sc, q, k, v, out, lse):
    hc = GS.HostCache(sc)
    G = sc.Hq // sc.Hkv
    worst = 0.0
    for b in range(sc.B):
        for h in range(sc.Hkv):
            ref, rlse = oracle_prefill(sc, hc, q, k, v, b, h)
            got = out[b, :, h * G:(h + 1) * G].float().cpu().numpy()
            err = _rel(got, ref)
            worst = max(worst, err)
            assert err <= REL_TOL, (b, h, err)
            if lse is not None:
                dl = np.abs(lse[b, :, h * G:(h + 1) * G].cpu().numpy() - rlse).max()
                assert dl <= LSE_TOL, (b, h, dl)
    print(f"worst rel err {worst:.2e}")


CASES = [
    # lengths, T, Hq, Hkv, g, mode
    ([3000], 64, 4, 1, 128, oscar.ROT_OSCAR),         # 42 history pages, last one ragged; 2 row tiles
    ([1000, 5000], 17, 8, 2, 32, oscar.ROT_OSCAR),    # ragged chunk, g32, two requests
    ([2000], 64, 16, 2, 64, oscar.ROT_OSCAR),         # GQA 8: 512 rows, 4 row tiles
    ([200], 1, 4, 1, 128, oscar.ROT_OSCAR),           # one token, no history, partial ring
    ([40, 0, 333], 5, 4, 1, 128, oscar.ROT_HADAMARD),  # partial sink, empty request, 13 history tokens
    ([700], 33, 4, 1, 128, oscar.ROT_NONE),
]


IMPLS = [oscar.PREFILL_TCGEN05, oscar.PREFILL_MMA_SYNC]


@pytest.mark.parametrize("impl", IMPLS, ids=["tcgen05", "mma_sync"])
@pytest.mark.parametrize("lengths,T,Hq,Hkv,g,mode", CASES)
def test_prefill_matches_oracle(lengths, T, Hq, Hkv, g, mode, impl):
    sc = GS.build(f"pf{len(lengths)}_{T}", lengths, Hq=Hq, Hkv=Hkv, g=g, mode=mode, extra_tokens=T, calib_n=512)
    try:
        q, k, v = chunk_inputs(sc, T, seed=31)
        seq0 = sc.cache["seq_lens"].clone()
        hist0 = sc.cache["hist_lens"].clone()
        out, lse = run_prefill(sc, q, k, v, impl=impl)
        assert oscar.oscar_get_error(sc.ctx) == 0
        # the chunk is not stored
        assert torch.equal(sc.cache["seq_lens"], seq0) and torch.equal(sc.cache["hist_lens"], hist0)
        check_all(sc, q, k, v, out, lse)
    finally:
        sc.close()


@pytest.mark.parametrize("impl", IMPLS, ids=["tcgen05", "mma_sync"])
def test_prefill_without_lse_and_repeatable(impl):
    sc = GS.build("pf_nolse", [1500], Hq=4, Hkv=1, g=128, extra_tokens=20, calib_n=512)
    try:
        q, k, v = chunk_inputs(sc, 20, seed=32)
        out_a, lse_a = run_prefill(sc, q, k, v, impl=impl)
        out_b, _ = run_prefill(sc, q, k, v, with_lse=False, impl=impl)
        assert torch.equal(out_a, out_b)  # same work split, same arithmetic
        check_all(sc, q, k, v, out_b, None)
    finally:
        sc.close()


def test_prefill_rejects_bad_chunk_length():
    sc = GS.build("pf_bad", [100], Hq=4, Hkv=1, g=128, extra_tokens=1, calib_n=256)
    try:
        q, k, v = chunk_inputs(sc, 1, seed=33)
        scratch = oscar.alloc_scratch(sc.cfg, prefill=True)
        out = torch.empty_like(q)
        for T in (0, 65):
            with pytest.raises(oscar.OscarError):
                oscar.oscar_prefill(sc.ctx, 0, sc.cache, q, k, v, T, out, None, scratch, 1)
    finally:
        sc.close()


@pytest.mark.parametrize("impl", IMPLS, ids=["tcgen05", "mma_sync"])
def test_prefill_qwen3_8b_100k_sampled(impl):
    """32 q / 8 kv heads, g128, 100,000 cached tokens, a 64-token chunk: tokens
    0, 31 and 63 of every head checked."""
    sc = GS.build("pf100k", [100000], Hq=32, Hkv=8, g=128, extra_tokens=64, calib_n=1024)
    try:
        q, k, v = chunk_inputs(sc, 64, seed=34)
        out, lse = run_prefill(sc, q, k, v, impl=impl)
        assert oscar.oscar_get_error(sc.ctx) == 0
        hc = GS.HostCache(sc)
        G = 4
        toks = [0, 31, 63]
        for h in range(8):
            ref, rlse = oracle_prefill(sc, hc, q, k, v, 0, h, tokens=toks)
            got = out[0, toks, h * G:(h + 1) * G].float().cpu().numpy()
            assert _rel(got, ref) <= REL_TOL, (h, _rel(got, ref))
            assert np.abs(lse[0, toks, h * G:(h + 1) * G].cpu().numpy() - rlse).max() <= LSE_TOL, h
    finally:
        sc.close()


@pytest.mark.parametrize("impl", IMPLS, ids=["tcgen05", "mma_sync"])
def test_prefill_missing_history_page_reports_and_skips_it(impl):
    """A history page whose table entry is -1: the call records OSCAR_ERR_NO_PAGE
    and the page's 64 tokens take no part; everything else is still exact."""
    T = 16
    sc = GS.build("pf_hole", [2000], Hq=4, Hkv=1, g=64, extra_tokens=T, calib_n=512)
    try:
        q, k, v = chunk_inputs(sc, T, seed=35)
        hc = GS.HostCache(sc)  # before the hole
        hole = 7
        sc.cache["page_table"][0, hole] = -1
        out, lse = run_prefill(sc, q, k, v, impl=impl)
        assert oscar.oscar_get_error(sc.ctx) == oscar.ERR_NO_PAGE
        f = hc.history_int2(0, 0, sc.g)
        keep = np.ones(len(f["k_codes"]), dtype=bool)
        keep[hole * 64:(hole + 1) * 64] = False
        hk = O.dequantize(f["k_codes"][keep], f["k_s"][keep], f["k_z"][keep], sc.g)
        hv = O.dequantize(f["v_codes"][keep], f["v_s"][keep], f["v_z"][keep], sc.g)
        wk, wv = hc.window(0, 0)
        ref, rlse = O.chunk_prefill_attention(q[0].float().cpu().numpy(), k[0, :, 0].float().cpu().numpy(),
                                              v[0, :, 0].float().cpu().numpy(), wk, wv, hk, hv,
                                              O.rotation(sc.U_K[0], sc.mode), O.rotation(sc.U_V[0], sc.mode))
        got = out[0].float().cpu().numpy()
        assert _rel(got, ref) <= REL_TOL, _rel(got, ref)
        assert np.abs(lse[0].cpu().numpy() - rlse).max() <= LSE_TOL
    finally:
        sc.close()
