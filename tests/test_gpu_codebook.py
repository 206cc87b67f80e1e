"""GPU parity of the Lloyd-Max codebook path through the C ABI: the
quantiser's codes and scales bit for bit, the codebook fit, the decode over a
cache written with a codebook (import, append with demotion, the fused step),
the chunked prefill over it, the clip errors with a codebook, and the
host-side rules (uniform levels keep the default kernels, bad pairs are
rejected)."""
import numpy as np
import pytest
import torch

import oracle as O
from bit_kv_cache_int2_gb300 import build as B
from bit_kv_cache_int2_gb300 import oscar, synth

pytestmark = pytest.mark.gpu

import gpu_scenario as GS  # noqa: E402

REL_TOL = 1e-2  # max|gpu - oracle| / max|oracle| on decode outputs
LSE_TOL = 1e-2
FIT_TOL = 1e-4  # (a, b): the GPU rotates in fp32, the oracle in fp64 then rounds

CODEBOOKS = [(0.4528, 1.5104), (0.2, 0.9), (0.0, 2.1), (0.7, 1.3)]


@pytest.fixture(scope="module", autouse=True)
def built():
    B.build()
    oscar.lib()


def _rel(a, b):
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-30))


def _hook_inputs(n, seed):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((n, 128)) * rng.uniform(0.01, 30, (n, 1))).astype(np.float32)
    x[0] = 5.0  # constant groups -> s = 0
    x[1] = np.tile(np.array([0.0, 1.0, 2.0, 3.0, 0.5, 1.5, 2.5, 3.0], np.float32), 16)  # exact ties (uniform)
    x[2] = np.linspace(-3e5, 3e5, 128, dtype=np.float32)  # saturated scale
    x[3] = np.linspace(-1e-7, 1e-7, 128, dtype=np.float32)
    return x


def _run_hook(x, g, clip, which, ab):
    n = x.shape[0]
    ng = 128 // g
    xd = torch.from_numpy(x).cuda()
    codes = torch.zeros(n * 32, dtype=torch.uint8, device="cuda")
    sz = torch.zeros(n * ng * 2, dtype=torch.float16, device="cuda")
    if ab is None:
        oscar.oscar_quantize_rotated_f32(xd, g, clip, which, codes, sz)
    else:
        oscar.oscar_quantize_codebook_f32(xd, g, clip, ab[0], ab[1], which, codes, sz)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), sz.cpu().numpy().reshape(n, ng, 2)


@pytest.mark.parametrize("g", [32, 128])
@pytest.mark.parametrize("clip", [1.0, 0.9])
@pytest.mark.parametrize("which", [0, 1])
@pytest.mark.parametrize("ab", CODEBOOKS + [O.UNIFORM_CODEBOOK])
def test_codebook_quantiser_bit_exact(g, clip, which, ab):
    n = 192
    x = _hook_inputs(n, seed=g + which + int(clip * 10))
    # values at the codebook's own thresholds in the first group of row 4:
    # min 0, max 3 at clip 1 gives s = 1, z = 0 and t = x
    lo, hi = O.codebook_thresholds(*ab)
    x[4] = np.float32(1.0)
    x[4, :8] = np.array([0.0, 3.0, lo, hi, 1.5, np.nextafter(lo, 9), np.nextafter(hi, -9), 2.0], np.float32)
    got, gsz = _run_hook(x, g, clip, which, ab)
    ref_codes = np.zeros((n, 128), np.uint8)
    for i in range(n):
        c, s, z = O.quantize_vector_codebook(x[i], g, clip, *ab)
        ref_codes[i] = c
        np.testing.assert_array_equal(gsz[i, :, 0].view(np.uint16), s.view(np.uint16))
        np.testing.assert_array_equal(gsz[i, :, 1].view(np.uint16), z.view(np.uint16))
    if which == 0:
        ref = np.concatenate([O.pack_k_row(r) for r in ref_codes])
    else:
        ref = np.concatenate([O.pack_v_block(ref_codes[64 * k:64 * (k + 1)]) for k in range(n // 64)])
    np.testing.assert_array_equal(got, ref)
    if ab == O.UNIFORM_CODEBOOK:  # the uniform levels are the plain quantiser, byte for byte
        plain, psz = _run_hook(x, g, clip, which, None)
        np.testing.assert_array_equal(got, plain)
        np.testing.assert_array_equal(gsz.view(np.uint16), psz.view(np.uint16))


def _calib_ctx(G, g, mode, clip_k, clip_v, seed):
    Hkv = 2
    cfg = oscar.make_config(1, G * Hkv, Hkv, g, max_batch=1, max_pages_per_req=1, num_pages=1)
    ctx = oscar.oscar_create(cfg)
    stats = [synth.head_stats(seed, "cbfit", 0, h, n_out=4, f_key=20.0) for h in range(Hkv)]
    sets = [synth.calibration_set(seed, "cbfit", 0, h, stats[h], G=G, n=512) for h in range(Hkv)]
    if mode == oscar.ROT_OSCAR:
        U = [O.calibrate(*(t.float().numpy() for t in s)) for s in sets]
        UK = np.stack([u[0] for u in U]).astype(np.float32)
        UV = np.stack([u[1] for u in U]).astype(np.float32)
    else:
        UK = UV = np.stack([np.eye(128, dtype=np.float32)] * Hkv)
    oscar.oscar_set_rotation(ctx, 0, UK, UV, [clip_k] * Hkv, [clip_v] * Hkv, mode)
    return cfg, ctx, sets, UK, UV


@pytest.mark.parametrize("g,mode,clips", [(128, oscar.ROT_OSCAR, (0.95, 0.9)), (32, oscar.ROT_HADAMARD, (1.0, 0.8)),
                                          (64, oscar.ROT_NONE, (0.9, 1.0))])
def test_codebook_fit_matches_oracle(g, mode, clips):
    cfg, ctx, sets, UK, UV = _calib_ctx(4, g, mode, clips[0], clips[1], seed=g)
    try:
        for h, (Q, K, V) in enumerate(sets):
            for which, X, U, clip in ((0, K, UK, clips[0]), (1, V, UV, clips[1])):
                N = X.shape[0]
                Xd = X.cuda().contiguous()
                scratch = oscar.codebook_scratch(N)
                a, b, up = oscar.oscar_fit_codebook(ctx, 0, h, which, Xd, N, scratch)
                Xr = O.rotate_to_f32(X.float().numpy(), O.rotation(U[h].astype(np.float64), mode))
                ao, bo, upo = O.fit_codebook(Xr, g, clip)
                assert abs(a - ao) <= FIT_TOL * bo and abs(b - bo) <= FIT_TOL * bo, (h, which, a, ao, b, bo)
                assert abs(up - upo) <= 2 and up >= 1
                print(f"g={g} mode={mode} head {h} {'KV'[which]}: a={a:.5f} b={b:.5f} updates={up}")
    finally:
        oscar.oscar_destroy(ctx)


def _codebooks(Hkv, seed):
    rng = np.random.default_rng(seed)
    k = np.stack([[rng.uniform(0.3, 0.6), rng.uniform(1.2, 1.7)] for _ in range(Hkv)]).astype(np.float32)
    v = np.stack([[rng.uniform(0.3, 0.6), rng.uniform(1.2, 1.7)] for _ in range(Hkv)]).astype(np.float32)
    return k, v


def _check_decode(sc, q, out, lse):
    hc = GS.HostCache(sc)
    qn = q.float().cpu().numpy()
    for b, L in enumerate(sc.lengths):
        got = out[b].float().cpu().numpy()
        if int(hc.seq[b]) == 0:
            assert np.all(got == 0)
            continue
        ref, rlse = GS.oracle_decode(sc, hc, qn, b)
        assert _rel(got, ref) <= REL_TOL, (b, _rel(got, ref))
        assert np.abs(lse[b].cpu().numpy() - rlse).max() <= LSE_TOL, b
    return hc


@pytest.mark.parametrize("G,g", [(4, 128), (8, 32), (2, 64), (1, 128)])
def test_codebook_decode_matches_oracle(G, g):
    lengths = [0, 1, 319, 321, 385, 700, 64 * 9 + 320 + 17, 3000]
    sc = GS.build(f"cbdec{G}{g}", lengths, Hq=2 * G, Hkv=2, g=g, interleave=True, calib_n=512,
                  codebook=_codebooks(2, G * 100 + g))
    try:
        q = GS.queries(sc, seed=5)
        for impl in (oscar.DECODE_TENSOR, oscar.DECODE_CUDA_CORE):  # the option does not matter
            for part in (oscar.PARTITION_ITEMS, oscar.PARTITION_BALANCED):
                oscar.oscar_set_option(sc.ctx, oscar.OPT_DECODE_PARTITION, part)
                out, lse = GS.decode(sc, q, impl)
                assert oscar.oscar_get_error(sc.ctx) == 0
                hc = _check_decode(sc, q, out, lse)
        n, bad = GS.compare_history(sc, hc, 6, 1, list(range(64, 64 + 593)), list(range(593)))
        assert bad <= 1e-4 * n
    finally:
        sc.close()


def test_codebook_append_demote_and_fused_step():
    """Appends with demotion (oscar_append) and the fused step
    (oscar_decode_step) under a codebook: same cache and outputs bit for bit,
    codes as the oracle quantises them, outputs as the oracle computes them."""
    lengths = [300, 64, 1500]
    cb = _codebooks(2, 7)
    scs = [GS.build("cbstep", lengths, Hq=8, Hkv=2, g=128, extra_tokens=90, calib_n=512, codebook=cb)
           for _ in range(2)]
    try:
        a, b = scs
        scratch = [oscar.alloc_scratch(s_.cfg) for s_ in scs]
        for t in range(90):
            k = torch.stack([a.K[i][:, lengths[i] + t] for i in range(3)]).contiguous()
            v = torch.stack([a.V[i][:, lengths[i] + t] for i in range(3)]).contiguous()
            q = GS.queries(a, seed=400 + t)
            outs = []
            for j, s_ in enumerate(scs):
                out = torch.empty_like(q)
                lse = torch.empty(q.shape[0], q.shape[1], dtype=torch.float32, device=q.device)
                if j == 0:
                    oscar.oscar_decode_step(s_.ctx, 0, s_.cache, k, v, q, out, lse, scratch[j], 3)
                else:
                    oscar.oscar_append(s_.ctx, 0, s_.cache, k, v, 3)
                    oscar.oscar_decode(s_.ctx, 0, s_.cache, q, out, lse, scratch[j], 3)
                outs.append((out, lse))
            torch.cuda.synchronize()
            assert torch.equal(outs[0][0], outs[1][0]), t
        for s_ in scs:
            assert oscar.oscar_get_error(s_.ctx) == 0
        for key in ("pool", "ring_k", "seq_lens", "hist_lens"):
            assert torch.equal(a.cache[key], b.cache[key]), key
        a.lengths = [L + 90 for L in lengths]
        hc = _check_decode(a, q, *outs[0])
        H0 = int(hc.hist[0])
        assert H0 == 390 - 320
        n, bad = GS.compare_history(a, hc, 0, 1, list(range(64, 64 + H0)), list(range(H0)))
        assert bad <= 1e-4 * n
    finally:
        for s_ in scs:
            s_.close()


def test_uniform_codebook_keeps_the_default_decode_bit_for_bit():
    lengths = [700, 2000]
    u = np.tile(np.float32(O.UNIFORM_CODEBOOK), (2, 1))
    scs = [GS.build("cbuni", lengths, Hq=8, Hkv=2, g=128, calib_n=512, codebook=cbk) for cbk in (None, (u, u))]
    try:
        q = GS.queries(scs[0], seed=9)
        o0, l0 = GS.decode(scs[0], q)
        o1, l1 = GS.decode(scs[1], q)
        assert torch.equal(scs[0].cache["pool"], scs[1].cache["pool"])
        assert torch.equal(o0, o1) and torch.equal(l0, l1)
    finally:
        for s_ in scs:
            s_.close()


def test_codebook_clip_errors_match_oracle():
    G, N, g = 4, 192, 64
    Hkv = 2
    cfg = oscar.make_config(1, G * Hkv, Hkv, g, max_batch=1, max_pages_per_req=1, num_pages=1)
    ctx = oscar.oscar_create(cfg)
    try:
        st = synth.head_stats(3, "cbclip", 0, 0, n_out=8, f_key=30.0)
        Q, K, V = (t.cuda().contiguous() for t in synth.calibration_set(3, "cbclip", 0, 0, st, G=G, n=N))
        eye = np.stack([np.eye(128, dtype=np.float32)] * Hkv)
        oscar.oscar_set_rotation(ctx, 0, eye, eye, [1.0] * Hkv, [1.0] * Hkv, oscar.ROT_HADAMARD)
        cbk, cbv = _codebooks(Hkv, 3)
        oscar.oscar_set_codebook(ctx, 0, cbk, cbv)
        ratios = [1.0, 0.9, 0.8]
        scratch = oscar.calibration_scratch(G, N, len(ratios))
        ek, ev, bk, bv = oscar.oscar_clip_errors(ctx, 0, 1, Q, K, V, N, ratios, scratch)
        Qn, Kn, Vn = (t.float().cpu().numpy() for t in (Q, K, V))
        R = O.rotation(np.eye(128), O.ROT_HADAMARD)
        ck = (float(cbk[1][0]), float(cbk[1][1]))
        cv = (float(cbv[1][0]), float(cbv[1][1]))
        ek_o, ev_o, _, _ = O.clip_search(Qn, Kn, Vn, R, R, g, ratios, ck, cv)
        np.testing.assert_allclose(ek, ek_o, rtol=2e-3)
        np.testing.assert_allclose(ev, ev_o, rtol=2e-3)
    finally:
        oscar.oscar_destroy(ctx)


def test_codebook_host_rules():
    cfg = oscar.make_config(1, 8, 2, 128, max_batch=1, max_pages_per_req=4, num_pages=8)
    ctx = oscar.oscar_create(cfg)
    try:
        for bad in ([[0.6, 0.5], [0.5, 1.5]], [[0.5, 3.5], [0.5, 1.5]], [[-0.1, 1.0], [0.5, 1.5]],
                    [[np.nan, 1.0], [0.5, 1.5]]):
            with pytest.raises(oscar.OscarError):
                oscar.oscar_set_codebook(ctx, 0, bad, None)
        with pytest.raises(oscar.OscarError):
            oscar.oscar_set_codebook(ctx, 1, None, None)  # no such layer
        oscar.oscar_set_codebook(ctx, 0, [[0.45, 1.5], [0.5, 1.5]], None)
        cache = oscar.alloc_cache(cfg, "cuda")
        q = torch.zeros(1, 4, 8, 128, dtype=torch.bfloat16, device="cuda")
        k = torch.zeros(1, 4, 2, 128, dtype=torch.bfloat16, device="cuda")
        out = torch.empty_like(q)
        scratch = oscar.alloc_scratch(cfg, "cuda", prefill=True)
        for impl in (oscar.PREFILL_TCGEN05, oscar.PREFILL_MMA_SYNC):  # both run (the mma.sync kernel)
            oscar.oscar_set_option(ctx, oscar.OPT_PREFILL_IMPL, impl)
            oscar.oscar_prefill(ctx, 0, cache, q, k, k, 4, out, None, scratch, 1)
        oscar.oscar_set_codebook(ctx, 0, None, None)  # back to uniform
        oscar.oscar_prefill(ctx, 0, cache, q, k, k, 4, out, None, scratch, 1)
        torch.cuda.synchronize()
        X = torch.zeros(16, 128, dtype=torch.bfloat16, device="cuda")
        with pytest.raises(oscar.OscarError):
            oscar.oscar_fit_codebook(ctx, 0, 0, 0, X, 16, oscar.codebook_scratch(8))  # scratch too small
        with pytest.raises(oscar.OscarError):
            oscar.oscar_fit_codebook(ctx, 0, 2, 0, X, 16, oscar.codebook_scratch(16))  # kv head out of range
        a, b, up = oscar.oscar_fit_codebook(ctx, 0, 0, 1, X, 16, oscar.codebook_scratch(16))
        # every group has a zero scale: no values, the start is kept (as the oracle does)
        assert (a, b, up) == O.lloyd_max_folded(np.zeros(0))
    finally:
        oscar.oscar_destroy(ctx)


@pytest.mark.parametrize("G,g,T", [(4, 128, 64), (8, 32, 17), (2, 64, 40)])
def test_codebook_prefill_matches_oracle(G, g, T):
    """Chunked prefill over caches written with per-head codebooks (the
    mma.sync kernel dequantises s·level(code) + z) against the oracle."""
    from test_gpu_prefill import check_all, chunk_inputs, run_prefill

    lengths = [0, 330, 1000, 64 * 7 + 320 + 9]
    sc = GS.build(f"cbpf{G}{g}", lengths, Hq=2 * G, Hkv=2, g=g, interleave=True, calib_n=512, extra_tokens=T,
                  codebook=_codebooks(2, 31 * G + g))
    try:
        q, k, v = chunk_inputs(sc, T, seed=G + g)
        for impl in (oscar.PREFILL_TCGEN05, oscar.PREFILL_MMA_SYNC):
            out, lse = run_prefill(sc, q, k, v, impl=impl)
            assert oscar.oscar_get_error(sc.ctx) == 0
            check_all(sc, q, k, v, out, lse)
    finally:
        sc.close()
