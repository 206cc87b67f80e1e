"""GPU checks of the BF16-history append and of the synthetic serving loop:
the appended cache state is exact, and the outputs of requests decoded inside
the loop (admitted, moved between slots, stepped with others) match the oracle
on the loop's own cache contents, for INT2 and BF16 history."""
import types

import numpy as np
import pytest
import torch

import oracle as O
from bit_kv_cache_int2_gb300 import build as B
from bit_kv_cache_int2_gb300 import oscar, serving, synth

pytestmark = pytest.mark.gpu

import gpu_scenario as GS  # noqa: E402

REL_TOL = 1e-2
LSE_TOL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def built():
    B.build()
    oscar.lib()


def _rel(a, b):
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-30))


def test_bf16_history_append_matches_oracle():
    lengths, n_app = [250, 700], 150
    sc = GS.build("bfapp", lengths, Hq=4, Hkv=2, g=128, bf16_history=True, mode=oscar.ROT_NONE,
                  extra_tokens=n_app, calib_n=256)
    try:
        for t in range(n_app):
            k = torch.stack([sc.K[b][:, L + t] for b, L in enumerate(lengths)]).contiguous()
            v = torch.stack([sc.V[b][:, L + t] for b, L in enumerate(lengths)]).contiguous()
            oscar.oscar_append_bf16_history(sc.ctx, sc.cache, k, v, len(lengths))
        assert oscar.oscar_get_error(sc.ctx) == 0
        hc = GS.HostCache(sc)
        for b, L in enumerate(lengths):
            n = L + n_app
            H = max(n - 320, 0)
            assert (int(hc.seq[b]), int(hc.hist[b])) == (n, H)
            hk, hv = hc.history_bf16(b, 0)
            for h in range(2):
                hk, hv = hc.history_bf16(b, h)
                np.testing.assert_array_equal(hk, sc.K[b][h, 64:64 + H].float().cpu().numpy())
                np.testing.assert_array_equal(hv, sc.V[b][h, 64:64 + H].float().cpu().numpy())
                wk, wv = hc.window(b, h)
                ref_k = np.concatenate([sc.K[b][h, :min(n, 64)].float().cpu().numpy(),
                                        sc.K[b][h, 64 + H:n].float().cpu().numpy()])
                np.testing.assert_array_equal(wk, ref_k)
        q = GS.queries(sc, seed=41)
        out, lse = GS.decode(sc, q)
        qn = q.float().cpu().numpy()
        for b in range(len(lengths)):
            ref, rlse = GS.oracle_decode(sc, hc, qn, b)
            assert _rel(out[b].float().cpu().numpy(), ref) <= REL_TOL
            assert np.abs(lse[b].cpu().numpy() - rlse).max() <= LSE_TOL
    finally:
        sc.close()


def _draw_fn(stats, Hkv, G, seed):
    def draw(req):
        n = req.prefix + req.gen
        K = torch.stack([synth.draw_keys(stats[h], n, synth.stream_seed(seed, "srvK", req.rid, h), "cuda")
                         for h in range(Hkv)])
        V = torch.stack([synth.draw_values(stats[h], n, synth.stream_seed(seed, "srvV", req.rid, h), "cuda")
                         for h in range(Hkv)])
        Q = torch.stack([synth.draw_queries(stats[h], req.gen * G, synth.stream_seed(seed, "srvQ", req.rid, h),
                                            "cuda").view(req.gen, G, 128) for h in range(Hkv)], dim=1)
        return K.contiguous(), V.contiguous(), Q.reshape(req.gen, Hkv * G, 128).contiguous()
    return draw


@pytest.mark.parametrize("fmt", ["int2", "bf16"])
def test_serving_loop_outputs_match_oracle(fmt):
    Hq, Hkv, g, max_batch = 8, 2, 64, 4
    G = Hq // Hkv
    rng = np.random.default_rng(7)
    reqs = [serving.Request(rid=i, prefix=int(rng.integers(200, 1300)), gen=int(rng.integers(4, 24)))
            for i in range(9)]
    pool_pages = 40  # room for two or three requests at a time
    mpr = max(serving.pages_needed(r.prefix, r.gen) for r in reqs)
    cfg = oscar.make_config(1, Hq, Hkv, g, max_batch=max_batch, max_pages_per_req=mpr, num_pages=pool_pages)
    ctx = oscar.oscar_create(cfg)
    mode = oscar.ROT_HADAMARD if fmt == "int2" else oscar.ROT_NONE
    eye = np.stack([np.eye(128, dtype=np.float32)] * Hkv)
    oscar.oscar_set_rotation(ctx, 0, eye, eye, [0.95] * Hkv, [0.95] * Hkv, mode)
    cache = oscar.alloc_cache(cfg, "cuda", bf16_history=(fmt == "bf16"))
    stats = [synth.head_stats(3, "serve", 0, h) for h in range(Hkv)]
    view = types.SimpleNamespace(cache=cache, cfg=cfg, bf16_history=(fmt == "bf16"), Hq=Hq, Hkv=Hkv, g=g,
                                 U_K=eye, U_V=eye, mode=mode)
    checked = []

    def on_step(active, q, out):
        if len(checked) >= 4:
            return
        step = sched.steps
        if step % 7 != 3:
            return
        torch.cuda.synchronize()
        hc = GS.HostCache(view)
        qn = q.float().cpu().numpy()
        for s in range(len(active)):
            ref, rlse = GS.oracle_decode(view, hc, qn, s)
            got = out[s].float().cpu().numpy()
            assert _rel(got, ref) <= REL_TOL, (fmt, step, s, _rel(got, ref))
        checked.append((step, len(active)))

    try:
        backend = serving.DeviceBackend(fmt, ctx, cfg, cache, _draw_fn(stats, Hkv, G, 11), on_step=on_step)
        sched = serving.Scheduler(serving.PagePool(pool_pages), max_batch, backend, mpr)
        for r in reqs:
            sched.submit(r)
        done = sched.run()
        torch.cuda.synchronize()
        assert oscar.oscar_get_error(ctx) == 0
        assert sorted(r.rid for r in done) == list(range(len(reqs)))
        assert sched.pool.available == pool_pages
        assert checked and max(n for _, n in checked) >= 2  # batches of several requests were checked
        print(fmt, "checked steps", checked)
    finally:
        oscar.oscar_destroy(ctx)
