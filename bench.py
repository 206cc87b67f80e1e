"""Benchmark of the OSCAR INT2 decode-attention step on one GB300.

Workload (default): Qwen3-8B-shaped single layer -- 32 query / 8 KV heads,
head_dim 128, batch 1, 100,000-token context (full prefix hit: 64 BF16 sink
tokens, 99,680 INT2 history tokens in 64-token pages with a random page table,
256 BF16 recent tokens), group size 128, clip 0.95, seeded synthetic
outlier/anisotropic K/V/Q.  One step = append one token (which demotes the
oldest recent token into INT2 history) + decode attention for the new query.

Prints one JSON line.  ``--impl reference`` times the CPU oracle instead (the
reference arm of this build: a plain fp64 NumPy restatement of the method).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import tempfile
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "INT2 decode-attn µs/call & HBM GB/s at 100K ctx; speedup vs own BF16 kernel"
UNIT = "us/call"

WORKLOADS = {
    # Qwen3-8B-shaped single layer at 100K context, batch 1, g = 128
    "qwen3_8b_100k": dict(B=1, Hq=32, Hkv=8, g=128, L=100_000, clip=0.95, n_out=4, f_key=20.0),
}


def decode_source_hash():
    import hashlib

    h = hashlib.sha256()
    for f in ("oscar_decode.cu", "oscar_internal.cuh"):
        with open(os.path.join(ROOT, "bit_kv_cache_int2_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def recorded_traffic():
    """DRAM bytes per decode launch from the committed ncu capture, if it was
    taken on the current decode sources (else None)."""
    try:
        with open(os.path.join(ROOT, "profiles", "decode_main_traffic.json")) as f:
            d = json.load(f)
        if d.get("source_sha256") == decode_source_hash():
            return float(d["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def tensor_peak():
    """Dense fp16/bf16 tensor TFLOP/s (burst: the prefill is timed alone)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def prefill_flops(lengths, T, Hq):
    """Algorithmic FLOPs of one chunked prefill: chunk token t of a request with
    L cached tokens scores and sums over L + t + 1 keys, 4·d FLOPs each per query head."""
    return sum(Hq * 4 * 128 * (L + t + 1) for L in lengths for t in range(T))


# --------------------------------------------------------------- multi-rank
def rank_env():
    """(world size, rank, local rank) from the launcher's environment (1, 0, 0 alone)."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(ms, dist, device):
    """The slowest rank's time: every rank gets the maximum (one all-reduce, then
    a barrier).  dist None means one process."""
    import torch

    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    if dist is not None:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        dist.barrier()
    return float(t.item())


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        # the raw samples; BENCH_CLOCKS_DIR keeps them somewhere of the caller's choosing
        out_dir = os.environ.get("BENCH_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(out_dir, f"clocks_bench_{os.getpid()}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 10:
                    rows.append(parts)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        load = []
        mx = None
        for r in rows:
            try:
                sm, smax, util = float(r[1]), float(r[2]), float(r[4])
            except ValueError:
                continue
            mx = smax
            if util > 0:
                load.append(sm)
            for i, n in enumerate(names):
                if r[6 + i].lower().startswith("active"):
                    reasons.add(n)
        allsm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        med = statistics.median(load) if load else (statistics.median(allsm) if allsm else None)
        return {"sm_mhz": med, "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(rows),
                "samples_under_load": len(load)}


# --------------------------------------------------------------- workload
def algorithmic_bytes(H, L, Hkv, g):
    """Bytes the decode must read: packed codes + fp16 s/z + BF16 windows + page table."""
    hist = H * (64 + (128 // g) * 8)
    recent = max(L - 64 - H, 0) if L > 64 else 0
    window = (min(L, 64) + recent) * 128 * 2 * 2
    pages = (H + 63) // 64 * 4
    return Hkv * (hist + window) + pages


def build_workload(wl, dev, n_copies, extra, seed=0, bf16_copies=0):
    import numpy as np
    import torch

    from bit_kv_cache_int2_gb300 import oscar, synth

    B, Hq, Hkv, g, L = wl["B"], wl["Hq"], wl["Hkv"], wl["g"], wl["L"]
    G = Hq // Hkv
    pages = (L + extra - 320 + 63) // 64 + 1
    cfg = oscar.make_config(1, Hq, Hkv, g, max_batch=B, max_pages_per_req=pages, num_pages=pages * B)
    ctx = oscar.oscar_create(cfg)
    stats = [synth.head_stats(seed, "bench", 0, h, n_out=wl["n_out"], f_key=wl["f_key"]) for h in range(Hkv)]
    # rotation bases from the library's GPU calibration (covariances on the
    # device, eigenvectors by cuSOLVER) on 2048 seeded calibration tokens
    UK, UV = [], []
    cscr = oscar.calibration_scratch(G, 2048, 0, dev)
    for h in range(Hkv):
        Qc, Kc, Vc = (t.to(dev).contiguous() for t in synth.calibration_set(seed, "bench", 0, h, stats[h], G=G,
                                                                          n=2048))
        uq, us, _, _ = oscar.oscar_calibrate(ctx, Qc, Kc, Vc, 2048, cscr)
        UK.append(uq)
        UV.append(us)
    del cscr
    UK, UV = np.stack(UK), np.stack(UV)
    oscar.oscar_set_rotation(ctx, 0, UK, UV, [wl["clip"]] * Hkv, [wl["clip"]] * Hkv, oscar.ROT_OSCAR)
    base = oscar.alloc_cache(cfg, dev)
    pt = synth.page_table(pages * B, [pages] * B, synth.stream_seed(seed, "bench", "pages"), True, pages)
    base["page_table"].copy_(pt.to(dev))
    n_all = L + extra
    Ks = torch.empty(B, Hkv, n_all, 128, dtype=torch.bfloat16, device=dev)
    Vs = torch.empty_like(Ks)
    for b in range(B):
        for h in range(Hkv):
            Ks[b, h] = synth.draw_keys(stats[h], n_all, synth.stream_seed(seed, "bench", b, h, "K"), dev)
            Vs[b, h] = synth.draw_values(stats[h], n_all, synth.stream_seed(seed, "bench", b, h, "V"), dev)
    oscar.oscar_import_tokens(ctx, 0, base, Ks[:, :, :L].contiguous(), Vs[:, :, :L].contiguous(), B, L)
    torch.cuda.synchronize()
    copies = [base] + [{k: v.clone() for k, v in base.items()} for _ in range(n_copies - 1)]
    bf = []
    if bf16_copies:
        bcfg = oscar.make_config(1, Hq, Hkv, g, max_batch=B, max_pages_per_req=pages, num_pages=pages * B)
        bctx = oscar.oscar_create(bcfg)
        bb = oscar.alloc_cache(bcfg, dev, bf16_history=True)
        bb["page_table"].copy_(pt.to(dev))
        oscar.oscar_import_bf16_history(bctx, bb, Ks[:, :, :L].contiguous(), Vs[:, :, :L].contiguous(), B, L)
        torch.cuda.synchronize()
        bf = [bb] + [{k: v.clone() for k, v in bb.items()} for _ in range(bf16_copies - 1)]
    else:
        bctx = None
    qs = torch.stack([torch.cat([synth.draw_queries(stats[h], G, synth.stream_seed(seed, "benchQ", b, h), dev)
                                 for h in range(Hkv)]) for b in range(B)]).contiguous()
    return dict(cfg=cfg, ctx=ctx, copies=copies, K=Ks, V=Vs, q=qs, U=(UK, UV), bf=bf, bctx=bctx, stats=stats)


BATCHED = {
    # Qwen3-4B-shaped layer, batch 32, per-request context uniform in [8K, 32K]
    "qwen3_4b_b32_8k_32k": dict(B=32, Hq=32, Hkv=8, g=128, lens=(8192, 32768), clip=0.95, n_out=4, f_key=20.0,
                                bf16=False),
    # Qwen3-32B-shaped layer (GQA 8), batch 8 at 131,072 tokens, INT2 and BF16 history
    "qwen3_32b_b8_131k": dict(B=8, Hq=64, Hkv=8, g=128, lens=(131072, 131072), clip=0.9, n_out=8, f_key=30.0,
                              bf16=True),
    # one layer of the Qwen3-8B-shaped stack: batch 16 at 65,536 tokens, g = 32
    "qwen3_8b_layer_b16_64k_g32": dict(B=16, Hq=32, Hkv=8, g=32, lens=(65536, 65536), clip=0.95, n_out=4,
                                       f_key=20.0, bf16=False),
}


def batched_measurement(dev, peak, steps=120, seed=0, configs=None, decode_warmup=5, decode_calls=100,
                        partition=0):
    """Decode step (append with demotion + attention) and attention alone at
    the batched configurations (`configs`, default BATCHED), rotating over
    cache copies larger than 3x L2.  Rotations are Hadamard-only: the
    kernels' work does not depend on R."""
    import numpy as np
    import torch

    from bit_kv_cache_int2_gb300 import oscar, synth

    l2 = torch.cuda.get_device_properties(torch.device(dev)).L2_cache_size
    res = {}
    for name, c in (BATCHED if configs is None else configs).items():
        Bsz, Hq, Hkv, g = c["B"], c["Hq"], c["Hkv"], c["g"]
        rng = np.random.default_rng(synth.stream_seed(seed, name, "lens"))
        lens = [int(x) for x in rng.integers(c["lens"][0], c["lens"][1] + 1, Bsz)]
        hist = [max(L - 320, 0) for L in lens]
        per_copy = sum(algorithmic_bytes(H, L, Hkv, g) for H, L in zip(hist, lens))
        n_copies = max(2, -(-3 * l2 // per_copy))
        extra = steps // n_copies + 8
        ppr = [(L + extra - 320 + 63) // 64 for L in lens]
        mpr, npages = max(ppr), sum(ppr)
        cfg = oscar.make_config(1, Hq, Hkv, g, max_batch=Bsz, max_pages_per_req=mpr, num_pages=npages)
        ctx = oscar.oscar_create(cfg)
        if partition:
            oscar.oscar_set_option(ctx, oscar.OPT_DECODE_PARTITION, partition)
        eye = np.stack([np.eye(128, dtype=np.float32)] * Hkv)
        oscar.oscar_set_rotation(ctx, 0, eye, eye, [c["clip"]] * Hkv, [c["clip"]] * Hkv, oscar.ROT_HADAMARD)
        base = oscar.alloc_cache(cfg, dev)
        base["page_table"].copy_(synth.page_table(npages, ppr, synth.stream_seed(seed, name, "pages"), True,
                                                  mpr).to(dev))
        stats = [synth.head_stats(seed, name, 0, h, n_out=c["n_out"], f_key=c["f_key"]) for h in range(Hkv)]
        bctx = oscar.oscar_create(cfg) if c["bf16"] else None
        bbase = oscar.alloc_cache(cfg, dev, bf16_history=True) if c["bf16"] else None
        if bbase is not None:
            bbase["page_table"].copy_(base["page_table"])
        knew = torch.empty(extra, Bsz, Hkv, 128, dtype=torch.bfloat16, device=dev)
        vnew = torch.empty_like(knew)
        for b, L in enumerate(lens):
            K = torch.stack([synth.draw_keys(stats[h], L + extra, synth.stream_seed(seed, name, b, h, "K"), dev)
                             for h in range(Hkv)])
            V = torch.stack([synth.draw_values(stats[h], L + extra, synth.stream_seed(seed, name, b, h, "V"), dev)
                             for h in range(Hkv)])
            knew[:, b] = K[:, L:].permute(1, 0, 2)
            vnew[:, b] = V[:, L:].permute(1, 0, 2)
            for cache, cx, bf in ((base, ctx, False), (bbase, bctx, True)):
                if cache is None:
                    continue
                view = {k: (v[b:b + 1] if k in ("page_table", "sink_k", "sink_v", "ring_k", "ring_v", "seq_lens",
                                                "hist_lens") else v) for k, v in cache.items()}
                Kp, Vp = K[:, :L].unsqueeze(0).contiguous(), V[:, :L].unsqueeze(0).contiguous()
                if bf:
                    oscar.oscar_import_bf16_history(cx, view, Kp, Vp, 1, L)
                else:
                    oscar.oscar_import_tokens(cx, 0, view, Kp, Vp, 1, L)
            del K, V
        torch.cuda.synchronize()
        copies = [base] + [{k: v.clone() for k, v in base.items()} for _ in range(n_copies - 1)]
        q = torch.stack([torch.cat([synth.draw_queries(stats[h], Hq // Hkv, synth.stream_seed(seed, name, "Q", b, h),
                                                       dev) for h in range(Hkv)]) for b in range(Bsz)]).contiguous()
        out = torch.empty_like(q)
        scratch = oscar.alloc_scratch(cfg, dev)
        dec = [oscar.bind_decode(ctx, 0, cc, q, out, None, scratch, Bsz) for cc in copies]
        stp = [oscar.bind_decode_step(ctx, 0, cc, q, out, None, scratch, Bsz) for cc in copies]
        nstep = [0] * n_copies
        tok = Bsz * Hkv * 128 * 2

        def step(i):
            j = i % n_copies
            stp[j](knew.data_ptr() + nstep[j] * tok, vnew.data_ptr() + nstep[j] * tok)
            nstep[j] += 1

        def timed(fn, n):
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for i in range(n):
                fn(i)
            e1.record()
            torch.cuda.synchronize()
            return e0.elapsed_time(e1) * 1e3 / n

        for i in range(n_copies):
            step(i)
        us_step = timed(step, steps - n_copies)
        for i in range(decode_warmup):
            dec[i % n_copies]()
        us_dec = timed(lambda i: dec[i % n_copies](), decode_calls)
        assert oscar.oscar_get_error(ctx) == 0 and torch.isfinite(out.float()).all()
        r = {"batch": Bsz, "q_heads": Hq, "kv_heads": Hkv, "group_size": g, "context": list(c["lens"]),
             "tokens": sum(lens), "step_us": us_step, "decode_us": us_dec, "bytes_per_decode": per_copy,
             "decode_hbm_gbs": per_copy / (us_dec * 1e-6) / 1e9, "decode_frac": per_copy / (us_dec * 1e-6) / 1e9 / peak,
             "tokens_per_s": Bsz / (us_step * 1e-6), "cache_copies": n_copies}
        del dec, stp, copies
        if bbase is not None:
            bcopies = [bbase, {k: v.clone() for k, v in bbase.items()}]
            bscr = oscar.alloc_scratch(cfg, dev)
            for i in range(3):
                oscar.oscar_decode_bf16_history(bctx, bcopies[i % 2], q, out, None, bscr, Bsz)
            us_bf = timed(lambda i: oscar.oscar_decode_bf16_history(bctx, bcopies[i % 2], q, out, None, bscr, Bsz), 20)
            r["bf16_history_decode_us"] = us_bf
            r["speedup_vs_bf16"] = us_bf / us_dec
            del bcopies
            oscar.oscar_destroy(bctx)
        del base, bbase, knew, vnew
        oscar.oscar_destroy(ctx)
        torch.cuda.empty_cache()
        res[name] = r
    return res


def stack_measurement(dev, peak, layers=36, Bsz=16, L=65536, g=32, steps=64, warm=3, seed=0):
    """The Qwen3-8B-shaped decode-attention stack: `layers` layers of 32 query /
    8 KV heads, batch 16 at 65,536 tokens, group size 32, per-layer rotations
    calibrated on the GPU from seeded synthetic calibration sets; `steps`
    consecutive decode steps, each running every layer's oscar_decode_step
    (append with one demotion per request, then attention).  Steady-state
    us per step (all layers) and HBM GB/s of the decode's algorithmic bytes."""
    import numpy as np
    import torch

    from bit_kv_cache_int2_gb300 import oscar, synth

    Hq, Hkv = 32, 8
    G = Hq // Hkv
    ppr = (L + warm + steps - 320 + 63) // 64
    cfg = oscar.make_config(layers, Hq, Hkv, g, max_batch=Bsz, max_pages_per_req=ppr, num_pages=Bsz * ppr)
    ctx = oscar.oscar_create(cfg)
    cscr = oscar.calibration_scratch(G, 2048, 0, dev)
    caches, calls = [], []
    scratch = oscar.alloc_scratch(cfg, dev)
    out = torch.empty(Bsz, Hq, 128, dtype=torch.bfloat16, device=dev)
    n_new = warm + steps
    knew = torch.empty(layers, n_new, Bsz, Hkv, 128, dtype=torch.bfloat16, device=dev)
    vnew = torch.empty_like(knew)
    qs = torch.empty(layers, n_new, Bsz, Hq, 128, dtype=torch.bfloat16, device=dev)
    t0 = time.perf_counter()
    for layer in range(layers):
        stats = [synth.head_stats(seed, "stack", layer, h, n_out=4, f_key=20.0) for h in range(Hkv)]
        UK, UV = [], []
        for h in range(Hkv):
            Qc, Kc, Vc = (t.to(dev).contiguous() for t in synth.calibration_set(seed, "stack", layer, h, stats[h],
                                                                              G=G, n=2048))
            uk, uv, _, _ = oscar.oscar_calibrate(ctx, Qc, Kc, Vc, 2048, cscr)
            UK.append(uk)
            UV.append(uv)
        oscar.oscar_set_rotation(ctx, layer, np.stack(UK), np.stack(UV), [0.95] * Hkv, [0.95] * Hkv,
                                 oscar.ROT_OSCAR)
        cache = oscar.alloc_cache(cfg, dev)
        cache["page_table"].copy_(synth.page_table(Bsz * ppr, [ppr] * Bsz, synth.stream_seed(seed, "stack", layer),
                                                   True, ppr).to(dev))
        K = torch.empty(Bsz, Hkv, L + n_new, 128, dtype=torch.bfloat16, device=dev)
        V = torch.empty_like(K)
        for b in range(Bsz):
            for h in range(Hkv):
                K[b, h] = synth.draw_keys(stats[h], L + n_new, synth.stream_seed(seed, "stack", layer, b, h, "K"), dev)
                V[b, h] = synth.draw_values(stats[h], L + n_new, synth.stream_seed(seed, "stack", layer, b, h, "V"),
                                            dev)
        oscar.oscar_import_tokens(ctx, layer, cache, K[:, :, :L].contiguous(), V[:, :, :L].contiguous(), Bsz, L)
        knew[layer] = K[:, :, L:].permute(2, 0, 1, 3)
        vnew[layer] = V[:, :, L:].permute(2, 0, 1, 3)
        qs[layer] = torch.stack([torch.cat([synth.draw_queries(stats[h], n_new * G, synth.stream_seed(
            seed, "stackQ", layer, b, h), dev).view(n_new, G, 128) for h in range(Hkv)], dim=1)
            for b in range(Bsz)], dim=1)
        del K, V
        caches.append(cache)
        calls.append(oscar.bind_decode_step_ptrs(ctx, layer, cache, out, None, scratch, Bsz))
    torch.cuda.synchronize()
    setup_s = time.perf_counter() - t0
    tok = Bsz * Hkv * 128 * 2
    qb = Bsz * Hq * 128 * 2

    def step(t):
        for layer in range(layers):
            calls[layer](knew[layer, t].data_ptr(), vnew[layer, t].data_ptr(), qs[layer, t].data_ptr())

    for t in range(warm):
        step(t)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for t in range(warm, n_new):
        step(t)
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / steps
    assert oscar.oscar_get_error(ctx) == 0 and torch.isfinite(out.float()).all()
    H_mid = L + warm + steps // 2 - 320
    per_layer = Bsz * algorithmic_bytes(H_mid, L + warm + steps // 2, Hkv, g)
    res = {"layers": layers, "batch": Bsz, "context": L, "group_size": g, "steps": steps, "us_per_step": us,
           "us_per_layer": us / layers, "bytes_per_step": layers * per_layer,
           "hbm_gbs": layers * per_layer / (us * 1e-6) / 1e9,
           "frac": layers * per_layer / (us * 1e-6) / 1e9 / peak, "tokens_per_s": Bsz / (us * 1e-6),
           "cache_gb": layers * sum(v.numel() * v.element_size() for v in caches[0].values()) / 1e9,
           "setup_s": setup_s,
           "note": "every step runs oscar_decode_step on each layer in turn (append with one demotion per request, "
                   "then attention); the 36 layers' caches (~29 GB) stream from HBM each step; bytes are the "
                   "decode's algorithmic bytes at the mid-run length"}
    del caches, calls, knew, vnew, qs
    oscar.oscar_destroy(ctx)
    torch.cuda.empty_cache()
    return res


def synth_queries(st, T, G, b, h, dev):
    """Seeded prefill queries of KV head h of request b: [T][G][128]."""
    from bit_kv_cache_int2_gb300 import synth

    return synth.draw_queries(st, T * G, synth.stream_seed(0, "benchPQ", b, h), dev).view(T, G, 128)


# ------------------------------------------------------------- oracle leg
def oracle_sample(cache_host, wl, U, q, heads, budget_s=20.0, demote_tokens=None):
    """Times the oracle's decode (+ one demotion) for KV heads of one request."""
    import numpy as np

    import oracle as O

    pool, pt, sink_k, sink_v, ring_k, ring_v, L, H = cache_host
    g, Hkv, G = wl["g"], wl["Hkv"], wl["Hq"] // wl["Hkv"]
    head_bytes = O.int2_head_block_bytes(g)
    page_bytes = head_bytes * Hkv
    t0 = time.perf_counter()
    done = 0
    for h in heads:
        pages = (H + 63) // 64
        blocks = np.stack([pool[int(p) * page_bytes + h * head_bytes:int(p) * page_bytes + (h + 1) * head_bytes]
                           for p in pt[:pages]])
        f = O.parse_head_block(blocks, g)
        hk = O.dequantize(f["k_codes"].reshape(-1, 128)[:H], f["k_s"].reshape(-1, 128 // g)[:H],
                          f["k_z"].reshape(-1, 128 // g)[:H], g)
        hv = O.dequantize(f["v_codes"].reshape(-1, 128)[:H], f["v_s"].reshape(-1, 128 // g)[:H],
                          f["v_z"].reshape(-1, 128 // g)[:H], g)
        slots = [(p - 64) % 256 for p in range(64 + H, L)]
        wk = np.concatenate([sink_k[h, :min(L, 64)], ring_k[h, slots]])
        wv = np.concatenate([sink_v[h, :min(L, 64)], ring_v[h, slots]])
        O.three_region_attention(q[h * G:(h + 1) * G], wk, wv, hk, hv, O.rotation(U[0][h]), O.rotation(U[1][h]))
        if demote_tokens is not None:
            R = O.rotation(U[0][h])
            O.quantize_vector(O.rotate_to_f32(demote_tokens[0][h], R), g, wl["clip"])
            R = O.rotation(U[1][h])
            O.quantize_vector(O.rotate_to_f32(demote_tokens[1][h], R), g, wl["clip"])
        done += 1
        if time.perf_counter() - t0 > budget_s:
            break
    el = time.perf_counter() - t0
    return el / done * Hkv, done


def oracle_prefill_sample(cache_host, wl, U, q, k, v, tokens=(0, 63)):
    """Times the oracle's chunked prefill for KV head 0 of one request on a
    sample of chunk tokens and scales it to the whole call: the history
    dequantisation once per KV head, the attention once per (token, KV head).
    q [T][Hq][128], k, v [T][Hkv][128] float64."""
    import numpy as np

    import oracle as O

    pool, pt, sink_k, sink_v, ring_k, ring_v, L, H = cache_host
    g, Hkv, G = wl["g"], wl["Hkv"], wl["Hq"] // wl["Hkv"]
    T = q.shape[0]
    head_bytes = O.int2_head_block_bytes(g)
    page_bytes = head_bytes * Hkv
    h = 0
    t0 = time.perf_counter()
    pages = (H + 63) // 64
    blocks = np.stack([pool[int(p) * page_bytes + h * head_bytes:int(p) * page_bytes + (h + 1) * head_bytes]
                       for p in pt[:pages]])
    f = O.parse_head_block(blocks, g)
    hk = O.dequantize(f["k_codes"].reshape(-1, 128)[:H], f["k_s"].reshape(-1, 128 // g)[:H],
                      f["k_z"].reshape(-1, 128 // g)[:H], g)
    hv = O.dequantize(f["v_codes"].reshape(-1, 128)[:H], f["v_s"].reshape(-1, 128 // g)[:H],
                      f["v_z"].reshape(-1, 128 // g)[:H], g)
    slots = [(p - 64) % 256 for p in range(64 + H, L)]
    wk = np.concatenate([sink_k[h, :min(L, 64)], ring_k[h, slots]])
    wv = np.concatenate([sink_v[h, :min(L, 64)], ring_v[h, slots]])
    t1 = time.perf_counter()
    O.chunk_prefill_attention(q[:, h * G:(h + 1) * G], k[:, h], v[:, h], wk, wv, hk, hv,
                              O.rotation(U[0][h]), O.rotation(U[1][h]), tokens=list(tokens))
    t2 = time.perf_counter()
    return Hkv * (t1 - t0) + Hkv * T * (t2 - t1) / len(tokens)


def oracle_calibration_sample(cal_set, ratios, n_heads):
    """The oracle's calibration (covariances + eigenbases) of one kv head and its
    clip search for one ratio, scaled to every kv head and ratio of the bench."""
    import oracle as O

    Q, K, V = (t.float().cpu().numpy() for t in cal_set)
    t0 = time.perf_counter()
    U_K, U_V = O.calibrate(Q, K, V)
    t1 = time.perf_counter()
    O.key_clip_error(Q, K, O.rotation(U_K), 128, ratios[0])
    O.value_clip_error(Q, K, V, O.rotation(U_V), 128, ratios[0])
    t2 = time.perf_counter()
    return {"calibrate_ms": (t1 - t0) * 1e3 * n_heads, "clip_search_ms": (t2 - t1) * 1e3 * n_heads * len(ratios),
            "cores": blas_threads(), "kind": "oracle",
            "sample": f"kv head 0 (calibration) and ratio 1.0 (clip search), scaled to {n_heads} kv heads and every ratio"}


def serving_measurement(wl, dev, n_req=48, gen=64, lo=8192, hi=24576, budget_requests=4, seed=0):
    """The same request list run by the synthetic serving loop under one KV
    memory budget, with INT2 history and with BF16 history.  The budget is what
    `budget_requests` average requests need in BF16 (history pages plus their
    BF16 sink/recent windows); each format gets as many batch slots and pages
    as fit in it.  Returns the bench's `serving` object."""
    import numpy as np
    import torch

    from bit_kv_cache_int2_gb300 import oscar, serving, synth

    Hq, Hkv, g = wl["Hq"], wl["Hkv"], wl["g"]
    G = Hq // Hkv
    rng = np.random.default_rng(seed)
    lengths = [int(x) for x in rng.integers(lo, hi + 1, n_req)]
    stats = [synth.head_stats(seed, "serve", 0, h, n_out=wl["n_out"], f_key=wl["f_key"]) for h in range(Hkv)]
    streams = {}
    for i, L in enumerate(lengths):
        n = L + gen
        K = torch.stack([synth.draw_keys(stats[h], n, synth.stream_seed(seed, "sK", i, h), dev) for h in range(Hkv)])
        V = torch.stack([synth.draw_values(stats[h], n, synth.stream_seed(seed, "sV", i, h), dev) for h in range(Hkv)])
        Q = torch.stack([synth.draw_queries(stats[h], gen * G, synth.stream_seed(seed, "sQ", i, h), dev).view(gen, G, 128)
                         for h in range(Hkv)], dim=1).reshape(gen, Hq, 128)
        streams[i] = (K.contiguous(), V.contiguous(), Q.contiguous())
    window_bytes = Hkv * 320 * 128 * 2 * 2  # sink + recent K and V per slot
    page_bytes = {"int2": Hkv * (4096 + 64 * (128 // g) * 8), "bf16": Hkv * 64 * 128 * 2 * 2}
    mean_pages = float(np.mean([serving.pages_needed(L, gen) for L in lengths]))
    budget = budget_requests * (mean_pages * page_bytes["bf16"] + window_bytes)
    mpr = max(serving.pages_needed(L, gen) for L in lengths)
    res = {}
    for fmt in ("int2", "bf16"):
        per_req = mean_pages * page_bytes[fmt] + window_bytes
        slots = int(max(1, min(64, budget // per_req)))
        pool_pages = int((budget - slots * window_bytes) // page_bytes[fmt])
        cfg = oscar.make_config(1, Hq, Hkv, g, max_batch=slots, max_pages_per_req=mpr, num_pages=pool_pages)
        ctx = oscar.oscar_create(cfg)
        eye = np.stack([np.eye(128, dtype=np.float32)] * Hkv)
        oscar.oscar_set_rotation(ctx, 0, eye, eye, [wl["clip"]] * Hkv, [wl["clip"]] * Hkv,
                                 oscar.ROT_HADAMARD if fmt == "int2" else oscar.ROT_NONE)
        cache = oscar.alloc_cache(cfg, dev, bf16_history=(fmt == "bf16"))
        batches = []
        backend = serving.DeviceBackend(fmt, ctx, cfg, cache, lambda r: streams[r.rid],
                                        on_step=lambda active, q, out: batches.append(len(active)), time_steps=True)
        reqs = [serving.Request(rid=i, prefix=L, gen=gen) for i, L in enumerate(lengths)]
        done, steps, sec = serving.run_job(backend, pool_pages, slots, mpr, reqs)
        assert oscar.oscar_get_error(ctx) == 0 and len(done) == n_req
        dsec = serving.step_seconds(backend)
        isec = serving.import_seconds(backend)
        res[fmt] = {"slots": slots, "pool_pages": pool_pages, "steps": steps, "seconds": sec,
                    "tokens_per_s": n_req * gen / sec, "decode_seconds": dsec, "import_seconds": isec,
                    "decode_tokens_per_s": n_req * gen / dsec, "mean_batch": float(np.mean(batches)),
                    "max_batch": int(max(batches))}
        oscar.oscar_destroy(ctx)
        del cache, backend
    torch.cuda.empty_cache()
    return {"requests": n_req, "generated_per_request": gen, "prefix_tokens": [lo, hi],
            "budget_mb": budget / 1e6, **res,
            "throughput_ratio": res["int2"]["tokens_per_s"] / res["bf16"]["tokens_per_s"],
            "decode_throughput_ratio": res["int2"]["decode_tokens_per_s"] / res["bf16"]["decode_tokens_per_s"],
            "note": "synthetic, one Qwen3-8B-shaped layer; each request imports its prefix from BF16 (standing in "
                    "for a prefix-cache hit; the INT2 import quantises it, which a stored INT2 prefix would not need) "
                    "and decodes with append + attention per step. tokens_per_s: wall time of the whole job (imports, "
                    "host scheduler in Python, steps); decode_tokens_per_s: device time of the decode steps only; "
                    "import_seconds: device time of the imports (CUDA events around each call)"}


def bench_config(args, wl):
    """The workload description both arms print (identical, so that the two
    lines name the same configuration)."""
    return {"workload": args.workload, "batch": wl["B"], "q_heads": wl["Hq"], "kv_heads": wl["Hkv"], "head_dim": 128,
            "context": wl["L"], "group_size": wl["g"], "clip": wl["clip"], "parallelism": "replicas",
            "l2": "every timed call reads a cache copy other than the last few: the copies rotated over total at "
                  "least 3x the L2 size (129 MB), so no call finds its history pages in L2 (the page copies are "
                  "marked evict-first; the copies' BF16 windows, 2% of a call's bytes, may stay in L2 between "
                  "calls, as a layer's windows can between decode steps)"}


def oracle_subprocess_seconds(host, wl, U, q, threads, budget_s):
    """oracle_sample run in a fresh interpreter whose BLAS and OpenMP pools
    are limited to `threads` (the pool size is fixed when numpy loads)."""
    import numpy as np

    with tempfile.TemporaryDirectory() as d:
        f = os.path.join(d, "in.npz")
        pool, pt, sk, sv, rk, rv, L, H = host
        np.savez(f, pool=pool, pt=pt, sk=sk, sv=sv, rk=rk, rv=rv, L=L, H=H, UK=U[0], UV=U[1], q=q)
        code = ("import json, sys, numpy as np; sys.path.insert(0, %r); import bench; d = np.load(%r); "
                "h = (d['pool'], d['pt'], d['sk'], d['sv'], d['rk'], d['rv'], int(d['L']), int(d['H'])); "
                "print(json.dumps(bench.oracle_sample(h, %r, (d['UK'], d['UV']), d['q'], list(range(%d)), "
                "budget_s=%r)))") % (ROOT, f, wl, wl["Hkv"], budget_s)
        env = dict(os.environ, OMP_NUM_THREADS=str(threads), OPENBLAS_NUM_THREADS=str(threads),
                   MKL_NUM_THREADS=str(threads))
        r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=600)
        if r.returncode != 0:
            return None, 0
        sec, done = json.loads(r.stdout.strip().splitlines()[-1])
        return sec, done


def blas_threads():
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(var):
            return int(os.environ[var])
    try:
        from threadpoolctl import threadpool_info

        n = [i.get("num_threads", 1) for i in threadpool_info()]
        if n:
            return max(n)
    except Exception:
        pass
    return os.cpu_count() or 1


# ------------------------------------------------------------------ arms
def run_reference(args, wl):
    """The oracle as the reference arm, on host cores, bounded sample."""
    import numpy as np
    import torch

    import oracle as O
    from bit_kv_cache_int2_gb300 import synth

    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    g, Hkv, Hq, L = wl["g"], wl["Hkv"], wl["Hq"], wl["L"]
    G = Hq // Hkv
    H = L - 320
    # one KV head's history, quantised by the oracle on 1024 seeded tokens and tiled
    h = 0
    st = synth.head_stats(0, "bench", 0, h, n_out=wl["n_out"], f_key=wl["f_key"])
    Qc, Kc, Vc = synth.calibration_set(0, "bench", 0, h, st, G=G, n=2048)
    U_Q, U_S = O.calibrate(Qc.float().numpy(), Kc.float().numpy(), Vc.float().numpy())
    U = (np.stack([U_Q.astype(np.float32)] * Hkv), np.stack([U_S.astype(np.float32)] * Hkv))
    base_k = synth.draw_keys(st, 1024, 1).float().numpy()
    base_v = synth.draw_values(st, 1024, 2).float().numpy()
    R_K, R_V = O.rotation(U[0][0]), O.rotation(U[1][0])
    blocks = []
    for p in range(16):
        kc, vc, ks, kz, vs, vz = [], [], [], [], [], []
        for t in range(64):
            c, s, z = O.quantize_vector(O.rotate_to_f32(base_k[64 * p + t], R_K), g, wl["clip"])
            kc.append(c); ks.append(s); kz.append(z)
            c, s, z = O.quantize_vector(O.rotate_to_f32(base_v[64 * p + t], R_V), g, wl["clip"])
            vc.append(c); vs.append(s); vz.append(z)
        ksz = np.stack([np.stack(ks), np.stack(kz)], -1).astype(np.float16).view(np.uint8).reshape(-1)
        vsz = np.stack([np.stack(vs), np.stack(vz)], -1).astype(np.float16).view(np.uint8).reshape(-1)
        blocks.append(np.concatenate([np.concatenate([O.pack_k_row(r) for r in kc]), O.pack_v_block(np.stack(vc)),
                                      ksz, vsz]))
    pages = (H + 63) // 64
    hb = O.int2_head_block_bytes(g)
    pool = np.zeros(pages * hb * Hkv, dtype=np.uint8)
    for p in range(pages):
        pool[p * hb * Hkv:p * hb * Hkv + hb] = blocks[p % 16]
    pt = np.arange(pages)
    sink = np.zeros((Hkv, 64, 128))
    ring = np.zeros((Hkv, 256, 128))
    sink[0] = synth.draw_keys(st, 64, 3).float().numpy()
    ring[0] = synth.draw_keys(st, 256, 4).float().numpy()
    q = synth.draw_queries(st, Hq, 5).float().numpy()
    tokens = (np.stack([base_k[0]] * Hkv), np.stack([base_v[0]] * Hkv))
    # Each step is a bounded sample: KV head 0 over the first S history tokens
    # (parse + dequantise + attention over them and the window, one demotion),
    # scaled to the whole step (H / S history, Hkv heads).  S is sized from one
    # timed probe so that W + K steps take about `budget` seconds.
    budget = 120.0
    probe_S = 4096
    t0 = time.perf_counter()
    oracle_sample((pool, pt, sink, sink, ring, ring, 320 + probe_S, probe_S), wl, U, q, [0], budget_s=60,
                  demote_tokens=tokens)
    t_probe = time.perf_counter() - t0
    per_step_s = budget / (args.warmup + args.steps)
    S = int(max(64, min(H, probe_S * per_step_s / max(t_probe, 1e-6))) // 64 * 64)
    scale = H / S
    per_step = []
    for i in range(args.warmup + args.steps):
        sec, _ = oracle_sample((pool, pt, sink, sink, ring, ring, 320 + S, S), wl, U, q, [0], budget_s=60,
                               demote_tokens=tokens)
        if i >= args.warmup:
            per_step.append(sec * scale)  # oracle_sample already scales one head to Hkv heads
    value = statistics.median(per_step) * 1e6
    # the time the oracle actually took per sampled step, before any scaling
    raw_us = value / (scale * Hkv)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": value / 1e3, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": bench_config(args, wl),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
                         "sample": f"per step: KV head 0 over {S} of the {H} history tokens (pages quantised by "
                                   f"the oracle from 1024 seeded tokens and tiled) + window + one demotion, "
                                   f"scaled x{scale:.1f} (history) and x{Hkv} (heads): an extrapolation, not a "
                                   f"timing of the whole step",
                         "measured_us_per_sampled_step": raw_us, "sampled_history_tokens": S,
                         "measured_us_per_sampled_history_token": raw_us / S, "extrapolated": True},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args, wl):
    import numpy as np
    import torch

    from bit_kv_cache_int2_gb300 import build as B
    from bit_kv_cache_int2_gb300 import oscar

    world, rank, local = rank_env()
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    B.build()
    W, K = args.warmup, args.steps
    l2 = torch.cuda.get_device_properties(local).L2_cache_size
    Hkv, g, Bsz = wl["Hkv"], wl["g"], wl["B"]
    per_copy = algorithmic_bytes(wl["L"] - 320, wl["L"], Hkv, g) * Bsz
    n_copies = max(2, -(-3 * l2 // per_copy))  # rotate over >= 3x L2 of caches
    Kp, nd, ne = min(K, 2000), max(200, min(K, 1000)), min(K, 1000)
    na = min(K, 200)  # demotion-only calls
    n_pc = max(200, K)  # steps timed one by one for the percentiles
    total_appends = W + K + n_pc + Kp + 2 * ne + na  # two end-to-end forms
    extra = max(total_appends // n_copies + 16, 80)  # appends per cache copy, with margin; >= a prefill chunk
    wk = build_workload(wl, dev, n_copies, extra, bf16_copies=2)
    ctx, cfg = wk["ctx"], wk["cfg"]
    scratch = oscar.alloc_scratch(cfg, dev)
    q = wk["q"]
    out = torch.empty_like(q)
    lse = torch.empty(Bsz, wl["Hq"], dtype=torch.float32, device=dev)
    L0 = wl["L"]
    state = {"n": [0] * n_copies}

    # the new tokens for every append, laid out [B][Hkv][128] contiguous per step
    n_new = extra
    kv_new = (wk["K"][:, :, L0:L0 + n_new].permute(2, 0, 1, 3).contiguous(),
              wk["V"][:, :, L0:L0 + n_new].permute(2, 0, 1, 3).contiguous())
    # arguments marshalled once per cache copy (the Python binding's per-call
    # overhead would otherwise approach the GPU time of a step)
    tok_bytes = Bsz * Hkv * 128 * 2
    k_base, v_base = kv_new[0].data_ptr(), kv_new[1].data_ptr()
    steps = [oscar.bind_decode_step(ctx, 0, wk["copies"][c], q, out, lse, scratch, Bsz) for c in range(n_copies)]
    decodes = [oscar.bind_decode(ctx, 0, wk["copies"][c], q, out, lse, scratch, Bsz) for c in range(n_copies)]

    def step(i):
        c = i % n_copies
        t = state["n"][c]
        steps[c](k_base + t * tok_bytes, v_base + t * tok_bytes)  # oscar_decode_step: append + decode
        state["n"][c] += 1
    stream = torch.cuda.current_stream()
    sampler = ClockSampler(local)
    sampler.start()
    for i in range(W):
        step(i)
    torch.cuda.synchronize()
    # ---- headline: K steps of append + decode
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(W, W + K):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    ms = max_over_ranks(ms, dist, dev)
    ms_per_step = ms / K
    err = oscar.oscar_get_error(ctx)
    assert err == 0, f"device error {err}"
    assert torch.isfinite(out.float()).all()
    # ---- the same steps timed one by one: median and spread over >= 200 steps
    pc_step = per_call_times(lambda i: step(W + K + i), n_pc, stream)
    step_med, step_p10, step_p90 = percentiles(pc_step)
    base_after_pc = W + K + n_pc
    # ---- per-kernel times over the same kind of steps (profiling pass)
    oscar.oscar_profile_enable(ctx, True)
    oscar.oscar_profile_read(ctx, 0, reset=True)
    lens_before = [int(c["hist_lens"][0]) for c in wk["copies"]]
    for i in range(base_after_pc, base_after_pc + Kp):
        step(i)
    torch.cuda.synchronize()
    prof = {}
    for kid, name in oscar.KERNEL_NAMES.items():
        n, tot = oscar.oscar_profile_read(ctx, kid)
        if n:
            prof[name] = {"launches": n, "avg_us": tot * 1e3 / n}
    oscar.oscar_profile_read(ctx, 0, reset=True)
    oscar.oscar_profile_enable(ctx, False)
    # algorithmic bytes of the decode launches in the profiled pass
    H_avg = statistics.mean(lens_before) + 0.5 * Kp / n_copies
    bytes_main = algorithmic_bytes(H_avg, wl["L"], Hkv, g) * Bsz
    peak, peak_kind = peaks()
    main_us = prof["decode_main"]["avg_us"]
    achieved = bytes_main / (main_us * 1e-6) / 1e9
    # ---- decode only: INT2 vs BF16 history (same q)
    def time_calls(fn, n):
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for i in range(n):
            fn(i)
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) * 1e3 / n

    for i in range(5):
        oscar.oscar_decode(ctx, 0, wk["copies"][i % n_copies], q, out, lse, scratch, Bsz)
    int2_us = time_calls(lambda i: decodes[i % n_copies](), nd)
    int2_med, int2_p10, int2_p90 = percentiles(per_call_times(lambda i: decodes[i % n_copies](), nd, stream))
    bf_out = torch.empty_like(q)
    bscratch = oscar.alloc_scratch(cfg, dev)
    for i in range(5):
        oscar.oscar_decode_bf16_history(wk["bctx"], wk["bf"][i % 2], q, bf_out, None, bscratch, Bsz)
    bf16_call = lambda i: oscar.oscar_decode_bf16_history(wk["bctx"], wk["bf"][i % 2], q, bf_out, None, bscratch, Bsz)
    bf16_us = time_calls(bf16_call, nd)
    bf16_med, bf16_p10, bf16_p90 = percentiles(per_call_times(bf16_call, nd, stream))
    # ---- the other INT2 decode kernels on the same caches and q (the choice
    # of the default is measured, not assumed)
    variants = {}
    for name, impl in (("tensor_single", oscar.DECODE_TENSOR_SINGLE), ("cuda_core", oscar.DECODE_CUDA_CORE),
                       ("tcgen05", oscar.DECODE_TCGEN05)):
        oscar.oscar_set_option(ctx, oscar.OPT_DECODE_IMPL, impl)
        calls_v = [oscar.bind_decode(ctx, 0, wk["copies"][c], q, out, lse, scratch, Bsz) for c in range(n_copies)]
        for i in range(3):
            calls_v[i % n_copies]()
        variants[name] = time_calls(lambda i: calls_v[i % n_copies](), 50 if name == "cuda_core" else 200)
    oscar.oscar_set_option(ctx, oscar.OPT_DECODE_IMPL, oscar.DECODE_TENSOR)
    assert oscar.oscar_get_error(ctx) == 0
    bf16_bytes = Hkv * Bsz * ((wl["L"] - 320) * 512 + 320 * 512) + ((wl["L"] - 320 + 63) // 64) * 4
    # ---- demotion alone (oscar_append; one token per request, each demoting one)
    appends = [oscar.bind_append(ctx, 0, wk["copies"][c], Bsz) for c in range(n_copies)]

    def append_only(i):
        c = i % n_copies
        t = state["n"][c]
        appends[c](k_base + t * tok_bytes, v_base + t * tok_bytes)
        state["n"][c] += 1

    app_us = time_calls(append_only, na)
    # per (request, kv head) and K|V: the evicted ring token and the new token in,
    # the new token into the ring, the codes and scale/zero of the demoted token out
    app_bytes = Bsz * Hkv * 2 * (3 * 256 + 32 + (128 // g) * 4)
    # ---- chunked prefill of 64 tokens over the same caches (attention only)
    T_pf = 64
    n_pf = min(K, 100)
    q_pf = torch.stack([torch.cat([synth_queries(wk["stats"][h], T_pf, wl["Hq"] // Hkv, b, h, dev)
                                   for h in range(Hkv)], dim=1) for b in range(Bsz)]).contiguous()
    k_pf = wk["K"][:, :, L0:L0 + T_pf].permute(0, 2, 1, 3).contiguous()
    v_pf = wk["V"][:, :, L0:L0 + T_pf].permute(0, 2, 1, 3).contiguous()
    out_pf = torch.empty_like(q_pf)
    pscratch = oscar.alloc_scratch(cfg, dev, prefill=True)
    pf_lens = [int(c["seq_lens"].sum()) for c in wk["copies"]]
    for i in range(3):
        oscar.oscar_prefill(ctx, 0, wk["copies"][i % n_copies], q_pf, k_pf, v_pf, T_pf, out_pf, None, pscratch, Bsz)
    pf_us = time_calls(lambda i: oscar.oscar_prefill(ctx, 0, wk["copies"][i % n_copies], q_pf, k_pf, v_pf, T_pf,
                                                     out_pf, None, pscratch, Bsz), n_pf)
    oscar.oscar_profile_enable(ctx, True)
    for i in range(min(n_pf, 20)):
        oscar.oscar_prefill(ctx, 0, wk["copies"][i % n_copies], q_pf, k_pf, v_pf, T_pf, out_pf, None, pscratch, Bsz)
    torch.cuda.synchronize()
    pf_prof = {}
    for kid in (oscar.KERNEL_PREFILL_PREP, oscar.KERNEL_PREFILL_ATTN, oscar.KERNEL_PREFILL_MERGE):
        n, tot = oscar.oscar_profile_read(ctx, kid)
        pf_prof[oscar.KERNEL_NAMES[kid]] = round(tot * 1e3 / max(n, 1), 3)
    oscar.oscar_profile_read(ctx, 0, reset=True)
    oscar.oscar_profile_enable(ctx, False)
    assert oscar.oscar_get_error(ctx) == 0
    assert torch.isfinite(out_pf.float()).all()
    pf_flops = statistics.mean(prefill_flops([L // Bsz] * Bsz, T_pf, wl["Hq"]) for L in pf_lens)
    tpk, tpk_kind = tensor_peak()
    pf_attn_tf = pf_flops / (pf_prof["prefill_attn"] * 1e-6) / 1e12
    # ---- offline calibration on the GPU: bases of every kv head, then the clip search
    from bit_kv_cache_int2_gb300 import synth

    G_cal, N_cal = wl["Hq"] // Hkv, 2048
    ratios = [1.0, 0.975, 0.95, 0.925, 0.9, 0.85, 0.8, 0.7]
    cal_sets = [tuple(t.to(dev).contiguous() for t in synth.calibration_set(0, "bench", 0, h, wk["stats"][h],
                                                                            G=G_cal, n=N_cal)) for h in range(Hkv)]
    cscr = oscar.calibration_scratch(G_cal, N_cal, len(ratios), dev)
    oscar.oscar_calibrate(ctx, *cal_sets[0], N_cal, cscr)  # warm-up (opens cuSOLVER)
    oscar.oscar_clip_errors(ctx, 0, 0, *cal_sets[0], N_cal, ratios, cscr)
    t0 = time.perf_counter()
    for h in range(Hkv):
        oscar.oscar_calibrate(ctx, *cal_sets[h], N_cal, cscr)
    t1 = time.perf_counter()
    for h in range(Hkv):
        oscar.oscar_clip_errors(ctx, 0, h, *cal_sets[h], N_cal, ratios, cscr)
    t2 = time.perf_counter()
    causal_pairs = N_cal * (N_cal + 1) / 2
    cal_flops = Hkv * (2 * 2 * G_cal * N_cal * 128 * 128 + G_cal * causal_pairs * 128 * 4)
    clip_flops = Hkv * (2 * G_cal * N_cal * 128 * 128 + len(ratios) * (2 * N_cal * 128 * 128 + G_cal * causal_pairs * 128 * 4))
    fp32_peak = 152 * 128 * 2 * 2.07e9 / 1e12  # FMA lanes x 2 FLOP x max SM clock
    # ---- Lloyd-Max codebook: per-head fits on the calibration keys and values,
    # the attention errors they leave against the uniform levels, and the decode
    # over cache copies written with them (a second context)
    cctx = oscar.oscar_create(cfg)
    oscar.oscar_set_rotation(cctx, 0, wk["U"][0], wk["U"][1], [wl["clip"]] * Hkv, [wl["clip"]] * Hkv,
                             oscar.ROT_OSCAR)
    fscr = oscar.codebook_scratch(N_cal, dev)
    oscar.oscar_fit_codebook(cctx, 0, 0, 0, cal_sets[0][1], N_cal, fscr)  # warm-up
    t3 = time.perf_counter()
    kab, vab, ups = [], [], []
    for h in range(Hkv):
        for which, dst in ((0, kab), (1, vab)):
            a_, b_, u_ = oscar.oscar_fit_codebook(cctx, 0, h, which, cal_sets[h][1 + which], N_cal, fscr)
            dst.append((a_, b_))
            ups.append(u_)
    t4 = time.perf_counter()
    oscar.oscar_set_codebook(cctx, 0, kab, vab)
    err = {"uniform": [0.0, 0.0], "codebook": [0.0, 0.0]}
    for name, cx in (("uniform", ctx), ("codebook", cctx)):
        for h in range(Hkv):
            ek_, ev_, _, _ = oscar.oscar_clip_errors(cx, 0, h, *cal_sets[h], N_cal, [wl["clip"]], cscr)
            err[name][0] += float(ek_[0])
            err[name][1] += float(ev_[0])
    cb_base = oscar.alloc_cache(cfg, dev)
    cb_base["page_table"].copy_(wk["copies"][0]["page_table"])
    oscar.oscar_import_tokens(cctx, 0, cb_base, wk["K"][:, :, :L0].contiguous(), wk["V"][:, :, :L0].contiguous(),
                              Bsz, L0)
    torch.cuda.synchronize()
    cb_copies = [cb_base] + [{k: v.clone() for k, v in cb_base.items()} for _ in range(n_copies - 1)]
    cdec = [oscar.bind_decode(cctx, 0, cb_copies[c], q, out, lse, scratch, Bsz) for c in range(n_copies)]
    for i in range(5):
        cdec[i % n_copies]()
    cb_us = time_calls(lambda i: cdec[i % n_copies](), nd)
    oscar.oscar_profile_enable(cctx, True)
    for i in range(50):
        cdec[i % n_copies]()
    ncb, tcb = oscar.oscar_profile_read(cctx, oscar.KERNEL_DECODE_MAIN, reset=True)
    oscar.oscar_profile_enable(cctx, False)
    cb_main_us = tcb * 1e3 / max(ncb, 1)
    for i in range(3):
        oscar.oscar_prefill(cctx, 0, cb_copies[i % n_copies], q_pf, k_pf, v_pf, T_pf, out_pf, None, pscratch, Bsz)
    cb_pf_us = time_calls(lambda i: oscar.oscar_prefill(cctx, 0, cb_copies[i % n_copies], q_pf, k_pf, v_pf, T_pf,
                                                        out_pf, None, pscratch, Bsz), 20)
    assert torch.isfinite(out_pf.float()).all()
    cb_bytes = algorithmic_bytes(L0 - 320, L0, Hkv, g) * Bsz
    assert oscar.oscar_get_error(cctx) == 0
    assert torch.isfinite(out.float()).all()
    codebook = {"fit_ms": (t4 - t3) * 1e3, "fits": 2 * Hkv, "mean_updates": float(np.mean(ups)),
                "k_ab": [[round(a_, 5), round(b_, 5)] for a_, b_ in kab],
                "v_ab": [[round(a_, 5), round(b_, 5)] for a_, b_ in vab],
                "logit_error_ratio": err["codebook"][0] / err["uniform"][0],
                "output_error_ratio": err["codebook"][1] / err["uniform"][1],
                "decode_us": cb_us, "decode_main_us": cb_main_us,
                "decode_main_hbm_gbs": cb_bytes / (cb_main_us * 1e-6) / 1e9,
                "decode_main_frac": cb_bytes / (cb_main_us * 1e-6) / 1e9 / peak,
                "vs_uniform_decode": cb_us / int2_us,
                "prefill_us": cb_pf_us,
                "note": "symmetric 4-level Lloyd-Max levels per kv head for K and V, fitted on the GPU from the "
                        "2048-token calibration sets at the workload's clip ratio; errors are the clip-search "
                        "objectives summed over kv heads (codebook / uniform); the codebook decode takes two "
                        "tensor-core products per operand (bit planes) over the same cache bytes; the prefill over a codebook "
                        "layer runs the mma.sync kernel (64-token chunk)"}
    del cb_copies, cb_base, cdec
    oscar.oscar_destroy(cctx)
    # ---- the batched configurations (parity-test shapes), timed here too
    batched = batched_measurement(dev, peak)
    batched["qwen3_8b_stack_36x_b16_64k_g32"] = stack_measurement(dev, peak)
    # ---- synthetic serving loop under one KV memory budget, INT2 vs BF16 history
    serve = serving_measurement(wl, dev)
    # ---- end to end through the public API with host buffers.  Each step's q,
    # k_new and v_new sit in one pinned host record and its output goes to a
    # pinned host buffer; every step moves those bytes across the host link.
    # (a) in place: the step's kernels read the record and write the output
    #     over NVLink-C2C (pinned host memory is addressable by the kernels);
    # (b) copies: one host-to-device copy of the record and one device-to-host
    #     copy of the output around the call.
    nq, nk = q.numel(), kv_new[0][0].numel()
    rec_h = torch.empty(n_new, nq + 2 * nk, dtype=q.dtype).pin_memory()
    rec_h[:, :nq] = q.reshape(1, -1).cpu()
    rec_h[:, nq:nq + nk] = kv_new[0].reshape(n_new, -1).cpu()
    rec_h[:, nq + nk:] = kv_new[1].reshape(n_new, -1).cpu()
    out_h = torch.empty(q.shape, dtype=q.dtype).pin_memory()
    rec_d = torch.empty(nq + 2 * nk, dtype=q.dtype, device=dev)
    q_d = rec_d[:nq].view(q.shape)
    base_i = W + K + Kp
    rec_bytes = rec_h.shape[1] * rec_h.element_size()
    rec0 = rec_h.data_ptr()
    zsteps = [oscar.bind_decode_step_ptrs(ctx, 0, wk["copies"][c], out_h, None, scratch, Bsz)
              for c in range(n_copies)]
    csteps = [oscar.bind_decode_step(ctx, 0, wk["copies"][c], q_d, out, None, scratch, Bsz) for c in range(n_copies)]
    kd_ptr = rec_d.data_ptr() + nq * 2
    vd_ptr = kd_ptr + nk * 2

    def e2e_in_place(i):
        c = i % n_copies
        t = state["n"][c]
        r = rec0 + t * rec_bytes
        zsteps[c](r + nq * 2, r + (nq + nk) * 2, r)
        state["n"][c] += 1

    def e2e_copies(i):
        c = i % n_copies
        t = state["n"][c]
        rec_d.copy_(rec_h[t], non_blocking=True)
        csteps[c](kd_ptr, vd_ptr)
        out_h.copy_(out, non_blocking=True)
        state["n"][c] += 1

    e2e_us = time_calls(lambda i: e2e_in_place(base_i + i), ne)
    torch.cuda.synchronize()
    e2e_ok = bool(torch.isfinite(out_h.float()).all())
    e2e_copy_us = time_calls(lambda i: e2e_copies(base_i + ne + i), ne)
    clocks = sampler.stop()
    h2d = q.numel() * 2 + kv_new[0][0].numel() * 2 * 2
    d2h = q.numel() * 2
    # ---- CPU oracle on the GPU's own cache (bounded sample)
    cpu = None
    prefill_cpu = None
    calib_cpu = None
    if rank == 0:
        c0 = wk["copies"][0]
        L = int(c0["seq_lens"][0])
        H = int(c0["hist_lens"][0])
        host = (c0["pool"].cpu().numpy(), c0["page_table"][0].cpu().numpy(),
                c0["sink_k"][0].float().cpu().numpy().astype(np.float64),
                c0["sink_v"][0].float().cpu().numpy().astype(np.float64),
                c0["ring_k"][0].float().cpu().numpy().astype(np.float64),
                c0["ring_v"][0].float().cpu().numpy().astype(np.float64), L, H)
        qh = q[0].float().cpu().numpy().astype(np.float64)
        sec, done = oracle_sample(host, wl, wk["U"], qh, list(range(Hkv)), budget_s=args.cpu_budget)
        sec1, done1 = oracle_subprocess_seconds(host, wl, wk["U"], qh, 1, args.cpu_budget)
        cpu = {"value": sec * 1e6, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
               "sample": f"{done} of {Hkv} KV heads of one decode step on the GPU-built cache, scaled to {Hkv}",
               "single_thread_value": None if sec1 is None else sec1 * 1e6,
               "single_thread_sample": f"{done1} of {Hkv} KV heads, one BLAS / OpenMP thread, scaled to {Hkv}"}
        psec = oracle_prefill_sample(host, wl, wk["U"], q_pf[0].float().cpu().numpy().astype(np.float64),
                                     k_pf[0].float().cpu().numpy().astype(np.float64),
                                     v_pf[0].float().cpu().numpy().astype(np.float64))
        prefill_cpu = {"value": psec * 1e6, "unit": "us/call", "cores": blas_threads(), "kind": "oracle",
                       "sample": f"KV head 0, chunk tokens 0 and 63; scaled to {T_pf} tokens x {Hkv} KV heads"}
        calib_cpu = oracle_calibration_sample(cal_sets[0], ratios, Hkv)
    n_launch = 3 * K  # append + q rotation, decode, merge per step
    value = ms_per_step * 1e3 / world
    vs_bf16 = {"int2_decode_us_median": int2_med, "bf16_history_decode_us_median": bf16_med,
               "speedup_vs_bf16": bf16_med / int2_med, "int2_decode_us_mean": int2_us,
               "bf16_history_decode_us_mean": bf16_us, "speedup_vs_bf16_mean": bf16_us / int2_us}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": ms_per_step, "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "int2 codes, f16/bf16 tensor-core MMA, fp32 accumulate", "data": "synthetic",
        "config": bench_config(args, wl),
        "step_us": {"mean": value, "median": step_med, "p10": step_p10, "p90": step_p90, "calls": n_pc,
                    "note": "mean over the K bulk-timed steps (value); median and spread from a second run of "
                            f"{n_pc} steps with an event around each (which ends the programmatic overlap "
                            "between consecutive steps)"},
        "tokens_per_s": world * Bsz / (ms_per_step * 1e-3),
        "decode_us": int2_us, "bf16_history_decode_us": bf16_us, "speedup_vs_bf16": bf16_us / int2_us,
        "decode_us_percentiles": {"int2": [int2_p10, int2_med, int2_p90], "bf16_history": [bf16_p10, bf16_med, bf16_p90],
                                  "calls": nd, "order": "p10, median, p90"},
        "decode_variants_us": dict(variants, tensor_pairs_default=int2_us,
                                   note="oscar_decode on the same caches and q with OSCAR_OPT_DECODE_IMPL set to each "
                                        "INT2 kernel (mean per call)"),
        "bf16_history_hbm_gbs": bf16_bytes / (bf16_us * 1e-6) / 1e9,
        "kernels_us": {k: round(v["avg_us"], 3) for k, v in prof.items()},
        "demotion": {"us_per_call": app_us, "bytes_per_call": app_bytes,
                     "achieved_gbs": app_bytes / (app_us * 1e-6) / 1e9,
                     "frac": app_bytes / (app_us * 1e-6) / 1e9 / peak,
                     "note": "one token per (request, kv head): latency-bound, not bandwidth-bound"},
        "prefill": {"chunk_tokens": T_pf, "us_per_call": pf_us, "kernels_us": pf_prof,
                    "flops_per_call": pf_flops, "tflops": pf_flops / (pf_us * 1e-6) / 1e12,
                    "attn_tflops": pf_attn_tf, "peak_tflops": tpk, "peak_kind": tpk_kind,
                    "attn_frac": pf_attn_tf / tpk, "cpu_baseline": prefill_cpu,
                    "note": "64 new tokens per request attending to the same 100K cache; tcgen05.mma "
                            "kind::f16 (M=128) with Q, S, P, O in tensor memory; bound: tensor; peak = "
                            "dense bf16 burst (fp16 runs at the same rate)"},
        "serving": serve,
        "batched": batched,
        "codebook": codebook,
        "calibration": {"kv_heads": Hkv, "tokens": N_cal, "query_heads_per_kv": G_cal, "ratios": len(ratios),
                        "calibrate_ms": (t1 - t0) * 1e3, "clip_search_ms": (t2 - t1) * 1e3,
                        "tflops": (cal_flops + clip_flops) / (t2 - t0) / 1e12, "bound": "alu",
                        "peak_tflops": fp32_peak, "frac": (cal_flops + clip_flops) / (t2 - t0) / 1e12 / fp32_peak,
                        "cpu_baseline": calib_cpu,
                        "note": "offline; fp32 CUDA-core kernels + cuSOLVER dsyevd; wall time of the synchronous calls"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": recorded_traffic(), "kernel": "decode_main",
                     "bytes_per_launch": bytes_main, "peak_kind": peak_kind, "kernel_us": main_us,
                     "vs_bf16_history": vs_bf16},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_us, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "form": "pinned host record read and output written in place by the kernels over NVLink-C2C",
                "with_copy_calls_us": e2e_copy_us, "outputs_finite": e2e_ok},
        "gpu_launches": n_launch,
        "clocks": clocks,
        "vs_bf16_history": vs_bf16,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def percentiles(xs):
    """median, p10, p90 of a list of per-call times."""
    import numpy as np

    a = np.asarray(xs, dtype=np.float64)
    return float(np.median(a)), float(np.percentile(a, 10)), float(np.percentile(a, 90))


def per_call_times(fn, n, stream):
    """CUDA-event time of each of n back-to-back calls on `stream` (µs): one
    event before every call and one after the last, so call i spans events i
    and i + 1.  The host enqueues ahead of the device, so each interval is the
    call's device time (an event between two calls ends their programmatic
    overlap, which a bulk-timed run keeps)."""
    import torch

    ev = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
    torch.cuda.synchronize()
    for i in range(n):
        ev[i].record(stream)
        fn(i)
    ev[n].record(stream)
    torch.cuda.synchronize()
    return [ev[i].elapsed_time(ev[i + 1]) * 1e3 for i in range(n)]


LEGS = ("decode", "step", "bf16", "append", "cuda_core", "tensor_single", "tcgen05", "prefill", "calibration")


def run_leg(args, wl):
    """One operation of the hot path on the 100K workload, alone: --warmup
    untimed calls, then --steps calls timed one by one with CUDA events,
    rotating over cache copies larger than 3x L2.  A short command for
    profiling one kernel (the full bench runs every other measurement too).
      decode        oscar_decode (INT2, default implementation)
      step          oscar_decode_step (append with its demotion + decode)
      bf16          oscar_decode_bf16_history (the BF16-history baseline)
      append        oscar_append (one token per request and kv head, each demoting one)
      cuda_core     oscar_decode with OSCAR_DECODE_CUDA_CORE
      tensor_single oscar_decode with OSCAR_DECODE_TENSOR_SINGLE
      tcgen05       oscar_decode with OSCAR_DECODE_TCGEN05
      prefill       oscar_prefill, a 64-token chunk
      calibration   oscar_calibrate then oscar_clip_errors (8 ratios) of one kv head's
                    2048-token calibration set, the heads in turn"""
    import torch

    from bit_kv_cache_int2_gb300 import build as B
    from bit_kv_cache_int2_gb300 import oscar

    B.build()
    dev = "cuda:0"
    stream = torch.cuda.current_stream()
    if args.context:
        wl = dict(wl, L=args.context)
    Hkv, g, Bsz, L0 = wl["Hkv"], wl["g"], wl["B"], wl["L"]
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    bf16 = args.leg == "bf16"
    per_copy = (Hkv * Bsz * ((L0 - 320) * 512 + 320 * 512) + ((L0 - 320 + 63) // 64) * 4 if bf16 else
                algorithmic_bytes(L0 - 320, L0, Hkv, g) * Bsz)
    n_copies = max(2, -(-3 * l2 // per_copy))
    n_calls = args.warmup + args.steps
    appends = args.leg in ("step", "append")
    extra = max(n_calls // n_copies + 16, 80) if appends else 16
    if args.leg == "calibration":
        n_copies = 1
    wk = build_workload(wl, dev, 1 if bf16 else n_copies, extra, bf16_copies=n_copies if bf16 else 0)
    ctx, cfg, q = wk["ctx"], wk["cfg"], wk["q"]
    out = torch.empty_like(q)
    scratch = oscar.alloc_scratch(cfg, dev, prefill=args.leg == "prefill")
    if args.leg == "cuda_core":
        oscar.oscar_set_option(ctx, oscar.OPT_DECODE_IMPL, 1)
    if args.leg == "tensor_single":
        oscar.oscar_set_option(ctx, oscar.OPT_DECODE_IMPL, 2)
    if args.leg == "tcgen05":
        oscar.oscar_set_option(ctx, oscar.OPT_DECODE_IMPL, 3)
    part = {"auto": oscar.PARTITION_AUTO, "items": oscar.PARTITION_ITEMS,
            "balanced": oscar.PARTITION_BALANCED}[args.partition]
    if part != oscar.PARTITION_AUTO:
        oscar.oscar_set_option(ctx, oscar.OPT_DECODE_PARTITION, part)
    tok_bytes = Bsz * Hkv * 128 * 2
    kv_new = (wk["K"][:, :, L0:L0 + extra].permute(2, 0, 1, 3).contiguous(),
              wk["V"][:, :, L0:L0 + extra].permute(2, 0, 1, 3).contiguous())
    k_base, v_base = kv_new[0].data_ptr(), kv_new[1].data_ptr()
    cnt = [0] * n_copies
    bytes_per_call = per_copy
    if args.leg in ("decode", "cuda_core", "tensor_single", "tcgen05"):
        calls = [oscar.bind_decode(ctx, 0, c, q, out, None, scratch, Bsz) for c in wk["copies"]]
        fn = lambda i: calls[i % n_copies]()
    elif args.leg == "bf16":
        fn = lambda i: oscar.oscar_decode_bf16_history(wk["bctx"], wk["bf"][i % n_copies], q, out, None, scratch,
                                                       Bsz)
    elif args.leg in ("step", "append"):
        calls = [oscar.bind_decode_step(ctx, 0, c, q, out, None, scratch, Bsz) if args.leg == "step" else
                 oscar.bind_append(ctx, 0, c, Bsz) for c in wk["copies"]]

        def fn(i):
            c = i % n_copies
            calls[c](k_base + cnt[c] * tok_bytes, v_base + cnt[c] * tok_bytes)
            cnt[c] += 1
        if args.leg == "append":
            bytes_per_call = Bsz * Hkv * 2 * (3 * 256 + 32 + (128 // g) * 4)
    elif args.leg == "calibration":
        from bit_kv_cache_int2_gb300 import synth

        G_cal, N_cal = wl["Hq"] // Hkv, 2048
        ratios = [1.0, 0.975, 0.95, 0.925, 0.9, 0.85, 0.8, 0.7]
        cal_sets = [tuple(t.to(dev).contiguous() for t in synth.calibration_set(0, "bench", 0, h, wk["stats"][h],
                                                                                G=G_cal, n=N_cal))
                    for h in range(Hkv)]
        cscr = oscar.calibration_scratch(G_cal, N_cal, len(ratios), dev)

        def fn(i):
            h = i % Hkv
            oscar.oscar_calibrate(ctx, *cal_sets[h], N_cal, cscr)
            oscar.oscar_clip_errors(ctx, 0, h, *cal_sets[h], N_cal, ratios, cscr)
        bytes_per_call = None
    else:  # prefill
        T_pf = 64
        q_pf = torch.stack([torch.cat([synth_queries(wk["stats"][h], T_pf, wl["Hq"] // Hkv, b, h, dev)
                                       for h in range(Hkv)], dim=1) for b in range(Bsz)]).contiguous()
        k_pf = wk["K"][:, :, L0:L0 + T_pf].permute(0, 2, 1, 3).contiguous()
        v_pf = wk["V"][:, :, L0:L0 + T_pf].permute(0, 2, 1, 3).contiguous()
        out_pf = torch.empty_like(q_pf)
        fn = lambda i: oscar.oscar_prefill(ctx, 0, wk["copies"][i % n_copies], q_pf, k_pf, v_pf, T_pf, out_pf, None,
                                           scratch, Bsz)
        bytes_per_call = None
    for i in range(args.warmup):
        fn(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.warmup, n_calls):
        fn(i)
    e1.record(stream)
    torch.cuda.synchronize()
    mean_us = e0.elapsed_time(e1) * 1e3 / args.steps
    err = oscar.oscar_get_error(wk["bctx"] if bf16 else ctx)
    assert err == 0, f"device error {err}"
    line = {"leg": args.leg, "workload": args.workload, "context": L0, "partition": args.partition,
            "calls": args.steps, "mean_us": mean_us,
            "cache_copies": n_copies}
    if not appends:  # a second pass, timed call by call
        med, p10, p90 = percentiles(per_call_times(lambda i: fn(args.warmup + i), args.steps, stream))
        line.update({"median_us": med, "p10_us": p10, "p90_us": p90})
    if bytes_per_call:
        peak, kind = peaks()
        line.update({"bytes_per_call": bytes_per_call, "hbm_gbs": bytes_per_call / (mean_us * 1e-6) / 1e9,
                     "frac_of_" + kind + "_hbm": bytes_per_call / (mean_us * 1e-6) / 1e9 / peak})
    print(json.dumps(line), flush=True)


def run_batched_leg(args):
    """One batched configuration alone (--config, a BATCHED name; INT2 only):
    16 decode steps (append with demotion + attention), then --warmup untimed
    and --steps timed oscar_decode calls over cache copies larger than 3x L2.
    A short command for profiling the decode kernel at that configuration:
    the timed decode launches follow 16 + --warmup others."""
    from bit_kv_cache_int2_gb300 import build as B

    B.build()
    name = args.config
    if name not in BATCHED:
        raise SystemExit(f"--config must be one of {sorted(BATCHED)}")
    peak, kind = peaks()
    from bit_kv_cache_int2_gb300 import oscar

    part = {"auto": oscar.PARTITION_AUTO, "items": oscar.PARTITION_ITEMS,
            "balanced": oscar.PARTITION_BALANCED}[args.partition]
    r = batched_measurement("cuda:0", peak, steps=16, configs={name: dict(BATCHED[name], bf16=False)},
                            decode_warmup=args.warmup, decode_calls=args.steps, partition=part)[name]
    print(json.dumps({"leg": "batched", "config": name, "partition": args.partition, "calls": args.steps,
                      "step_us": r["step_us"], "decode_us": r["decode_us"], "bytes_per_decode": r["bytes_per_decode"],
                      "hbm_gbs": r["decode_hbm_gbs"], "frac_of_" + kind + "_hbm": r["decode_frac"],
                      "cache_copies": r["cache_copies"]}), flush=True)


def run_codebook_leg(args, wl):
    """Only the Lloyd-Max codebook decode on the workload: fits from the
    calibration sets, a cache written with them, and --steps timed decodes
    over copies larger than 3x L2.  A short command for profiling that kernel
    (the full bench reaches it after every other leg)."""
    import numpy as np
    import torch

    from bit_kv_cache_int2_gb300 import build as B
    from bit_kv_cache_int2_gb300 import oscar, synth

    B.build()
    dev = "cuda:0"
    Hkv, g, Bsz = wl["Hkv"], wl["g"], wl["B"]
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    per_copy = algorithmic_bytes(wl["L"] - 320, wl["L"], Hkv, g) * Bsz
    n_copies = max(2, -(-3 * l2 // per_copy))
    wk = build_workload(wl, dev, 1, 16)
    cfg, L0 = wk["cfg"], wl["L"]
    cctx = oscar.oscar_create(cfg)
    oscar.oscar_set_rotation(cctx, 0, wk["U"][0], wk["U"][1], [wl["clip"]] * Hkv, [wl["clip"]] * Hkv,
                             oscar.ROT_OSCAR)
    G_cal, N_cal = wl["Hq"] // Hkv, 2048
    fscr = oscar.codebook_scratch(N_cal, dev)
    kab, vab = [], []
    for h in range(Hkv):
        _, Kc, Vc = (t.to(dev).contiguous() for t in synth.calibration_set(0, "bench", 0, h, wk["stats"][h], G=G_cal,
                                                                         n=N_cal))
        kab.append(oscar.oscar_fit_codebook(cctx, 0, h, 0, Kc, N_cal, fscr)[:2])
        vab.append(oscar.oscar_fit_codebook(cctx, 0, h, 1, Vc, N_cal, fscr)[:2])
    oscar.oscar_set_codebook(cctx, 0, kab, vab)
    base = oscar.alloc_cache(cfg, dev)
    base["page_table"].copy_(wk["copies"][0]["page_table"])
    oscar.oscar_import_tokens(cctx, 0, base, wk["K"][:, :, :L0].contiguous(), wk["V"][:, :, :L0].contiguous(), Bsz,
                              L0)
    torch.cuda.synchronize()
    copies = [base] + [{k: v.clone() for k, v in base.items()} for _ in range(n_copies - 1)]
    q = wk["q"]
    out = torch.empty_like(q)
    scratch = oscar.alloc_scratch(cfg, dev)
    dec = [oscar.bind_decode(cctx, 0, c, q, out, None, scratch, Bsz) for c in copies]
    for i in range(args.warmup):
        dec[i % n_copies]()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(args.steps):
        dec[i % n_copies]()
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / args.steps
    assert oscar.oscar_get_error(cctx) == 0 and bool(torch.isfinite(out.float()).all())
    print(json.dumps({"leg": "codebook_decode", "workload": args.workload, "us_per_call": us,
                      "bytes_per_call": per_copy, "hbm_gbs": per_copy / (us * 1e-6) / 1e9, "cache_copies": n_copies,
                      "k_ab": np.round(np.array(kab), 5).tolist(), "v_ab": np.round(np.array(vab), 5).tolist()}),
          flush=True)
    oscar.oscar_destroy(cctx)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="qwen3_8b_100k", choices=sorted(WORKLOADS))
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--context", type=int, default=0,
                    help="single-operation legs: context length instead of the workload's (0: the workload's)")
    ap.add_argument("--partition", choices=["auto", "items", "balanced"], default="auto",
                    help="single-operation legs: the decode kernels' work partition (OSCAR_OPT_DECODE_PARTITION)")
    ap.add_argument("--leg", choices=["all", "codebook", "batched"] + list(LEGS), default="all",
                    help="one operation alone on the workload, a short command to profile it (see run_leg); "
                         "codebook: only the Lloyd-Max codebook decode; batched: one batched configuration "
                         "(--config)")
    ap.add_argument("--config", default="qwen3_32b_b8_131k", choices=sorted(BATCHED),
                    help="--leg batched: the batched configuration")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    wl = WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, wl)
    elif args.leg == "codebook":
        run_codebook_leg(args, wl)
    elif args.leg == "batched":
        run_batched_leg(args)
    elif args.leg in LEGS:
        run_leg(args, wl)
    else:
        run_ours(args, wl)


if __name__ == "__main__":
    main()
