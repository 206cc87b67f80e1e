"""Builds seeded caches through the C ABI and computes what the oracle says
about them.  Used by the GPU parity tests, smoke() and bench.py's checks."""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

import oracle as O
from bit_kv_cache_int2_gb300 import oscar, synth


@dataclasses.dataclass
class Scenario:
    cfg: object
    ctx: object
    cache: dict
    lengths: list
    Hq: int
    Hkv: int
    g: int
    U_K: np.ndarray  # [Hkv][128][128] float32
    U_V: np.ndarray
    clip_k: float
    clip_v: float
    mode: int
    K: list  # per request: bf16 tensor [Hkv][n][128] on the device (all tokens ever written)
    V: list
    stats: list  # per kv head HeadStats
    bf16_history: bool = False
    codebook: tuple = None  # (k_ab, v_ab), each [Hkv][2] (a, b), or None (uniform levels)

    def cb(self, which, h):
        """(a, b) of kv head h for "k" or "v", None for the uniform quantiser."""
        if self.codebook is None:
            return None
        ab = self.codebook[0 if which == "k" else 1]
        return None if ab is None else (float(np.float32(ab[h][0])), float(np.float32(ab[h][1])))

    @property
    def B(self):
        return len(self.lengths)

    def close(self):
        if self.ctx is not None:
            oscar.oscar_destroy(self.ctx)
            self.ctx = None


def request_view(cache: dict, b: int) -> dict:
    """Cache dict whose per-request arrays start at request b (same pool)."""
    v = dict(cache)
    for k in ("page_table", "sink_k", "sink_v", "ring_k", "ring_v", "seq_lens", "hist_lens"):
        v[k] = cache[k][b:b + 1]
    return v


def calibrate_heads(base, wl, layer, Hkv, G, stats, calib_n=2048):
    UK, UV = [], []
    for h in range(Hkv):
        Qc, Kc, Vc = synth.calibration_set(base, wl, layer, h, stats[h], G=G, n=calib_n)
        uq, us = O.calibrate(Qc.float().numpy(), Kc.float().numpy(), Vc.float().numpy())
        UK.append(uq.astype(np.float32))
        UV.append(us.astype(np.float32))
    return np.stack(UK), np.stack(UV)


def build(wl: str, lengths, Hq=4, Hkv=1, g=128, clip_k=0.95, clip_v=0.95, n_out=4, f_key=20.0,
          seed=0, interleave=False, mode=oscar.ROT_OSCAR, extra_tokens=0, calib_n=2048,
          bf16_history=False, device="cuda", spare_pages=2, U=None, codebook=None) -> Scenario:
    """Import every request's prefix (lengths[b] tokens) into a fresh cache.

    extra_tokens: how many more tokens per request to draw (for later appends)."""
    B = len(lengths)
    G = Hq // Hkv
    hist = [max(L - 320, 0) for L in lengths]
    max_hist = [max(L + extra_tokens - 320, 0) for L in lengths]
    pages_per_req = [(h + 63) // 64 for h in max_hist]
    mpr = max(1, max(pages_per_req))
    num_pages = max(1, sum(pages_per_req) + spare_pages)
    cfg = oscar.make_config(1, Hq, Hkv, g, max_batch=B, max_pages_per_req=mpr, num_pages=num_pages)
    ctx = oscar.oscar_create(cfg)
    stats = [synth.head_stats(seed, wl, 0, h, n_out=n_out, f_key=f_key) for h in range(Hkv)]
    if U is None:
        if mode == oscar.ROT_OSCAR:
            U_K, U_V = calibrate_heads(seed, wl, 0, Hkv, G, stats, calib_n)
        else:
            U_K = U_V = np.stack([np.eye(128, dtype=np.float32)] * Hkv)
    else:
        U_K, U_V = U
    oscar.oscar_set_rotation(ctx, 0, U_K, U_V, [clip_k] * Hkv, [clip_v] * Hkv, mode)
    if codebook is not None:
        oscar.oscar_set_codebook(ctx, 0, codebook[0], codebook[1])
    cache = oscar.alloc_cache(cfg, device, bf16_history=bf16_history)
    pt = synth.page_table(num_pages, pages_per_req, synth.stream_seed(seed, wl, "pages"), interleave, mpr)
    cache["page_table"].copy_(pt.to(device))
    Ks, Vs = [], []
    for b, L in enumerate(lengths):
        n_all = L + extra_tokens
        k = torch.stack([synth.draw_keys(stats[h], n_all, synth.stream_seed(seed, wl, b, h, "K"), device)
                         for h in range(Hkv)])
        v = torch.stack([synth.draw_values(stats[h], n_all, synth.stream_seed(seed, wl, b, h, "V"), device)
                         for h in range(Hkv)])
        Ks.append(k)
        Vs.append(v)
        if L > 0:
            view = request_view(cache, b)
            kin = k[:, :L].unsqueeze(0).contiguous()
            vin = v[:, :L].unsqueeze(0).contiguous()
            if bf16_history:
                oscar.oscar_import_bf16_history(ctx, view, kin, vin, 1, L)
            else:
                oscar.oscar_import_tokens(ctx, 0, view, kin, vin, 1, L)
    torch.cuda.synchronize()
    return Scenario(cfg, ctx, cache, list(lengths), Hq, Hkv, g, U_K, U_V, clip_k, clip_v, mode, Ks, Vs,
                    stats, bf16_history, codebook)


def queries(sc: Scenario, seed=0, tag="Q"):
    G = sc.Hq // sc.Hkv
    qs = []
    for b in range(sc.B):
        rows = [synth.draw_queries(sc.stats[h], G, synth.stream_seed(seed, tag, b, h), "cuda")
                for h in range(sc.Hkv)]
        qs.append(torch.cat(rows))
    return torch.stack(qs).contiguous()  # [B][Hq][128]


def decode(sc: Scenario, q, impl=0):
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[0], q.shape[1], dtype=torch.float32, device=q.device)
    scratch = oscar.alloc_scratch(sc.cfg)
    oscar.oscar_set_option(sc.ctx, oscar.OPT_DECODE_IMPL, impl)
    if sc.bf16_history:
        oscar.oscar_decode_bf16_history(sc.ctx, sc.cache, q, out, lse, scratch, sc.B)
    else:
        oscar.oscar_decode(sc.ctx, 0, sc.cache, q, out, lse, scratch, sc.B)
    torch.cuda.synchronize()
    return out, lse


class HostCache:
    """A host copy of the cache buffers, for the oracle."""

    def __init__(self, sc: Scenario):
        c = sc.cache
        self.pool = c["pool"].cpu().numpy()
        self.pt = c["page_table"].cpu().numpy()
        self.sink_k = c["sink_k"].float().cpu().numpy()
        self.sink_v = c["sink_v"].float().cpu().numpy()
        self.ring_k = c["ring_k"].float().cpu().numpy()
        self.ring_v = c["ring_v"].float().cpu().numpy()
        self.seq = c["seq_lens"].cpu().numpy()
        self.hist = c["hist_lens"].cpu().numpy()
        info = oscar.oscar_layout(sc.cfg)
        self.head_bytes = info.bf16_head_bytes if sc.bf16_history else info.int2_head_bytes
        self.page_bytes = self.head_bytes * sc.Hkv

    def head_blocks(self, b, h, H):
        pages = (H + 63) // 64
        ids = self.pt[b, :pages]
        assert (ids >= 0).all()
        offs = ids.astype(np.int64) * self.page_bytes + h * self.head_bytes
        return np.stack([self.pool[o:o + self.head_bytes] for o in offs]) if pages else None

    def window(self, b, h):
        L, H = int(self.seq[b]), int(self.hist[b])
        ks = [self.sink_k[b, h, :min(L, 64)]]
        vs = [self.sink_v[b, h, :min(L, 64)]]
        slots = [(p - 64) % 256 for p in range(64 + H, L)]
        ks.append(self.ring_k[b, h, slots])
        vs.append(self.ring_v[b, h, slots])
        return np.concatenate(ks), np.concatenate(vs)

    def history_int2(self, b, h, g):
        H = int(self.hist[b])
        if H == 0:
            return None
        f = O.parse_head_block(self.head_blocks(b, h, H), g)
        return {k: v.reshape((-1,) + v.shape[2:])[:H] for k, v in f.items()}

    def history_bf16(self, b, h):
        H = int(self.hist[b])
        if H == 0:
            return np.zeros((0, 128)), np.zeros((0, 128))
        blk = self.head_blocks(b, h, H)
        k = blk[:, :16384].copy().view(np.uint16).reshape(-1, 128)[:H]
        v = blk[:, 16384:].copy().view(np.uint16).reshape(-1, 128)[:H]
        to_f = lambda a: (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        return to_f(k), to_f(v)


def oracle_decode(sc: Scenario, hc: HostCache, q_np, b):
    """Oracle output [Hq][128] and lse [Hq] of request b on the GPU's own cache contents."""
    G = sc.Hq // sc.Hkv
    outs, lses = [], []
    for h in range(sc.Hkv):
        wk, wv = hc.window(b, h)
        qg = q_np[b, h * G:(h + 1) * G]
        if sc.bf16_history:
            hk, hv = hc.history_bf16(b, h)
            R = np.eye(128)
            o, l = O.three_region_attention(qg, wk, wv, hk, hv, R, R)
        else:
            f = hc.history_int2(b, h, sc.g)
            if f is None:
                hk = hv = np.zeros((0, 128))
            else:
                cbf = getattr(sc, "cb", None)  # views without codebooks use the uniform levels
                ck, cv = (cbf("k", h), cbf("v", h)) if cbf else (None, None)
                hk = (O.dequantize(f["k_codes"], f["k_s"], f["k_z"], sc.g) if ck is None
                      else O.dequantize_codebook(f["k_codes"], f["k_s"], f["k_z"], sc.g, *ck))
                hv = (O.dequantize(f["v_codes"], f["v_s"], f["v_z"], sc.g) if cv is None
                      else O.dequantize_codebook(f["v_codes"], f["v_s"], f["v_z"], sc.g, *cv))
            o, l = O.three_region_attention(qg, wk, wv, hk, hv, O.rotation(sc.U_K[h], sc.mode),
                                            O.rotation(sc.U_V[h], sc.mode))
        outs.append(o)
        lses.append(l)
    return np.concatenate(outs), np.concatenate(lses)


def expected_codes(sc: Scenario, b, h, positions, which):
    """Oracle quantisation of the tokens at absolute positions (fp64 rotation -> fp32)."""
    src = (sc.K if which == "k" else sc.V)[b][h][positions].float().cpu().numpy()
    U = (sc.U_K if which == "k" else sc.U_V)[h]
    clip = sc.clip_k if which == "k" else sc.clip_v
    R = O.rotation(U, sc.mode)
    xr = O.rotate_to_f32(src, R)
    codes = np.zeros(xr.shape, dtype=np.uint8)
    ng = 128 // sc.g
    s = np.zeros((len(positions), ng), dtype=np.float16)
    z = np.zeros((len(positions), ng), dtype=np.float16)
    cb = sc.cb(which, h)
    for i in range(len(positions)):
        if cb is None:
            codes[i], s[i], z[i] = O.quantize_vector(xr[i], sc.g, clip)
        else:
            codes[i], s[i], z[i] = O.quantize_vector_codebook(xr[i], sc.g, clip, *cb)
    return xr, codes, s, z


def compare_history(sc: Scenario, hc: HostCache, b, h, positions, hist_slots):
    """Checks GPU history codes/scales against the oracle's quantisation of the
    same tokens.  Returns (n_codes, n_mismatch); raises on an unexplained one."""
    f = hc.history_int2(b, h, sc.g)
    n_codes = 0
    n_bad = 0
    for which in ("k", "v"):
        cb = sc.cb(which, h)
        xr, codes, s, z = expected_codes(sc, b, h, positions, which)
        gc = f[which + "_codes"][hist_slots]
        gs = f[which + "_s"][hist_slots]
        gz = f[which + "_z"][hist_slots]
        # s within one fp16 ulp; z within one fp16 ulp taken at the group's
        # scale (the GPU rotates in fp32, so its quantiser inputs differ from the
        # oracle's by an absolute ~1e-7 of the vector norm; a zero point close to
        # 0 can then move by more than one of its own ulps, never by more than
        # one ulp of the group's scale).
        def ulp16(x):
            x = np.maximum(np.abs(np.asarray(x, np.float64)), 2.0 ** -14)
            return 2.0 ** (np.floor(np.log2(x)) - 10)

        ai = gs.view(np.int16).astype(np.int32)
        ei = s.view(np.int16).astype(np.int32)
        ok_s = (np.abs(ai - ei) <= 1) & ((np.sign(gs.astype(np.float32)) == np.sign(s.astype(np.float32))) | (gs == s))
        sf = s.astype(np.float64)
        ok_z = np.abs(gz.astype(np.float64) - z.astype(np.float64)) <= ulp16(np.maximum(np.abs(z.astype(np.float64)), sf))
        for name, ok, a, e in (("scale", ok_s, gs, s), ("zero", ok_z, gz, z)):
            if not ok.all():
                info = []
                for (i, gr) in np.argwhere(~ok)[:5]:
                    grp = xr[i, gr * sc.g:(gr + 1) * sc.g]
                    info.append((int(i), int(gr), float(a[i, gr]), float(e[i, gr]), float(grp.min()), float(grp.max())))
                raise AssertionError(f"{which} {name} off by more than 1 ulp: (row, group, gpu, oracle, min, max) {info}")
        bad = np.argwhere(gc != codes)
        n_codes += codes.size
        n_bad += len(bad)
        for (i, c) in bad:
            gr = c // sc.g
            if gs[i, gr] != s[i, gr] or gz[i, gr] != z[i, gr]:
                continue  # explained by its group's scale / zero differing by an ulp
            sf, zf = np.float32(s[i, gr]), np.float32(z[i, gr])
            t = (float(xr[i, c]) - float(zf)) / float(sf)
            if cb is None:
                frac = t - np.floor(t)
                assert abs(frac - 0.5) < 1e-4 or abs(t - 3.5) < 1e-4, (which, i, c, t, gc[i, c], codes[i, c])
            else:  # next to one of the codebook's thresholds
                lo, hi = O.codebook_thresholds(*cb)
                assert min(abs(t - float(lo)), abs(t - 1.5), abs(t - float(hi))) < 1e-4, (which, i, c, t)
    return n_codes, n_bad
