"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs."""
import numpy as np
import pytest
import torch

import oracle as O
from bit_kv_cache_int2_gb300 import build as B
from bit_kv_cache_int2_gb300 import oscar

pytestmark = pytest.mark.gpu

import gpu_scenario as GS  # noqa: E402

REL_TOL = 1e-2  # max|gpu - oracle| / max|oracle| on decode outputs
LSE_TOL = 1e-2  # absolute, natural-log units


@pytest.fixture(scope="module", autouse=True)
def built():
    B.build()
    oscar.lib()


def _rel(a, b):
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-30))


# ------------------------------------------------------------ quantiser

def _hook_inputs(n, seed):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((n, 128)) * rng.uniform(0.01, 30, (n, 1))).astype(np.float32)
    x[0] = 5.0  # constant groups -> s = 0
    x[1] = np.tile(np.array([0.0, 1.0, 2.0, 3.0, 0.5, 1.5, 2.5, 3.0], np.float32), 16)  # exact levels and ties
    x[2] = np.linspace(-3e5, 3e5, 128, dtype=np.float32)  # saturated scale
    x[3] = np.linspace(-1e-7, 1e-7, 128, dtype=np.float32)  # scale rounds to 0 or an fp16 subnormal
    x[4, ::2] = 0.0
    x[4, 1::2] = 1e-3
    return x


@pytest.mark.parametrize("g", [32, 64, 128])
@pytest.mark.parametrize("clip", [1.0, 0.95, 0.9])
@pytest.mark.parametrize("which", [0, 1])
def test_quantize_hook_bit_exact(g, clip, which):
    n = 256
    x = _hook_inputs(n, seed=g + int(clip * 100) + which)
    ng = 128 // g
    xd = torch.from_numpy(x).cuda()
    codes = torch.zeros(n * 32, dtype=torch.uint8, device="cuda")
    sz = torch.zeros(n * ng * 2, dtype=torch.float16, device="cuda")
    oscar.oscar_quantize_rotated_f32(xd, g, clip, which, codes, sz)
    torch.cuda.synchronize()
    got = codes.cpu().numpy()
    gsz = sz.cpu().numpy().reshape(n, ng, 2)
    ref_codes = np.zeros((n, 128), np.uint8)
    for i in range(n):
        c, s, z = O.quantize_vector(x[i], g, clip)
        ref_codes[i] = c
        np.testing.assert_array_equal(gsz[i, :, 0].view(np.uint16), s.view(np.uint16), err_msg=f"s row {i}")
        np.testing.assert_array_equal(gsz[i, :, 1].view(np.uint16), z.view(np.uint16), err_msg=f"z row {i}")
    if which == 0:
        ref = np.concatenate([O.pack_k_row(r) for r in ref_codes])
    else:
        ref = np.concatenate([O.pack_v_block(ref_codes[64 * k:64 * (k + 1)]) for k in range(n // 64)])
    np.testing.assert_array_equal(got, ref)


def test_debug_rotate_matches_oracle():
    sc = GS.build("rot", [0], Hq=4, Hkv=2, calib_n=512)
    try:
        x = torch.randn(37, 128, device="cuda").to(torch.bfloat16) * 5
        y = torch.empty(37, 128, device="cuda")
        for which, U in ((0, sc.U_K), (1, sc.U_V)):
            for h in range(2):
                oscar.oscar_debug_rotate(sc.ctx, 0, which, h, x, y)
                torch.cuda.synchronize()
                ref = x.float().cpu().numpy().astype(np.float64) @ O.rotation(U[h], O.ROT_OSCAR)
                assert np.abs(y.cpu().numpy() - ref).max() <= 1e-5 * np.abs(ref).max()
    finally:
        sc.close()


# --------------------------------------------------------------- cfg 1

def test_cfg1_import_append_demote_and_decode():
    """Tiny single layer: B1, 1 kv head, GQA 4, 1024 tokens = 64 sink + 704
    history + 256 recent, shuffled pages, g128, clip 0.95; the last 64 tokens
    arrive by append, each demoting one token."""
    sc = GS.build("cfg1", [960], Hq=4, Hkv=1, g=128, extra_tokens=64)
    try:
        for t in range(960, 1024):
            k = sc.K[0][:, t].unsqueeze(0).contiguous()
            v = sc.V[0][:, t].unsqueeze(0).contiguous()
            oscar.oscar_append(sc.ctx, 0, sc.cache, k, v, 1)
        torch.cuda.synchronize()
        assert oscar.oscar_get_error(sc.ctx) == 0
        hc = GS.HostCache(sc)
        assert (int(hc.seq[0]), int(hc.hist[0])) == (1024, 704)
        # windows are exact copies
        kall = sc.K[0].float().cpu().numpy()
        vall = sc.V[0].float().cpu().numpy()
        wk, wv = hc.window(0, 0)
        pos = list(range(64)) + list(range(768, 1024))
        np.testing.assert_array_equal(wk, kall[0, pos])
        np.testing.assert_array_equal(wv, vall[0, pos])
        # history codes vs the oracle's quantisation of the same tokens
        n, bad = GS.compare_history(sc, hc, 0, 0, list(range(64, 768)), list(range(704)))
        assert bad <= 1e-4 * n
        q = GS.queries(sc, seed=1)
        qn = q.float().cpu().numpy()
        for impl in (oscar.DECODE_TENSOR, oscar.DECODE_CUDA_CORE, oscar.DECODE_TENSOR_SINGLE, oscar.DECODE_TCGEN05):
            out, lse = GS.decode(sc, q, impl)
            ref, rlse = GS.oracle_decode(sc, hc, qn, 0)
            assert _rel(out[0].float().cpu().numpy(), ref) <= REL_TOL
            assert np.abs(lse[0].cpu().numpy() - rlse).max() <= LSE_TOL
    finally:
        sc.close()


# ----------------------------------------------------- lengths and shapes

EDGE_LENGTHS = [0, 1, 2, 63, 64, 65, 100, 319, 320, 321, 383, 384, 385, 447, 448, 449, 700, 1024, 1100]


@pytest.mark.parametrize("part", [oscar.PARTITION_ITEMS, oscar.PARTITION_BALANCED])
@pytest.mark.parametrize("impl", [0, 1, 2, 3])
def test_decode_edge_lengths_gqa4_g128(impl, part):
    sc = GS.build("edge", EDGE_LENGTHS, Hq=8, Hkv=2, g=128, interleave=True, calib_n=512)
    try:
        oscar.oscar_set_option(sc.ctx, oscar.OPT_DECODE_PARTITION, part)
        q = GS.queries(sc, seed=2)
        out, lse = GS.decode(sc, q, impl)
        assert oscar.oscar_get_error(sc.ctx) == 0
        hc = GS.HostCache(sc)
        qn = q.float().cpu().numpy()
        for b, L in enumerate(EDGE_LENGTHS):
            got = out[b].float().cpu().numpy()
            if L == 0:
                assert np.all(got == 0) and np.all(np.isneginf(lse[b].cpu().numpy()))
                continue
            ref, rlse = GS.oracle_decode(sc, hc, qn, b)
            assert _rel(got, ref) <= REL_TOL, (L, _rel(got, ref))
            assert np.abs(lse[b].cpu().numpy() - rlse).max() <= LSE_TOL, L
    finally:
        sc.close()


@pytest.mark.parametrize("part", [oscar.PARTITION_ITEMS, oscar.PARTITION_BALANCED])
@pytest.mark.parametrize("G,g", [(1, 32), (2, 64), (8, 32), (8, 128), (4, 64), (1, 128)])
@pytest.mark.parametrize("impl", [0, 1, 2, 3])
def test_decode_gqa_and_group_sizes(G, g, impl, part):
    lengths = [333, 1000, 64 * 9 + 320 + 17]
    sc = GS.build(f"gq{G}{g}", lengths, Hq=2 * G, Hkv=2, g=g, calib_n=512)
    try:
        oscar.oscar_set_option(sc.ctx, oscar.OPT_DECODE_PARTITION, part)
        q = GS.queries(sc, seed=3)
        out, lse = GS.decode(sc, q, impl)
        hc = GS.HostCache(sc)
        qn = q.float().cpu().numpy()
        for b in range(len(lengths)):
            ref, rlse = GS.oracle_decode(sc, hc, qn, b)
            assert _rel(out[b].float().cpu().numpy(), ref) <= REL_TOL, (b, _rel(out[b].float().cpu().numpy(), ref))
            assert np.abs(lse[b].cpu().numpy() - rlse).max() <= LSE_TOL
        n, bad = GS.compare_history(sc, hc, 1, 1, list(range(64, 64 + 680)), list(range(680)))
        assert bad <= 1e-4 * n
    finally:
        sc.close()


@pytest.mark.parametrize("items", [0, 1, 3, 8, -1])
def test_decode_item_sizing_options(items):
    """The work list's item sizing (0 = automatic, else fixed items per CTA)
    changes only how the history is split: every setting matches the oracle
    on a ragged batch long enough for the automatic rule to split finely.
    items < 0: the balanced partition instead of the item list."""
    # ~21K history pages x kv heads: past the automatic rule's single-wave limit
    lengths = [9000, 320, 140000, 62345, 0, 700, 125000, 64 * 50 + 320 + 3]
    sc = GS.build("items", lengths, Hq=16, Hkv=4, g=128, interleave=True, calib_n=512)
    try:
        if items < 0:
            oscar.oscar_set_option(sc.ctx, oscar.OPT_DECODE_PARTITION, oscar.PARTITION_BALANCED)
        else:
            oscar.oscar_set_option(sc.ctx, oscar.OPT_DECODE_PARTITION, oscar.PARTITION_ITEMS)
            oscar.oscar_set_option(sc.ctx, oscar.OPT_ITEMS_PER_CTA, items)
        q = GS.queries(sc, seed=8)
        out, lse = GS.decode(sc, q)
        assert oscar.oscar_get_error(sc.ctx) == 0
        hc = GS.HostCache(sc)
        qn = q.float().cpu().numpy()
        for b, L in enumerate(lengths):
            if L == 0:
                assert np.all(out[b].float().cpu().numpy() == 0)
                continue
            ref, rlse = GS.oracle_decode(sc, hc, qn, b)
            assert _rel(out[b].float().cpu().numpy(), ref) <= REL_TOL, (items, b)
            assert np.abs(lse[b].cpu().numpy() - rlse).max() <= LSE_TOL
    finally:
        sc.close()


@pytest.mark.parametrize("part", [oscar.PARTITION_ITEMS, oscar.PARTITION_BALANCED])
def test_bf16_history_baseline_matches_dense_attention(part):
    lengths = [1, 300, 321, 1000, 2000]
    sc = GS.build("bf16h", lengths, Hq=8, Hkv=2, bf16_history=True, mode=oscar.ROT_NONE)
    try:
        oscar.oscar_set_option(sc.ctx, oscar.OPT_DECODE_PARTITION, part)
        q = GS.queries(sc, seed=4)
        out, lse = GS.decode(sc, q)
        hc = GS.HostCache(sc)
        qn = q.float().cpu().numpy()
        G = 4
        for b, L in enumerate(lengths):
            ref, rlse = GS.oracle_decode(sc, hc, qn, b)
            # the BF16 history holds the original tokens: plain dense attention
            kall = sc.K[b].float().cpu().numpy()
            vall = sc.V[b].float().cpu().numpy()
            for h in range(2):
                dense, _ = O.softmax_attention(qn[b, h * G:(h + 1) * G], kall[h, :L], vall[h, :L])
                np.testing.assert_allclose(ref[h * G:(h + 1) * G], dense, atol=1e-9)
            assert _rel(out[b].float().cpu().numpy(), ref) <= REL_TOL
            assert np.abs(lse[b].cpu().numpy() - rlse).max() <= LSE_TOL
    finally:
        sc.close()


# -------------------------------------------------- appends, demotes, wrap

def test_append_stream_wraps_ring_and_matches_oracle():
    """300 -> 700 tokens by appends (the ring wraps), with decodes on the way."""
    sc = GS.build("stream", [300, 64], Hq=4, Hkv=2, g=64, extra_tokens=400, calib_n=512)
    try:
        qn_all = []
        checks = {301, 320, 321, 384, 577, 700}
        for t in range(400):
            k = torch.stack([sc.K[b][:, [300, 64][b] + t] for b in range(2)]).contiguous()
            v = torch.stack([sc.V[b][:, [300, 64][b] + t] for b in range(2)]).contiguous()
            oscar.oscar_append(sc.ctx, 0, sc.cache, k, v, 2)
            L0 = 301 + t
            if L0 in checks:
                q = GS.queries(sc, seed=100 + t)
                out, lse = GS.decode(sc, q)
                hc = GS.HostCache(sc)
                assert int(hc.seq[0]) == L0 and int(hc.seq[1]) == 65 + t
                qn = q.float().cpu().numpy()
                for b in range(2):
                    ref, _ = GS.oracle_decode(sc, hc, qn, b)
                    assert _rel(out[b].float().cpu().numpy(), ref) <= REL_TOL, (L0, b)
        assert oscar.oscar_get_error(sc.ctx) == 0
        hc = GS.HostCache(sc)
        H0 = int(hc.hist[0])
        assert H0 == 700 - 320
        n, bad = GS.compare_history(sc, hc, 0, 1, list(range(64, 64 + H0)), list(range(H0)))
        assert bad <= 1e-4 * n
    finally:
        sc.close()


@pytest.mark.parametrize("part", [oscar.PARTITION_ITEMS, oscar.PARTITION_BALANCED])
def test_decode_step_equals_append_then_decode(part):
    """oscar_decode_step (append and query rotation in one kernel) gives the
    same cache and the same outputs, bit for bit, as oscar_append followed by
    oscar_decode, across ring wrap and demotions; the outputs match the oracle."""
    lengths = [300, 64, 1500]
    scs = [GS.build("stepx", lengths, Hq=8, Hkv=2, g=128, extra_tokens=120, calib_n=512) for _ in range(2)]
    try:
        a, b = scs
        for s_ in scs:
            oscar.oscar_set_option(s_.ctx, oscar.OPT_DECODE_PARTITION, part)
        scratch = [oscar.alloc_scratch(s_.cfg) for s_ in scs]
        for t in range(120):
            k = torch.stack([a.K[i][:, lengths[i] + t] for i in range(3)]).contiguous()
            v = torch.stack([a.V[i][:, lengths[i] + t] for i in range(3)]).contiguous()
            q = GS.queries(a, seed=300 + t)
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
            assert torch.equal(outs[0][1], outs[1][1]), t
        for s_ in scs:
            assert oscar.oscar_get_error(s_.ctx) == 0
        for key in ("pool", "sink_k", "sink_v", "ring_k", "ring_v", "seq_lens", "hist_lens"):
            assert torch.equal(a.cache[key], b.cache[key]), key
        hc = GS.HostCache(a)
        qn = q.float().cpu().numpy()
        for i in range(3):
            ref, rlse = GS.oracle_decode(a, hc, qn, i)
            assert _rel(outs[0][0][i].float().cpu().numpy(), ref) <= REL_TOL, i
    finally:
        for s_ in scs:
            s_.close()


def test_decode_step_with_pinned_host_operands():
    """k_new, v_new, q, out and lse in pinned host memory, read and written by
    the kernels in place, give the same cache and results, bit for bit, as
    device buffers."""
    lengths = [300, 1500]
    scs = [GS.build("pinned", lengths, Hq=8, Hkv=2, g=128, extra_tokens=20, calib_n=512) for _ in range(2)]
    try:
        scratch = [oscar.alloc_scratch(s_.cfg) for s_ in scs]
        for t in range(20):
            k = torch.stack([scs[0].K[i][:, lengths[i] + t] for i in range(2)]).contiguous()
            v = torch.stack([scs[0].V[i][:, lengths[i] + t] for i in range(2)]).contiguous()
            q = GS.queries(scs[0], seed=500 + t)
            out_d = torch.empty_like(q)
            lse_d = torch.empty(2, 8, dtype=torch.float32, device="cuda")
            oscar.oscar_decode_step(scs[0].ctx, 0, scs[0].cache, k, v, q, out_d, lse_d, scratch[0], 2)
            kh, vh, qh = (x.cpu().pin_memory() for x in (k, v, q))
            out_h = torch.empty(q.shape, dtype=q.dtype).pin_memory()
            lse_h = torch.empty(2, 8, dtype=torch.float32).pin_memory()
            oscar.oscar_decode_step(scs[1].ctx, 0, scs[1].cache, kh, vh, qh, out_h, lse_h, scratch[1], 2)
            torch.cuda.synchronize()
            assert torch.equal(out_d.cpu(), out_h), t
            assert torch.equal(lse_d.cpu(), lse_h), t
        for s_ in scs:
            assert oscar.oscar_get_error(s_.ctx) == 0
        for key in ("pool", "sink_k", "sink_v", "ring_k", "ring_v", "seq_lens", "hist_lens"):
            assert torch.equal(scs[0].cache[key], scs[1].cache[key]), key
    finally:
        for s_ in scs:
            s_.close()


def test_demote_then_append():
    sc = GS.build("demote", [400], Hq=4, Hkv=1, g=128, extra_tokens=10, calib_n=512)
    try:
        for _ in range(3):
            oscar.oscar_demote(sc.ctx, 0, sc.cache, 1)
        torch.cuda.synchronize()
        hc = GS.HostCache(sc)
        assert (int(hc.seq[0]), int(hc.hist[0])) == (400, 83)
        for t in range(5):
            k = sc.K[0][:, 400 + t].unsqueeze(0).contiguous()
            v = sc.V[0][:, 400 + t].unsqueeze(0).contiguous()
            oscar.oscar_append(sc.ctx, 0, sc.cache, k, v, 1)
        q = GS.queries(sc, seed=5)
        out, _ = GS.decode(sc, q)
        hc = GS.HostCache(sc)
        # window 253 -> 256 after 3 appends, then two appends each demote one
        assert (int(hc.seq[0]), int(hc.hist[0])) == (405, 85)
        ref, _ = GS.oracle_decode(sc, hc, q.float().cpu().numpy(), 0)
        assert _rel(out[0].float().cpu().numpy(), ref) <= REL_TOL
        n, bad = GS.compare_history(sc, hc, 0, 0, list(range(64, 64 + 85)), list(range(85)))
        assert bad <= 1e-4 * n
    finally:
        sc.close()


def test_rotation_modes_decode():
    for mode in (oscar.ROT_HADAMARD, oscar.ROT_NONE):
        sc = GS.build(f"mode{mode}", [900], Hq=4, Hkv=1, mode=mode)
        try:
            q = GS.queries(sc, seed=6)
            out, _ = GS.decode(sc, q)
            hc = GS.HostCache(sc)
            ref, _ = GS.oracle_decode(sc, hc, q.float().cpu().numpy(), 0)
            assert _rel(out[0].float().cpu().numpy(), ref) <= REL_TOL
            n, bad = GS.compare_history(sc, hc, 0, 0, list(range(64, 64 + 580)), list(range(580)))
            assert bad <= 1e-4 * n
        finally:
            sc.close()


# ------------------------------------------------------------- errors

def test_missing_page_is_reported_not_faulted():
    sc = GS.build("err", [500], Hq=4, Hkv=1, extra_tokens=70)
    try:
        hc = GS.HostCache(sc)
        H = int(hc.hist[0])
        pt = sc.cache["page_table"]
        saved = pt.clone()
        # the next demotion writes history slot H: take its page away
        pt[0, H // 64] = -1
        k = sc.K[0][:, 500].unsqueeze(0).contiguous()
        v = sc.V[0][:, 500].unsqueeze(0).contiguous()
        oscar.oscar_append(sc.ctx, 0, sc.cache, k, v, 1)
        assert oscar.oscar_get_error(sc.ctx) == oscar.ERR_NO_PAGE
        assert int(sc.cache["seq_lens"][0]) == 500  # request left unchanged
        pt.copy_(saved)
        # decode over a history whose page is missing: error word, no fault
        pt[0, 0] = -1
        q = GS.queries(sc, seed=7)
        GS.decode(sc, q)
        assert oscar.oscar_get_error(sc.ctx) == oscar.ERR_NO_PAGE
        pt[0, 0] = 10 ** 6
        GS.decode(sc, q)
        assert oscar.oscar_get_error(sc.ctx) == oscar.ERR_RANGE
        pt.copy_(saved)
        GS.decode(sc, q)
        assert oscar.oscar_get_error(sc.ctx) == 0
    finally:
        sc.close()


def test_import_into_nonempty_request_is_a_state_error():
    sc = GS.build("state", [400], Hq=4, Hkv=1)
    try:
        k = sc.K[0][:, :10].unsqueeze(0).contiguous()
        oscar.oscar_import_tokens(sc.ctx, 0, sc.cache, k, k, 1, 10)
        assert oscar.oscar_get_error(sc.ctx) == oscar.ERR_STATE
        assert int(sc.cache["seq_lens"][0]) == 400
    finally:
        sc.close()


def test_wait_timeout_is_reported_and_recoverable():
    """A page wait that runs out of its budget (OSCAR_OPT_WAIT_POLLS = 0: every
    first wait gives up at once) is reported as OSCAR_ERR_TIMEOUT by each
    decode kernel; the kernel drains its copies and returns, and with the
    default budget the next decode matches the oracle."""
    sc = GS.build("tmo", [5000, 1000], Hq=8, Hkv=2, g=128, calib_n=512)
    try:
        q = GS.queries(sc, seed=9)
        oscar.oscar_set_option(sc.ctx, oscar.OPT_WAIT_POLLS, 0)
        for impl in (oscar.DECODE_TENSOR, oscar.DECODE_TENSOR_SINGLE, oscar.DECODE_CUDA_CORE):
            GS.decode(sc, q, impl)
            assert oscar.oscar_get_error(sc.ctx) == oscar.ERR_TIMEOUT, impl
        with pytest.raises(oscar.OscarError):
            oscar.oscar_set_option(sc.ctx, oscar.OPT_WAIT_POLLS, -1)
        oscar.oscar_set_option(sc.ctx, oscar.OPT_WAIT_POLLS, oscar.WAIT_POLLS_DEFAULT)
        out, lse = GS.decode(sc, q, oscar.DECODE_TENSOR)
        assert oscar.oscar_get_error(sc.ctx) == 0
        hc = GS.HostCache(sc)
        qn = q.float().cpu().numpy()
        for b in range(2):
            ref, rlse = GS.oracle_decode(sc, hc, qn, b)
            assert _rel(out[b].float().cpu().numpy(), ref) <= REL_TOL
            assert np.abs(lse[b].cpu().numpy() - rlse).max() <= LSE_TOL
    finally:
        sc.close()
