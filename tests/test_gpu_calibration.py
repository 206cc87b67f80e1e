"""GPU parity of the offline calibration (oscar_calibrate, oscar_clip_errors)
against the oracle, through the C ABI: the covariances C_Q and C_S, their
eigenbases (up to what the eigengaps determine), and the clip errors of every
candidate ratio with the argmin they give."""
import numpy as np
import pytest
import torch

import oracle as O
from bit_kv_cache_int2_gb300 import build as B
from bit_kv_cache_int2_gb300 import oscar, synth

pytestmark = pytest.mark.gpu

COV_TOL = 1e-4    # max|gpu - oracle| / max|oracle| for C_Q, C_S (fp32 sums, fp32 attention)
ERR_TOL = 2e-3    # relative, clip errors (fp32 rotation and attention on the GPU)
RATIOS = [1.0, 0.95, 0.9, 0.85, 0.8, 0.7]


@pytest.fixture(scope="module", autouse=True)
def built():
    B.build()
    oscar.lib()


def calib_inputs(G, N, seed, n_out=4, f_key=20.0):
    st = synth.head_stats(seed, "calibtest", 0, 0, n_out=n_out, f_key=f_key)
    Q, K, V = synth.calibration_set(seed, "calibtest", 0, 0, st, G=G, n=N)
    return Q.cuda().contiguous(), K.cuda().contiguous(), V.cuda().contiguous()


def make_ctx(G, g=128):
    cfg = oscar.make_config(1, 4 * G, 4, g, max_batch=1, max_pages_per_req=1, num_pages=1)
    return cfg, oscar.oscar_create(cfg)


def check_basis(U_gpu, C_oracle):
    """U orthonormal; every column whose eigenvalue is separated from its
    neighbours (relative gap > 1e-3) equals the oracle's eigenvector, same sign."""
    U_o = O.eigenbasis(C_oracle)
    w = np.sort(np.linalg.eigvalsh(C_oracle))[::-1]
    U = U_gpu.astype(np.float64)
    assert np.abs(U.T @ U - np.eye(128)).max() < 1e-5
    scale = max(abs(w[0]), 1e-300)
    checked = 0
    for i in range(128):
        gap = min(abs(w[i] - w[i - 1]) if i > 0 else np.inf, abs(w[i] - w[i + 1]) if i < 127 else np.inf)
        if gap / scale > 1e-3:
            assert float(U[:, i] @ U_o[:, i]) > 1 - 1e-4, i
            checked += 1
    return checked


@pytest.mark.parametrize("G,N", [(4, 384), (2, 257), (8, 128)])
def test_calibrate_matches_oracle(G, N):
    cfg, ctx = make_ctx(G)
    try:
        Q, K, V = calib_inputs(G, N, seed=G * 1000 + N)
        scratch = oscar.calibration_scratch(G, N)
        U_K, U_V, C_Q, C_S = oscar.oscar_calibrate(ctx, Q, K, V, N, scratch)
        Qn, Kn, Vn = (t.float().cpu().numpy() for t in (Q, K, V))
        CQ_o = O.query_covariance(Qn)
        CS_o = O.score_weighted_value_covariance(Qn, Kn, Vn)
        assert np.abs(C_Q - CQ_o).max() / np.abs(CQ_o).max() < COV_TOL
        assert np.abs(C_S - CS_o).max() / np.abs(CS_o).max() < COV_TOL
        nk = check_basis(U_K, CQ_o)
        nv = check_basis(U_V, CS_o)
        assert nk >= 8 and nv >= 8  # the leading, well-separated directions at least
        print(f"G={G} N={N}: {nk} key and {nv} value eigenvectors compared")
    finally:
        oscar.oscar_destroy(ctx)


@pytest.mark.parametrize("g,mode", [(128, oscar.ROT_OSCAR), (32, oscar.ROT_HADAMARD), (64, oscar.ROT_NONE)])
def test_clip_errors_match_oracle(g, mode):
    G, N = 4, 192
    cfg, ctx = make_ctx(G, g)
    try:
        Q, K, V = calib_inputs(G, N, seed=77 + g, n_out=8, f_key=30.0)
        Qn, Kn, Vn = (t.float().cpu().numpy() for t in (Q, K, V))
        U_K, U_V = O.calibrate(Qn, Kn, Vn) if mode == oscar.ROT_OSCAR else (np.eye(128), np.eye(128))
        UK = np.stack([U_K.astype(np.float32)] * 4)
        UV = np.stack([U_V.astype(np.float32)] * 4)
        oscar.oscar_set_rotation(ctx, 0, UK, UV, [1.0] * 4, [1.0] * 4, mode)
        scratch = oscar.calibration_scratch(G, N, len(RATIOS))
        ek, ev, bk, bv = oscar.oscar_clip_errors(ctx, 0, 2, Q, K, V, N, RATIOS, scratch)
        R_K, R_V = O.rotation(U_K, mode), O.rotation(U_V, mode)
        ek_o, ev_o, _, _ = O.clip_search(Qn, Kn, Vn, R_K, R_V, g, RATIOS)
        np.testing.assert_allclose(ek, ek_o, rtol=ERR_TOL)
        np.testing.assert_allclose(ev, ev_o, rtol=ERR_TOL)
        # the chosen ratio is optimal under the oracle's errors too (ties within tolerance)
        assert ek_o[bk] <= ek_o.min() * (1 + ERR_TOL)
        assert ev_o[bv] <= ev_o.min() * (1 + ERR_TOL)
        print(f"g={g} mode={mode}: key ratio {RATIOS[bk]}, value ratio {RATIOS[bv]}")
    finally:
        oscar.oscar_destroy(ctx)


def test_calibration_rejects_bad_arguments():
    cfg, ctx = make_ctx(4)
    try:
        Q, K, V = calib_inputs(4, 64, seed=5)
        scratch = oscar.calibration_scratch(4, 64, 2)
        small = oscar.calibration_scratch(4, 8, 0)
        with pytest.raises(oscar.OscarError):
            oscar.oscar_calibrate(ctx, Q, K, V, 64, small)  # scratch too small
        for bad in ([0.0, 1.0], [1.0, 1.5]):
            with pytest.raises(oscar.OscarError):
                oscar.oscar_clip_errors(ctx, 0, 0, Q, K, V, 64, bad, scratch)
        with pytest.raises(oscar.OscarError):
            oscar.oscar_clip_errors(ctx, 0, 4, Q, K, V, 64, [1.0], scratch)  # kv head out of range
    finally:
        oscar.oscar_destroy(ctx)


def test_calibrate_qwen3_8b_head_full_size():
    """One kv head of the Qwen3-8B-shaped layer with the 2048-token calibration
    set the benchmark uses: covariances and leading bases against the oracle."""
    G, N = 4, 2048
    cfg, ctx = make_ctx(G)
    try:
        st = synth.head_stats(0, "bench", 0, 3, n_out=4, f_key=20.0)
        Q, K, V = (t.cuda().contiguous() for t in synth.calibration_set(0, "bench", 0, 3, st, G=G, n=N))
        scratch = oscar.calibration_scratch(G, N)
        U_K, U_V, C_Q, C_S = oscar.oscar_calibrate(ctx, Q, K, V, N, scratch)
        Qn, Kn, Vn = (t.float().cpu().numpy() for t in (Q, K, V))
        CQ_o = O.query_covariance(Qn)
        CS_o = O.score_weighted_value_covariance(Qn, Kn, Vn)
        assert np.abs(C_Q - CQ_o).max() / np.abs(CQ_o).max() < COV_TOL
        assert np.abs(C_S - CS_o).max() / np.abs(CS_o).max() < COV_TOL
        assert check_basis(U_K, CQ_o) >= 8 and check_basis(U_V, CS_o) >= 8
    finally:
        oscar.oscar_destroy(ctx)
