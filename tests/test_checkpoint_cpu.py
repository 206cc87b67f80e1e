"""Calibration checkpoint (bit_kv_cache_int2_gb300.calibration): per-layer
rotation bases, clips, modes and codebooks survive a save/load round trip
exactly, apply_layer_params loads each layer through the C ABI calls, and a
file that does not fit the context is refused before any call."""
import numpy as np
import pytest

from bit_kv_cache_int2_gb300 import calibration, oscar


def _layers(n=3, Hkv=2, seed=0):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        U = [np.linalg.qr(rng.standard_normal((128, 128)))[0].astype(np.float32) for _ in range(2 * Hkv)]
        out.append({"U_K": np.stack(U[:Hkv]), "U_V": np.stack(U[Hkv:]),
                    "clip_k": rng.uniform(0.8, 1.0, Hkv).astype(np.float32),
                    "clip_v": rng.uniform(0.8, 1.0, Hkv).astype(np.float32), "mode": i % 3,
                    "k_ab": None if i == 1 else rng.uniform([0.2, 1.0], [0.5, 1.6], (Hkv, 2)).astype(np.float32),
                    "v_ab": None if i != 2 else rng.uniform([0.2, 1.0], [0.5, 1.6], (Hkv, 2)).astype(np.float32)})
    return out


def test_round_trip_is_exact(tmp_path):
    layers = _layers()
    path = tmp_path / "calib.npz"
    calibration.save_layer_params(path, layers)
    back = calibration.load_layer_params(path)
    assert len(back) == len(layers)
    for a, b in zip(layers, back):
        for key in ("U_K", "U_V", "clip_k", "clip_v"):
            np.testing.assert_array_equal(a[key], b[key])
        assert a["mode"] == b["mode"]
        for key in ("k_ab", "v_ab"):
            if a[key] is None:
                assert b[key] is None
            else:
                np.testing.assert_array_equal(a[key], b[key])
    with np.load(path) as f:
        assert int(f["num_kv_heads"]) == 2 and int(f["head_dim"]) == 128


def test_version_is_checked(tmp_path):
    path = tmp_path / "bad.npz"
    np.savez(path, version=np.array(99), num_layers=np.array(0))
    with pytest.raises(ValueError):
        calibration.load_layer_params(path)


def test_apply_sets_every_layer(monkeypatch):
    calls = []
    monkeypatch.setattr(oscar, "oscar_set_rotation", lambda ctx, i, UK, UV, ck, cv, mode: calls.append(("rot", i, mode)))
    monkeypatch.setattr(oscar, "oscar_set_codebook",
                        lambda ctx, i, kab, vab: calls.append(("cb", i, kab is None, vab is None)))
    cfg = oscar.make_config(3, 4, 2, 128, max_batch=1, max_pages_per_req=1, num_pages=1)
    calibration.apply_layer_params("ctx", cfg, _layers())
    assert calls == [("rot", 0, 0), ("cb", 0, False, True), ("rot", 1, 1), ("cb", 1, True, True),
                     ("rot", 2, 2), ("cb", 2, False, False)]


@pytest.mark.parametrize("case", ["fewer_kv_heads", "more_layers", "bad_clip", "bad_codebook"])
def test_mismatched_file_is_refused_before_any_call(monkeypatch, case):
    calls = []
    monkeypatch.setattr(oscar, "oscar_set_rotation", lambda *a: calls.append("rot"))
    monkeypatch.setattr(oscar, "oscar_set_codebook", lambda *a: calls.append("cb"))
    layers = _layers(n=3, Hkv=2)
    cfg = oscar.make_config(3, 8, 4 if case == "fewer_kv_heads" else 2, 128, max_batch=1, max_pages_per_req=1,
                            num_pages=1)
    if case == "more_layers":
        cfg = oscar.make_config(2, 4, 2, 128, max_batch=1, max_pages_per_req=1, num_pages=1)
    if case == "bad_clip":
        layers[2]["clip_v"] = np.ones(3, np.float32)
    if case == "bad_codebook":
        layers[1]["k_ab"] = np.ones((2, 3), np.float32)
    with pytest.raises(ValueError):
        calibration.apply_layer_params("ctx", cfg, layers)
    assert calls == []


def test_load_refuses_arrays_that_do_not_match_the_recorded_sizes(tmp_path):
    layers = _layers(n=2, Hkv=2)
    path = tmp_path / "calib.npz"
    calibration.save_layer_params(path, layers)
    with np.load(path) as f:
        arrays = {k: f[k] for k in f.files}
    arrays["l1_U_V"] = arrays["l1_U_V"][:1]
    np.savez(path, **arrays)
    with pytest.raises(ValueError):
        calibration.load_layer_params(path)
