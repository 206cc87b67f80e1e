"""Calibration checkpoint (bit_kv_cache_int2_gb300.calibration): per-layer
rotation bases, clips, modes and codebooks survive a save/load round trip
exactly, and apply_layer_params loads each layer through the C ABI calls."""
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
    calibration.apply_layer_params("ctx", _layers())
    assert calls == [("rot", 0, 0), ("cb", 0, False, True), ("rot", 1, 1), ("cb", 1, True, True),
                     ("rot", 2, 2), ("cb", 2, False, False)]
