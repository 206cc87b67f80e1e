"""Calibration checkpoint of OSCAR's rotations.

Per layer and KV head the offline calibration fixes the rotation bases and the
clip ratios [News "Together AI 开源 OSCAR…", section "OSCAR 的不同之处";
Blog "超越TurboQuant…", section "OSCAR把旋转对准attention"]:

* keys:   U_Q = eigenvectors of the query covariance C_Q,
* values: U_S = eigenvectors of the score-weighted value covariance C_S,

computed on the GPU by ``oscar.oscar_calibrate`` (covariances in CUDA kernels,
eigenvectors by cuSOLVER), with the clip ratios from ``oscar.oscar_clip_errors``
and the optional Lloyd-Max codebooks from ``oscar.oscar_fit_codebook``.  What
that produces is the only state that outlives a process; this module saves it
to one versioned .npz, reads it back and loads it into a context.  The KV cache
itself lives in the caller's memory.
"""
from __future__ import annotations

import numpy as np

CHECKPOINT_VERSION = 2
HEAD_DIM = 128


def _layer_kv_heads(L) -> int:
    return int(np.shape(L["U_K"])[0])


def save_layer_params(path, layers) -> None:
    """Writes per-layer calibration results to one .npz file.

    layers: list (one entry per layer) of dicts with U_K, U_V (float32
    [Hkv][128][128]), clip_k, clip_v (float32 [Hkv]), mode (an oscar rotation
    mode) and, optionally, k_ab / v_ab (float32 [Hkv][2] codebooks or None).
    Every layer must have the same Hkv; the file records it and head_dim."""
    if not layers:
        raise ValueError("no layers to save")
    hkv = _layer_kv_heads(layers[0])
    for i, L in enumerate(layers):
        _check_layer(L, hkv, f"layer {i}")
    arrays = {"version": np.array(CHECKPOINT_VERSION), "num_layers": np.array(len(layers)),
              "num_kv_heads": np.array(hkv), "head_dim": np.array(HEAD_DIM)}
    for i, L in enumerate(layers):
        arrays[f"l{i}_U_K"] = np.asarray(L["U_K"], dtype=np.float32)
        arrays[f"l{i}_U_V"] = np.asarray(L["U_V"], dtype=np.float32)
        arrays[f"l{i}_clip_k"] = np.asarray(L["clip_k"], dtype=np.float32)
        arrays[f"l{i}_clip_v"] = np.asarray(L["clip_v"], dtype=np.float32)
        arrays[f"l{i}_mode"] = np.array(int(L["mode"]))
        for key in ("k_ab", "v_ab"):
            if L.get(key) is not None:
                arrays[f"l{i}_{key}"] = np.asarray(L[key], dtype=np.float32)
    np.savez(path, **arrays)


def load_layer_params(path):
    """Reads a file written by save_layer_params; returns the list of dicts
    (k_ab / v_ab None where no codebook was stored).  Raises ValueError for
    another version or arrays whose shapes do not match the recorded sizes."""
    with np.load(path) as f:
        if int(f["version"]) != CHECKPOINT_VERSION:
            raise ValueError(f"unsupported calibration checkpoint version {int(f['version'])}")
        if int(f["head_dim"]) != HEAD_DIM:
            raise ValueError(f"checkpoint head_dim {int(f['head_dim'])} is not {HEAD_DIM}")
        hkv = int(f["num_kv_heads"])
        layers = []
        for i in range(int(f["num_layers"])):
            L = {k: f[f"l{i}_{k}"].copy() for k in ("U_K", "U_V", "clip_k", "clip_v")}
            L["mode"] = int(f[f"l{i}_mode"])
            for key in ("k_ab", "v_ab"):
                L[key] = f[f"l{i}_{key}"].copy() if f"l{i}_{key}" in f.files else None
            _check_layer(L, hkv, f"layer {i}")
            layers.append(L)
    return layers


def _check_layer(L, hkv: int, where: str) -> None:
    """Shapes the C ABI reads through bare pointers: bases [Hkv][128][128],
    clips [Hkv], codebooks [Hkv][2]."""
    want = {"U_K": (hkv, HEAD_DIM, HEAD_DIM), "U_V": (hkv, HEAD_DIM, HEAD_DIM), "clip_k": (hkv,), "clip_v": (hkv,)}
    for key, shape in want.items():
        if tuple(np.shape(L[key])) != shape:
            raise ValueError(f"{where}: {key} has shape {tuple(np.shape(L[key]))}, expected {shape}")
    for key in ("k_ab", "v_ab"):
        if L.get(key) is not None and tuple(np.shape(L[key])) != (hkv, 2):
            raise ValueError(f"{where}: {key} has shape {tuple(np.shape(L[key]))}, expected {(hkv, 2)}")


def apply_layer_params(ctx, cfg, layers) -> None:
    """Loads every layer's rotation, clips and codebooks into a context made
    from ``cfg`` (an oscar_config).  Every layer is checked against the
    configuration before the first call, so a mismatched file changes nothing."""
    from . import oscar

    if len(layers) > cfg.num_layers:
        raise ValueError(f"{len(layers)} layers in the checkpoint, the context has {cfg.num_layers}")
    if cfg.head_dim != HEAD_DIM:
        raise ValueError(f"context head_dim {cfg.head_dim} is not {HEAD_DIM}")
    for i, L in enumerate(layers):
        _check_layer(L, cfg.num_kv_heads, f"layer {i}")
    for i, L in enumerate(layers):
        oscar.oscar_set_rotation(ctx, i, L["U_K"], L["U_V"], L["clip_k"], L["clip_v"], L["mode"])
        oscar.oscar_set_codebook(ctx, i, L.get("k_ab"), L.get("v_ab"))
