"""Offline calibration of OSCAR's rotations (host, float64).

Per layer and KV head [News "Together AI 开源 OSCAR…", section "OSCAR 的不同之处";
Blog "超越TurboQuant…", section "OSCAR把旋转对准attention"]:

* keys:   U_Q = eigenvectors of the query covariance C_Q = (1/N) sum q^T q,
  pooled over the query heads that share the KV head;
* values: U_S = eigenvectors of C_S = (1/N) V^T S^T S V, S the causal
  attention scores of the calibration tokens, averaged over those heads;
* columns ordered by descending eigenvalue, each signed so its largest-magnitude
  entry is positive.

The library then applies x' = x·U·H·P_br.  This runs once, offline, and is not
on the decode path.
"""
from __future__ import annotations

import numpy as np


def _eig_desc(C: np.ndarray) -> np.ndarray:
    w, U = np.linalg.eigh(C)
    U = U[:, np.argsort(-w, kind="stable")]
    idx = np.argmax(np.abs(U), axis=0)
    sign = np.where(U[idx, np.arange(U.shape[1])] < 0, -1.0, 1.0)
    return U * sign[None, :]


def calibrate_kv_head(Q: np.ndarray, K: np.ndarray, V: np.ndarray):
    """Q: [G][N][d] calibration queries; K, V: [N][d].  Returns (U_Q, U_S) float32."""
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    G, N, d = Q.shape
    flat = Q.reshape(G * N, d)
    C_Q = flat.T @ flat / (G * N)
    causal = np.tril(np.ones((N, N), dtype=bool))
    C_S = np.zeros((d, d))
    for h in range(G):
        a = Q[h] @ K.T / np.sqrt(d)
        a = np.where(causal, a, -np.inf)
        a = np.exp(a - a.max(axis=1, keepdims=True))
        a /= a.sum(axis=1, keepdims=True)
        SV = a @ V
        C_S += SV.T @ SV
    C_S /= G * N
    return _eig_desc(C_Q).astype(np.float32), _eig_desc(C_S).astype(np.float32)


# ---------------------------------------------------------------- checkpoint
# What calibration produces is the only state that outlives a process: per
# layer the rotation bases and clip ratios, fixed offline [Blog, section
# "OSCAR把旋转对准attention"], and optionally the Lloyd-Max codebooks.  The
# KV cache itself lives in the caller's memory.

CHECKPOINT_VERSION = 1


def save_layer_params(path, layers) -> None:
    """Writes per-layer calibration results to one .npz file.

    layers: list (one entry per layer) of dicts with U_K, U_V (float32
    [Hkv][128][128]), clip_k, clip_v (float32 [Hkv]), mode (an oscar rotation
    mode) and, optionally, k_ab / v_ab (float32 [Hkv][2] codebooks or None)."""
    arrays = {"version": np.array(CHECKPOINT_VERSION), "num_layers": np.array(len(layers))}
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
    (k_ab / v_ab None where no codebook was stored)."""
    with np.load(path) as f:
        if int(f["version"]) != CHECKPOINT_VERSION:
            raise ValueError(f"unsupported calibration checkpoint version {int(f['version'])}")
        layers = []
        for i in range(int(f["num_layers"])):
            L = {k: f[f"l{i}_{k}"].copy() for k in ("U_K", "U_V", "clip_k", "clip_v")}
            L["mode"] = int(f[f"l{i}_mode"])
            for key in ("k_ab", "v_ab"):
                L[key] = f[f"l{i}_{key}"].copy() if f"l{i}_{key}" in f.files else None
            layers.append(L)
    return layers


def apply_layer_params(ctx, layers) -> None:
    """Loads every layer's rotation, clips and codebooks into a context."""
    from . import oscar

    for i, L in enumerate(layers):
        oscar.oscar_set_rotation(ctx, i, L["U_K"], L["U_V"], L["clip_k"], L["clip_v"], L["mode"])
        oscar.oscar_set_codebook(ctx, i, L.get("k_ab"), L.get("v_ab"))
