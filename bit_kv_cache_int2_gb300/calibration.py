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
