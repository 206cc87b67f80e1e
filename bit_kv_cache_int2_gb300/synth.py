"""Seeded synthetic inputs for the OSCAR INT2 KV-cache path.

This module only draws random tensors. It holds none of the method's
arithmetic (no rotation, quantisation or attention), so both the CUDA path
and the CPU oracle can take their inputs from it.

Distributions (the workloads the pages describe use Qwen3 head shapes; the
exact activation statistics are not published, so these stand in for them):

* keys    ~ N(0, 1), with ``n_out`` seeded channels scaled by ``f_out``
  (outlier channels, "为什么 INT2 KV 缓存量化很难？" in the news article
  "Together AI 开源 OSCAR").
* values  ~ N(0, 1), with 2 seeded channels scaled by 10.
* queries ~ N(0, Sigma), Sigma = B diag(lambda) B^T, lambda_i = i^-1.5
  (i = 1..d).  ``basis="aligned"`` puts the key-outlier channel unit vectors
  first (largest lambda first), then the remaining standard axes in index
  order; ``basis="haar"`` uses a seeded Haar-random orthogonal matrix.

All of K, V and Q are returned as bfloat16.  Every stream has its own seed,
derived from (base seed, workload id, layer, kv head, stream name).
"""
from __future__ import annotations

import dataclasses
import zlib

import numpy as np
import torch

STREAMS = ("calib", "K", "V", "Q", "newKV", "pages", "lengths", "outliers")


def stream_seed(base: int, *keys) -> int:
    """A 63-bit seed for one named stream, from numpy's SeedSequence."""
    ints = []
    for k in keys:
        if isinstance(k, str):
            ints.append(zlib.crc32(k.encode()))
        else:
            ints.append(int(k))
    ss = np.random.SeedSequence(entropy=int(base), spawn_key=tuple(ints))
    return int(ss.generate_state(1, dtype=np.uint64)[0] & ((1 << 63) - 1))


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


@dataclasses.dataclass(frozen=True)
class HeadStats:
    """Per (layer, kv head) distribution parameters."""

    key_outliers: tuple  # channel indices scaled by f_key
    value_outliers: tuple  # channel indices scaled by f_value
    f_key: float
    f_value: float
    basis: torch.Tensor  # [d][d] float64, columns = eigen-directions of Sigma
    lam: torch.Tensor  # [d] float64, descending


def head_stats(base: int, wl: str, layer: int, kvh: int, d: int = 128,
               n_out: int = 4, f_key: float = 20.0, n_vout: int = 2,
               f_value: float = 10.0, basis: str = "aligned") -> HeadStats:
    g = _gen("cpu", stream_seed(base, wl, layer, kvh, "outliers"))
    perm = torch.randperm(d, generator=g)
    kout = tuple(int(i) for i in perm[:n_out])
    perm_v = torch.randperm(d, generator=g)
    vout = tuple(int(i) for i in perm_v[:n_vout])
    lam = torch.arange(1, d + 1, dtype=torch.float64) ** -1.5
    if basis == "aligned":
        rest = [i for i in range(d) if i not in kout]
        order = list(kout) + rest
        B = torch.zeros(d, d, dtype=torch.float64)
        for col, ch in enumerate(order):
            B[ch, col] = 1.0
    elif basis == "haar":
        A = torch.randn(d, d, generator=g, dtype=torch.float64)
        Qm, Rm = torch.linalg.qr(A)
        B = Qm * torch.sign(torch.diagonal(Rm))[None, :]
    else:
        raise ValueError(basis)
    return HeadStats(kout, vout, f_key, f_value, B, lam)


def _scale_channels(x: torch.Tensor, chans, f: float) -> torch.Tensor:
    if len(chans):
        idx = torch.tensor(chans, device=x.device, dtype=torch.long)
        x[..., idx] *= f
    return x


def draw_keys(st: HeadStats, n: int, seed: int, device="cpu") -> torch.Tensor:
    g = _gen(device, seed)
    x = torch.randn(n, st.basis.shape[0], generator=g, device=device, dtype=torch.float32)
    return _scale_channels(x, st.key_outliers, st.f_key).to(torch.bfloat16)


def draw_values(st: HeadStats, n: int, seed: int, device="cpu") -> torch.Tensor:
    g = _gen(device, seed)
    x = torch.randn(n, st.basis.shape[0], generator=g, device=device, dtype=torch.float32)
    return _scale_channels(x, st.value_outliers, st.f_value).to(torch.bfloat16)


def draw_queries(st: HeadStats, n: int, seed: int, device="cpu") -> torch.Tensor:
    """n queries ~ N(0, B diag(lam) B^T), as bf16 [n][d]."""
    g = _gen(device, seed)
    d = st.basis.shape[0]
    z = torch.randn(n, d, generator=g, device=device, dtype=torch.float32)
    z = z * torch.sqrt(st.lam).to(device=device, dtype=torch.float32)[None, :]
    q = z @ st.basis.to(device=device, dtype=torch.float32).T
    return q.to(torch.bfloat16)


def calibration_set(base: int, wl: str, layer: int, kvh: int, st: HeadStats,
                    G: int, n: int = 2048):
    """(Q [G][n][d], K [n][d], V [n][d]) bf16 calibration tokens for one kv head."""
    s = stream_seed(base, wl, layer, kvh, "calib")
    K = draw_keys(st, n, s ^ 0x1)
    V = draw_values(st, n, s ^ 0x2)
    Q = torch.stack([draw_queries(st, n, s ^ (0x100 + h)) for h in range(G)])
    return Q, K, V


def page_table(num_pages: int, pages_per_req, seed: int, interleave: bool,
               max_pages_per_req: int) -> torch.Tensor:
    """int32 [B][max_pages_per_req] page table, -1 where unused.

    Pages come from a seeded permutation of the pool.  With ``interleave``
    the permutation is dealt out round-robin across requests, so a request's
    pages are spread through the pool among other requests' pages.
    """
    B = len(pages_per_req)
    need = int(sum(pages_per_req))
    if need > num_pages:
        raise ValueError("pool too small")
    g = _gen("cpu", seed)
    perm = torch.randperm(num_pages, generator=g)[:need].tolist()
    pt = torch.full((B, max_pages_per_req), -1, dtype=torch.int32)
    if interleave:
        cursor = 0
        k = 0
        while cursor < need:
            for b in range(B):
                if k < pages_per_req[b]:
                    pt[b, k] = perm[cursor]
                    cursor += 1
            k += 1
    else:
        cursor = 0
        for b in range(B):
            n = pages_per_req[b]
            pt[b, :n] = torch.tensor(perm[cursor:cursor + n], dtype=torch.int32)
            cursor += n
    return pt


def lengths(B: int, lo: int, hi: int, seed: int) -> list:
    """B request lengths uniform in [lo, hi] (inclusive)."""
    g = _gen("cpu", seed)
    return [int(x) for x in torch.randint(lo, hi + 1, (B,), generator=g)]
