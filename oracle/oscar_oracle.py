"""Plain CPU oracle for OSCAR's INT2 KV-cache decode path (test infrastructure).

Only tests, ``__graft_entry__.smoke()`` and the CPU-baseline legs of
``bench.py`` may use this module.  It shares no code with the CUDA library.

Sources (pages, cited by title and section):

* [News] "Together AI 开源 OSCAR：一种面向长上下文 LLM 服务的注意力感知 2 位
  KV 缓存量化系统" -- sections "OSCAR 的不同之处" (logit-error identity, C_Q,
  C_S, R = U·H_Had·P_br) and "服务系统：混合精度缓存布局" (sink 64 | INT2
  history | recent 256).
* [Blog] "超越TurboQuant：Together AI把2-bit KV Cache推向真实服务" -- section
  "OSCAR把旋转对准attention" (per layer / per head calibration, fixed
  rotation and clipping thresholds) and the pipeline figure
  "从离线校准到在线推理的pipeline" with the paragraph under it (recent window
  first, demotion by rotate -> clip -> quantize -> pack, 4 codes per byte,
  scale/zero-point dequantisation, INT2 and BF16 segments merged by online
  softmax).
* [Telegram] "OSCAR: открытая система двухбитного сжатия KV-кэша" -- first 64
  and last 256 tokens in BF16; calibration once, fixed rotation and clip.

Precision: attention, calibration and rotations in float64; the quantiser in
float32 with one IEEE rounding per operation (numpy float32 scalars/arrays),
because a float decides an integer code there and both sides must take that
decision in the same precision.

Readings where the pages are silent (each one is listed in the design notes):
clip = scale the group's min and max by the ratio c; zero point = an fp16
float offset (x_hat = code*s + z); round half to even; a zero scale gives
all-zero codes; groups are g consecutive channels after P_br; eigenvectors in
descending eigenvalue order, each column signed so its largest-|.| entry is
positive; C_Q and C_S pool the G query heads of a kv head; S is the causal
softmax(QK^T/sqrt(d)); softmax scale 1/sqrt(d); the recent window holds the
newest 256 tokens including the one just appended.  The clip search and the
Lloyd-Max codebook (symmetric levels on the uniform quantiser's normalised
value, fitted by the two-level fold) carry their readings in their sections
below.  Every function here is pinned by tests/test_oracle.py (closed forms,
worked examples, textbook tables, brute force); beyond the stated tolerances
only the bf16 rounding of decode outputs is unpinned.
"""
from __future__ import annotations

import numpy as np

SINK = 64
RECENT = 256
PAGE = 64

ROT_OSCAR = 0
ROT_HADAMARD = 1
ROT_NONE = 2


# --------------------------------------------------------------------------
# Rotation factors  [News, "OSCAR 的不同之处": R_K = U_Q·H_Had·P_br]
# --------------------------------------------------------------------------

def sylvester_hadamard(n: int) -> np.ndarray:
    """Normalised Sylvester Hadamard matrix: H_1 = [1], H_2n = [[H, H], [H, -H]],
    divided by sqrt(n) so that it is orthogonal."""
    if n < 1 or n & (n - 1):
        raise ValueError("n must be a power of two")
    H = np.ones((1, 1))
    while H.shape[0] < n:
        H = np.block([[H, H], [H, -H]])
    return H / np.sqrt(n)


def bit_reverse(j: int, bits: int) -> int:
    """Reverse the low ``bits`` bits of j, one bit at a time."""
    r = 0
    for _ in range(bits):
        r = (r << 1) | (j & 1)
        j >>= 1
    return r


def bit_reversal_matrix(n: int) -> np.ndarray:
    """P_br with (x P_br)_j = x_{bitrev(j)}: channel j swaps with bitrev(j)."""
    bits = n.bit_length() - 1
    P = np.zeros((n, n))
    for j in range(n):
        P[bit_reverse(j, bits), j] = 1.0
    return P


def rotation(U: np.ndarray, mode: int = ROT_OSCAR) -> np.ndarray:
    """The row-vector rotation x' = x R.

    OSCAR: R = U·H·P_br  [News, "OSCAR 的不同之处"; Blog, "OSCAR把旋转对准attention"].
    HADAMARD: R = H (the Hadamard-only baseline the news article's "结果"
    section compares against).  NONE: R = I (naive INT2).
    """
    U = np.asarray(U, dtype=np.float64)
    d = U.shape[0]
    if mode == ROT_OSCAR:
        return U @ sylvester_hadamard(d) @ bit_reversal_matrix(d)
    if mode == ROT_HADAMARD:
        return sylvester_hadamard(d)
    if mode == ROT_NONE:
        return np.eye(d)
    raise ValueError(mode)


# --------------------------------------------------------------------------
# Calibration  [News, "OSCAR 的不同之处"; Blog, "OSCAR把旋转对准attention"]
# --------------------------------------------------------------------------

def query_covariance(Q: np.ndarray) -> np.ndarray:
    """C_Q = (1/N) sum_n q_n^T q_n over the N rows q_n of Q (row vectors).

    For a kv head, Q stacks the calibration queries of all G query heads that
    read it (the keys are shared, so one rotation serves all of them)."""
    Q = np.asarray(Q, dtype=np.float64).reshape(-1, np.shape(Q)[-1])
    N = Q.shape[0]
    C = np.zeros((Q.shape[1], Q.shape[1]))
    for n in range(N):
        C += np.outer(Q[n], Q[n])
    return C / N


def causal_scores(Qh: np.ndarray, K: np.ndarray) -> np.ndarray:
    """S = softmax(Q K^T / sqrt(d)) with a causal mask (token n sees keys <= n)."""
    Qh = np.asarray(Qh, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    d = Qh.shape[1]
    logits = Qh @ K.T / np.sqrt(d)
    N = logits.shape[0]
    mask = np.triu(np.ones((N, N), dtype=bool), k=1)
    logits[mask] = -np.inf
    logits -= logits.max(axis=1, keepdims=True)
    e = np.exp(logits)
    return e / e.sum(axis=1, keepdims=True)


def score_weighted_value_covariance(Q: np.ndarray, K: np.ndarray, V: np.ndarray) -> np.ndarray:
    """C_S = (1/N) V^T S^T S V, averaged over the G query heads of the kv head.

    Q: [G][N][d] calibration queries, K, V: [N][d]."""
    Q = np.asarray(Q, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    G, N = Q.shape[0], Q.shape[1]
    C = np.zeros((V.shape[1], V.shape[1]))
    for h in range(G):
        SV = causal_scores(Q[h], K) @ V
        C += SV.T @ SV
    return C / (N * G)


def eigenbasis(C: np.ndarray) -> np.ndarray:
    """Eigenvectors of symmetric C as columns, by descending eigenvalue; each
    column signed so that its largest-magnitude entry (lowest index on ties)
    is positive."""
    w, U = np.linalg.eigh(np.asarray(C, dtype=np.float64))
    order = np.argsort(-w, kind="stable")
    U = U[:, order].copy()
    for j in range(U.shape[1]):
        i = int(np.argmax(np.abs(U[:, j])))
        if U[i, j] < 0:
            U[:, j] = -U[:, j]
    return U


def calibrate(Q: np.ndarray, K: np.ndarray, V: np.ndarray):
    """(U_Q, U_S) for one (layer, kv head) from calibration tokens."""
    U_Q = eigenbasis(query_covariance(Q))
    U_S = eigenbasis(score_weighted_value_covariance(Q, K, V))
    return U_Q, U_S


# --------------------------------------------------------------------------
# Quantiser  [Blog, pipeline figure: rotate -> clip -> quantize -> pack;
#             INT2 kernel dequantises with scale / zero point]
# --------------------------------------------------------------------------

HALF_MAX = np.float32(65504.0)


def half_rn_sat(x) -> np.float16:
    """float32 -> fp16, round to nearest even, saturating at +-65504."""
    with np.errstate(over="ignore"):
        h = np.float16(np.float32(x))
    if np.isinf(h):
        h = np.float16(np.copysign(65504.0, float(h)))
    return h


def quantize_group(x, clip: float):
    """One group of rotated channels -> (codes, s, z), float32 steps:

    mx, mn = max, min;  mx_c = c*mx, mn_c = c*mn;  s32 = (mx_c - mn_c)/3;
    s = half(s32), z = half(mn_c);  code = clamp(rint((x - z)/s), 0, 3),
    or all zeros when s == 0.
    """
    x = np.asarray(x, dtype=np.float32)
    c = np.float32(clip)
    mx = np.float32(x.max())
    mn = np.float32(x.min())
    mx_c = np.float32(c * mx)
    mn_c = np.float32(c * mn)
    s32 = np.float32(np.float32(mx_c - mn_c) / np.float32(3.0))
    s = half_rn_sat(s32)
    z = half_rn_sat(mn_c)
    if np.float32(s) == 0:
        return np.zeros(x.shape, dtype=np.uint8), s, z
    t = (x - np.float32(z)) / np.float32(s)
    assert t.dtype == np.float32
    codes = np.clip(np.rint(t), 0, 3).astype(np.uint8)
    return codes, s, z


def quantize_vector(x, g: int, clip: float):
    """A rotated d-vector -> codes [d], s [d/g], z [d/g] (groups of g consecutive channels)."""
    x = np.asarray(x, dtype=np.float32)
    d = x.shape[0]
    codes = np.zeros(d, dtype=np.uint8)
    s = np.zeros(d // g, dtype=np.float16)
    z = np.zeros(d // g, dtype=np.float16)
    for gr in range(d // g):
        c, si, zi = quantize_group(x[gr * g:(gr + 1) * g], clip)
        codes[gr * g:(gr + 1) * g] = c
        s[gr] = si
        z[gr] = zi
    return codes, s, z


def dequantize(codes, s, z, g: int) -> np.ndarray:
    """x_hat = code*s + z per group, float64."""
    codes = np.asarray(codes, dtype=np.float64)
    sg = np.repeat(np.asarray(s, dtype=np.float64), g, axis=-1)
    zg = np.repeat(np.asarray(z, dtype=np.float64), g, axis=-1)
    return codes * sg + zg


def rotate_to_f32(x_bf16_as_f32, R: np.ndarray) -> np.ndarray:
    """x' = x R in float64, rounded once to float32 for the quantiser."""
    return (np.asarray(x_bf16_as_f32, dtype=np.float64) @ R).astype(np.float32)


# --------------------------------------------------------------------------
# Packing: 4 two-bit codes per byte  [Blog, pipeline figure paragraph]
#
# Byte rule: the code at bit position b of a little-endian 32-bit word sits
# in byte b//8, bits b%8 .. b%8+1 (LSB first).  Where each code goes inside a
# page is the library's layout, restated here from its definition:
#   K codes, token-major, 8 words per token; channel c = 64A+16B+8C+2D+E
#     -> word 2D+A, bit 16E + 2(2B+C).
#   V codes, channel-major, 4 words per channel row per 64-token page;
#     token t = 16S+8A+2T+E -> word T, bit 16E + 2(2S+A).
#   s/z: one (s, z) fp16 pair per token and group, s first.
# --------------------------------------------------------------------------

def k_code_position(c: int):
    A, rem = divmod(c, 64)
    B, rem = divmod(rem, 16)
    C, rem = divmod(rem, 8)
    D, E = divmod(rem, 2)
    return 2 * D + A, 16 * E + 2 * (2 * B + C)


def v_code_position(t: int):
    S, rem = divmod(t, 16)
    A, rem = divmod(rem, 8)
    T, E = divmod(rem, 2)
    return T, 16 * E + 2 * (2 * S + A)


def pack_bits(codes_at, nbytes: int) -> np.ndarray:
    """codes_at: iterable of (word, bit, code) -> little-endian byte array."""
    out = np.zeros(nbytes, dtype=np.uint8)
    for word, bit, code in codes_at:
        byte = 4 * word + bit // 8
        out[byte] |= np.uint8((int(code) & 3) << (bit % 8))
    return out


def pack_k_row(codes) -> np.ndarray:
    """128 K codes of one token -> 32 bytes."""
    items = []
    for c, code in enumerate(codes):
        w, b = k_code_position(c)
        items.append((w, b, code))
    return pack_bits(items, 32)


def unpack_k_rows(rows: np.ndarray) -> np.ndarray:
    """[n][32] bytes -> [n][128] codes."""
    rows = np.asarray(rows, dtype=np.uint8)
    out = np.zeros(rows.shape[:-1] + (128,), dtype=np.uint8)
    for c in range(128):
        w, b = k_code_position(c)
        byte = 4 * w + b // 8
        out[..., c] = (rows[..., byte] >> (b % 8)) & 3
    return out


def pack_v_block(codes) -> np.ndarray:
    """[64 tokens][128 channels] V codes -> 2048 bytes (128 rows of 16 bytes)."""
    codes = np.asarray(codes)
    out = np.zeros(128 * 16, dtype=np.uint8)
    for ch in range(128):
        items = []
        for t in range(64):
            w, b = v_code_position(t)
            items.append((w, b, codes[t, ch]))
        out[ch * 16:(ch + 1) * 16] = pack_bits(items, 16)
    return out


def unpack_v_blocks(blocks: np.ndarray) -> np.ndarray:
    """[..][2048] bytes -> [..][64 tokens][128 channels] codes."""
    blocks = np.asarray(blocks, dtype=np.uint8)
    rows = blocks.reshape(blocks.shape[:-1] + (128, 16))
    out = np.zeros(blocks.shape[:-1] + (64, 128), dtype=np.uint8)
    for t in range(64):
        w, b = v_code_position(t)
        byte = 4 * w + b // 8
        out[..., t, :] = (rows[..., :, byte] >> (b % 8)) & 3
    return out


def int2_head_block_bytes(g: int, d: int = 128) -> int:
    return 64 * (d // 4) * 2 + 64 * (d // g) * 4 * 2


def parse_head_block(block: np.ndarray, g: int, d: int = 128):
    """Head blocks [..][bytes] of INT2 pages -> dict of codes and fp16 s/z arrays
    (k_codes [..][64][128], v_codes [..][64 tokens][128], *_s / *_z [..][64][d/g])."""
    block = np.ascontiguousarray(np.asarray(block, dtype=np.uint8))
    lead = block.shape[:-1]
    ng = d // g
    kc = block[..., 0:2048].reshape(lead + (64, 32))
    vc = block[..., 2048:4096]
    szb = 64 * ng * 4
    ksz = np.ascontiguousarray(block[..., 4096:4096 + szb]).view(np.float16).reshape(lead + (64, ng, 2))
    vsz = np.ascontiguousarray(block[..., 4096 + szb:4096 + 2 * szb]).view(np.float16).reshape(lead + (64, ng, 2))
    return {
        "k_codes": unpack_k_rows(kc),
        "v_codes": unpack_v_blocks(vc),
        "k_s": ksz[..., 0].copy(), "k_z": ksz[..., 1].copy(),
        "v_s": vsz[..., 0].copy(), "v_z": vsz[..., 1].copy(),
    }


# --------------------------------------------------------------------------
# Attention  [News, "服务系统：混合精度缓存布局"; Blog, pipeline figure]
# --------------------------------------------------------------------------

def softmax_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray):
    """Plain softmax attention for query rows q [G][d] over K, V [n][d]:
    o = softmax(q K^T / sqrt(d)) V; also returns lse = log sum exp(logits)."""
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    lam = q @ K.T / np.sqrt(q.shape[-1])
    m = lam.max(axis=-1, keepdims=True)
    e = np.exp(lam - m)
    lsum = e.sum(axis=-1, keepdims=True)
    return (e / lsum) @ V, (m + np.log(lsum))[..., 0]


def three_region_attention(q, win_k, win_v, hist_k_rot, hist_v_rot, R_K, R_V):
    """One kv head's decode attention over the three-region cache, float64.

    q [G][d] raw queries; win_k / win_v [n_w][d] the BF16 sink + recent
    tokens (unrotated); hist_k_rot / hist_v_rot [n_h][d] the dequantised
    history, which lives in the rotated basis (x' = x R).

    Logits: q.k/sqrt(d) on the window; (q R_K).k'/sqrt(d) on history.  One
    softmax over all of them.  Output: sum_w p v + (sum_h p v') R_V^T.
    Returns (o [G][d], lse [G]).
    """
    q = np.asarray(q, dtype=np.float64)
    d = q.shape[-1]
    R_K = np.asarray(R_K, dtype=np.float64)
    R_V = np.asarray(R_V, dtype=np.float64)
    wk = np.asarray(win_k, dtype=np.float64).reshape(-1, d)
    wv = np.asarray(win_v, dtype=np.float64).reshape(-1, d)
    hk = np.asarray(hist_k_rot, dtype=np.float64).reshape(-1, d)
    hv = np.asarray(hist_v_rot, dtype=np.float64).reshape(-1, d)
    lam_w = q @ wk.T / np.sqrt(d)
    lam_h = (q @ R_K) @ hk.T / np.sqrt(d)
    lam = np.concatenate([lam_w, lam_h], axis=-1)
    m = lam.max(axis=-1, keepdims=True)
    e = np.exp(lam - m)
    lsum = e.sum(axis=-1, keepdims=True)
    p = e / lsum
    nw = wk.shape[0]
    o = p[:, :nw] @ wv + (p[:, nw:] @ hv) @ R_V.T
    return o, (m + np.log(lsum))[..., 0]


def chunk_prefill_attention(q_chunk, k_chunk, v_chunk, win_k, win_v, hist_k_rot, hist_v_rot, R_K, R_V,
                            tokens=None):
    """Chunked prefill over the cache of one kv head, float64: T new tokens
    (a prefix-hit extension) attend to the cache as it stands -- the BF16 sink
    and recent window, the INT2 history in the rotated basis -- and causally
    to the chunk's own BF16 tokens: chunk query t sees chunk tokens 0..t.
    The chunk is not stored by this step.

    This is the plain reading of the "next" row of the pages' prefix-cache
    reuse (News, "服务系统：混合精度缓存布局"; Blog, pipeline paragraph): the
    decode attention of each chunk token with the earlier chunk tokens as extra
    full-precision window tokens.

    q_chunk [T][G][d]; k_chunk, v_chunk [T][d]; the rest as in
    three_region_attention.  Returns (o [T][G][d], lse [T][G]); with `tokens`
    (a list of chunk positions) only those rows, in that order.
    """
    q_chunk = np.asarray(q_chunk, dtype=np.float64)
    kc = np.asarray(k_chunk, dtype=np.float64)
    vc = np.asarray(v_chunk, dtype=np.float64)
    wk = np.asarray(win_k, dtype=np.float64).reshape(-1, q_chunk.shape[-1])
    wv = np.asarray(win_v, dtype=np.float64).reshape(-1, q_chunk.shape[-1])
    outs, lses = [], []
    for t in (range(q_chunk.shape[0]) if tokens is None else tokens):
        o, l = three_region_attention(q_chunk[t], np.concatenate([wk, kc[:t + 1]]),
                                      np.concatenate([wv, vc[:t + 1]]), hist_k_rot, hist_v_rot, R_K, R_V)
        outs.append(o)
        lses.append(l)
    return np.stack(outs), np.stack(lses)


def lse_merge(parts):
    """Merge online-softmax partials (m, l, o) -- o normalised by l -- into one.

    m = max m_i; l = sum l_i e^{m_i - m}; o = sum l_i e^{m_i - m} o_i / l.
    A part with l == 0 contributes nothing."""
    parts = [p for p in parts if p[1] > 0]
    m = max(p[0] for p in parts)
    w = [p[1] * np.exp(p[0] - m) for p in parts]
    lsum = sum(w)
    o = sum(wi * np.asarray(p[2], dtype=np.float64) for wi, p in zip(w, parts)) / lsum
    return m, lsum, o


def segment_partial(q_row, K, V):
    """(m, l, o) of one query row over one segment, o normalised by l."""
    q_row = np.asarray(q_row, dtype=np.float64)
    lam = np.asarray(K, dtype=np.float64) @ q_row / np.sqrt(q_row.shape[0])
    m = lam.max()
    e = np.exp(lam - m)
    return m, e.sum(), e @ np.asarray(V, dtype=np.float64) / e.sum()


# --------------------------------------------------------------------------
# Cache regions and state  [News, "服务系统：混合精度缓存布局";
#                            Blog, pipeline figure paragraph]
# --------------------------------------------------------------------------

def region_of(p: int, L: int, H: int):
    """Where absolute position p lives in a request with L tokens, H of them
    in INT2 history: ('sink', p) | ('hist', p - 64) | ('ring', (p - 64) % 256)."""
    if p < SINK:
        return "sink", p
    if p < SINK + H:
        return "hist", p - SINK
    return "ring", (p - SINK) % RECENT


class CacheModel:
    """One request's cache for one kv head, as the pages describe it.

    Appending writes the new token to the recent window; when the window
    already holds 256 tokens its oldest token is first demoted (rotated,
    clipped, quantised, packed) into INT2 history.  ``demote`` demotes the
    oldest recent token without appending.  Tokens are kept as their bf16
    values (float32 arrays) so the quantisation can be re-derived.
    """

    def __init__(self):
        self.L = 0
        self.H = 0
        self.tokens_k = []  # position -> bf16 key (float32 copy)
        self.tokens_v = []

    def recent_count(self):
        return max(self.L - SINK - self.H, 0)

    def demote(self):
        if self.recent_count() == 0:
            return False
        self.H += 1
        return True

    def append(self, k, v):
        if self.L >= SINK and self.recent_count() == RECENT:
            self.demote()
        self.tokens_k.append(np.asarray(k, dtype=np.float32))
        self.tokens_v.append(np.asarray(v, dtype=np.float32))
        self.L += 1

    def import_tokens(self, K, V):
        """Bulk import into an empty cache: same result as appending each token."""
        assert self.L == 0
        for k, v in zip(K, V):
            self.append(k, v)

    def window_positions(self):
        sink = list(range(min(self.L, SINK)))
        recent = list(range(SINK + self.H, self.L)) if self.L > SINK else []
        return sink + recent

    def history_positions(self):
        return list(range(SINK, SINK + self.H))


# --------------------------------------------------------------------------
# Closed forms  [News, "服务系统：混合精度缓存布局" and "结果"]
# --------------------------------------------------------------------------

def bits_per_element(g: int, L: int, scale_bits: int = 16, zero_bits: int = 16) -> float:
    """Average stored bits per KV element: history tokens cost 2 bits plus an
    fp16 scale and zero per group of g; the 320 sink + recent tokens cost 16."""
    bf16_tokens = min(L, SINK + RECENT)
    hist = L - bf16_tokens
    return (hist * (2 + (scale_bits + zero_bits) / g) + bf16_tokens * 16) / L


def logit_error_direct(Q, K, K_hat) -> float:
    """||Q K^T - Q K_hat^T||_F^2."""
    Q = np.asarray(Q, dtype=np.float64)
    D = Q @ np.asarray(K, dtype=np.float64).T - Q @ np.asarray(K_hat, dtype=np.float64).T
    return float(np.sum(D * D))


def logit_error_trace(Q, K, K_hat) -> float:
    """tr((K - K_hat) Q^T Q (K - K_hat)^T)  [News, "OSCAR 的不同之处"]."""
    Q = np.asarray(Q, dtype=np.float64)
    E = np.asarray(K, dtype=np.float64) - np.asarray(K_hat, dtype=np.float64)
    return float(np.trace(E @ (Q.T @ Q) @ E.T))


# --------------------------------------------------------------------------
# Clip search  [Blog, "OSCAR把旋转对准attention": rotation and clipping
#               thresholds are fixed offline per layer and head; News, "OSCAR
#               的不同之处": the key error that matters is the logit error]
# --------------------------------------------------------------------------
# Reading: a clip ratio is chosen from a candidate grid by the error it leaves
# in what attention computes -- for keys the logit error ||Q K^T - Q K_hat^T||_F^2
# over the calibration queries of all G heads, for values the output error
# sum_h ||S_h V - S_h V_hat||_F^2 with S_h the causal scores of head h.  Both are
# taken in the rotated basis, where they are equal to the unrotated ones
# (R is orthogonal and Q K^T = (Q R)(K R)^T).

def quantize_dequantize_rows(X, g: int, clip: float, codebook=None) -> np.ndarray:
    """Each row quantised with the demotion's quantiser and dequantised,
    float64; codebook = (a, b) uses the Lloyd-Max levels instead (below)."""
    X = np.asarray(X, dtype=np.float32)
    out = np.zeros(X.shape, dtype=np.float64)
    for n in range(X.shape[0]):
        if codebook is None:
            codes, s, z = quantize_vector(X[n], g, clip)
            out[n] = dequantize(codes, s, z, g)
        else:
            codes, s, z = quantize_vector_codebook(X[n], g, clip, *codebook)
            out[n] = dequantize_codebook(codes, s, z, g, *codebook)
    return out


def key_clip_error(Q, K, R_K, g: int, clip: float, codebook=None) -> float:
    """||Q' K'^T - Q' K_hat'^T||_F^2, Q' = Q R_K over the G heads' calibration
    queries (Q [G][N][d] or [rows][d]), K' = K R_K in fp32 as the demotion
    rotates, K_hat' its quantised and dequantised copy with ratio `clip`."""
    Qr = np.asarray(Q, dtype=np.float64).reshape(-1, np.shape(Q)[-1]) @ np.asarray(R_K, dtype=np.float64)
    Kr = rotate_to_f32(K, R_K)
    return logit_error_direct(Qr, Kr.astype(np.float64), quantize_dequantize_rows(Kr, g, clip, codebook))


def value_clip_error(Q, K, V, R_V, g: int, clip: float, codebook=None) -> float:
    """sum_h ||S_h (V' - V_hat')||_F^2, S_h = causal_scores(Q_h, K) (unrotated
    scores), V' = V R_V in fp32, V_hat' quantised and dequantised with `clip`."""
    Vr = rotate_to_f32(V, R_V)
    E = Vr.astype(np.float64) - quantize_dequantize_rows(Vr, g, clip, codebook)
    Q = np.asarray(Q, dtype=np.float64)
    total = 0.0
    for h in range(Q.shape[0]):
        Y = causal_scores(Q[h], K) @ E
        total += float(np.sum(Y * Y))
    return total


def clip_search(Q, K, V, R_K, R_V, g: int, ratios, codebook_k=None, codebook_v=None):
    """Errors of every candidate ratio and the argmin for keys and values."""
    ek = [key_clip_error(Q, K, R_K, g, c, codebook_k) for c in ratios]
    ev = [value_clip_error(Q, K, V, R_V, g, c, codebook_v) for c in ratios]
    return np.array(ek), np.array(ev), int(np.argmin(ek)), int(np.argmin(ev))


# --------------------------------------------------------------------------
# Lloyd-Max codebook  [Blog, closing paragraph on TurboQuant: the released code
#                      already pairs the attention-aware rotation with a
#                      Lloyd-Max codebook]
# --------------------------------------------------------------------------
# The pages name the codebook and nothing more.  Reading taken:
# * the group's scale and zero point are the uniform quantiser's, and so is the
#   normalised value t = (x - z)/s (float32); only the four values t is
#   rounded to change;
# * the levels are symmetric about 1.5: {1.5-b, 1.5-a, 1.5+a, 1.5+b} with
#   0 <= a < b.  Min-max normalisation centres t on 1.5 when the rotated
#   coordinates are symmetric about 0, which the rotation makes them;
# * a code is the level nearest to t, ties to the even code.  With the
#   midpoint m = (a + b)/2 that is: code = [t > 1.5-m] + [t >= 1.5] + [t > 1.5+m]
#   (float32), which for a = 1/2, b = 3/2 is clamp(rint(t), 0, 3) exactly;
# * fitting is Lloyd-Max -- alternate nearest-level cells and centroid levels
#   to lower the mean squared error of t -- which for symmetric levels is a
#   two-level problem on the folded value f = |t - 1.5|: a is the mean of f
#   over the inner cell (f <= m), b over the outer cell (f > m).  It starts
#   from the uniform levels and stops once the cells repeat, so the result is
#   a fixed point: each level is the centroid of its cell.  Groups with a zero
#   scale (all codes 0) carry no t and are left out.

UNIFORM_CODEBOOK = (0.5, 1.5)


def codebook_levels(a: float, b: float) -> np.ndarray:
    """The four levels of t for codes 0..3, float64."""
    return np.array([1.5 - b, 1.5 - a, 1.5 + a, 1.5 + b], dtype=np.float64)


def codebook_thresholds(a: float, b: float):
    """(lower, upper) float32 thresholds 1.5 -/+ m, m = (a + b)/2 in float32."""
    m = np.float32(np.float32(np.float32(a) + np.float32(b)) * np.float32(0.5))
    return np.float32(np.float32(1.5) - m), np.float32(np.float32(1.5) + m)


def codes_from_t(t, a: float, b: float) -> np.ndarray:
    """Nearest symmetric level for float32 t, ties to the even code."""
    t = np.asarray(t, dtype=np.float32)
    lo, hi = codebook_thresholds(a, b)
    return ((t > lo).astype(np.uint8) + (t >= np.float32(1.5)).astype(np.uint8) + (t > hi).astype(np.uint8))


def group_t(x, clip: float):
    """(t, s, z) of one group: the uniform quantiser's scale, zero point and
    float32 normalised values; t is None when the scale is zero."""
    x = np.asarray(x, dtype=np.float32)
    c = np.float32(clip)
    mx_c = np.float32(c * np.float32(x.max()))
    mn_c = np.float32(c * np.float32(x.min()))
    s = half_rn_sat(np.float32(np.float32(mx_c - mn_c) / np.float32(3.0)))
    z = half_rn_sat(mn_c)
    if np.float32(s) == 0:
        return None, s, z
    t = (x - np.float32(z)) / np.float32(s)
    assert t.dtype == np.float32
    return t, s, z


def quantize_group_codebook(x, clip: float, a: float, b: float):
    """One group -> (codes, s, z) with the symmetric codebook (a, b)."""
    t, s, z = group_t(x, clip)
    if t is None:
        return np.zeros(np.shape(x), dtype=np.uint8), s, z
    return codes_from_t(t, a, b), s, z


def quantize_vector_codebook(x, g: int, clip: float, a: float, b: float):
    """A rotated d-vector -> codes [d], s [d/g], z [d/g] with the codebook."""
    x = np.asarray(x, dtype=np.float32)
    d = x.shape[0]
    codes = np.zeros(d, dtype=np.uint8)
    s = np.zeros(d // g, dtype=np.float16)
    z = np.zeros(d // g, dtype=np.float16)
    for gr in range(d // g):
        c, si, zi = quantize_group_codebook(x[gr * g:(gr + 1) * g], clip, a, b)
        codes[gr * g:(gr + 1) * g] = c
        s[gr] = si
        z[gr] = zi
    return codes, s, z


def dequantize_codebook(codes, s, z, g: int, a: float, b: float) -> np.ndarray:
    """x_hat = level[code]*s + z per group, float64."""
    lv = codebook_levels(float(np.float32(a)), float(np.float32(b)))[np.asarray(codes, dtype=np.int64)]
    sg = np.repeat(np.asarray(s, dtype=np.float64), g, axis=-1)
    zg = np.repeat(np.asarray(z, dtype=np.float64), g, axis=-1)
    return lv * sg + zg


def folded_values(X, g: int, clip: float) -> np.ndarray:
    """f = |t - 1.5| (float32 subtraction) of every channel of every row of
    rotated float32 X [n][d], groups with a zero scale left out."""
    X = np.asarray(X, dtype=np.float32)
    out = []
    for n in range(X.shape[0]):
        for gr in range(X.shape[1] // g):
            t, _, _ = group_t(X[n, gr * g:(gr + 1) * g], clip)
            if t is not None:
                out.append(np.abs(t - np.float32(1.5)))
    return np.concatenate(out) if out else np.zeros(0, dtype=np.float32)


def lloyd_max_folded(f, max_iters: int = 100):
    """Two-level Lloyd-Max on folded values f >= 0, float64.

    Returns (a, b, updates): the inner and outer levels and how many centroid
    updates ran before the cells repeated (or max_iters)."""
    f = np.asarray(f, dtype=np.float64)
    a, b = UNIFORM_CODEBOOK
    prev = -1
    updates = 0
    for _ in range(max_iters):
        m = (a + b) / 2.0
        inner = f <= m
        n_in = int(np.count_nonzero(inner))
        if n_in == prev:
            break  # same cells as last time: a and b are their centroids
        if n_in > 0:
            a = float(np.sum(f[inner])) / n_in
        if n_in < f.size:
            b = float(np.sum(f[~inner])) / (f.size - n_in)
        prev = n_in
        updates += 1
    return a, b, updates


def fit_codebook(X_rot, g: int, clip: float, max_iters: int = 100):
    """The codebook (a, b) of one (layer, kv head, K or V) from rotated float32
    calibration rows, with the head's clip ratio."""
    return lloyd_max_folded(folded_values(X_rot, g, clip), max_iters)
