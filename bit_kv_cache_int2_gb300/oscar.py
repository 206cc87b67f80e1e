"""Python binding of liboscar's C ABI (argument marshalling only).

Every function here has the name of the C entry point it calls and does no
computation of its own: it turns torch tensors into device pointers, streams
into ``cudaStream_t`` handles and non-OK statuses into ``OscarError``.  All
work runs in the CUDA library.  If the library is missing this module raises;
there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
# the in-tree build; OSCAR_LIBRARY names another build of the same library
# (for example one compiled with different options) to load instead
LIB_PATH = os.environ.get("OSCAR_LIBRARY") or os.path.join(PKG, "liboscar.so")

HEAD_DIM = 128
PAGE_SIZE = 64
SINK_TOKENS = 64
RECENT_TOKENS = 256

OK = 0
ERR_INVALID_ARG = 1
ERR_UNSUPPORTED = 2
ERR_NO_PAGE = 3
ERR_RANGE = 4
ERR_TIMEOUT = 5
ERR_CUDA = 6
ERR_STATE = 7
ERR_TOO_LARGE = 8
NOALLOC_SCRATCH_BYTES = 8 << 20
CODEBOOK_MAX_ROWS = 1 << 20
UNIFORM_CODEBOOK = (0.5, 1.5)  # (a, b) of the levels {0, 1, 2, 3}

ROT_OSCAR = 0
ROT_HADAMARD = 1
ROT_NONE = 2

OPT_DECODE_IMPL = 0
DECODE_TENSOR = 0  # tensor cores; two pages per tile at G <= 4
DECODE_CUDA_CORE = 1
DECODE_TENSOR_SINGLE = 2  # tensor cores, one page per tile
DECODE_TCGEN05 = 3  # tcgen05.mma, codes unpacked into tensor memory, one CTA per SM
OPT_CTAS_PER_SM = 1
OPT_ITEMS_PER_CTA = 2
OPT_PREFILL_IMPL = 3
PREFILL_TCGEN05 = 0  # tcgen05.mma, S/P/O in tensor memory
PREFILL_MMA_SYNC = 1  # mma.sync
OPT_WAIT_POLLS = 4  # poll budget of each history page's first wait in the decode kernel
OPT_DECODE_PARTITION = 5  # 0 automatic, 1 item list, 2 balanced
PARTITION_AUTO, PARTITION_ITEMS, PARTITION_BALANCED = 0, 1, 2
WAIT_POLLS_DEFAULT = 1 << 22


class OscarError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


class oscar_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "num_layers", "num_q_heads", "num_kv_heads", "head_dim", "group_size", "page_size",
        "sink_tokens", "recent_tokens", "max_batch", "max_pages_per_req", "num_pages")]


class oscar_layout_info(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in (
        "int2_head_bytes", "int2_page_bytes", "off_k_codes", "off_v_codes", "off_k_sz", "off_v_sz",
        "bf16_head_bytes", "bf16_page_bytes", "sink_bytes", "ring_bytes", "decode_scratch_bytes",
        "prefill_scratch_bytes")]


class oscar_cache(ctypes.Structure):
    _fields_ = [("pool", ctypes.c_void_p), ("page_table", ctypes.c_void_p),
                ("sink_k", ctypes.c_void_p), ("sink_v", ctypes.c_void_p),
                ("ring_k", ctypes.c_void_p), ("ring_v", ctypes.c_void_p),
                ("seq_lens", ctypes.c_void_p), ("hist_lens", ctypes.c_void_p)]


_lib = None

_SIGS = {
    "oscar_version": ([], ctypes.c_int),
    "oscar_status_string": ([ctypes.c_int], ctypes.c_char_p),
    "oscar_layout": ([ctypes.POINTER(oscar_config), ctypes.POINTER(oscar_layout_info)], ctypes.c_int),
    "oscar_create": ([ctypes.POINTER(oscar_config), ctypes.POINTER(ctypes.c_void_p)], ctypes.c_int),
    "oscar_destroy": ([ctypes.c_void_p], ctypes.c_int),
    "oscar_set_option": ([ctypes.c_void_p, ctypes.c_int, ctypes.c_int], ctypes.c_int),
    "oscar_set_rotation": ([ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p], ctypes.c_int),
    "oscar_append": ([ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(oscar_cache), ctypes.c_void_p,
                      ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p], ctypes.c_int),
    "oscar_demote": ([ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(oscar_cache), ctypes.c_int,
                      ctypes.c_void_p], ctypes.c_int),
    "oscar_import_tokens": ([ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(oscar_cache), ctypes.c_void_p,
                             ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p], ctypes.c_int),
    "oscar_decode": ([ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(oscar_cache), ctypes.c_void_p,
                      ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int,
                      ctypes.c_void_p], ctypes.c_int),
    "oscar_decode_noalloc": ([ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(oscar_cache), ctypes.c_void_p,
                              ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p], ctypes.c_int),
    "oscar_decode_bf16_history": ([ctypes.c_void_p, ctypes.POINTER(oscar_cache), ctypes.c_void_p,
                                   ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                                   ctypes.c_int, ctypes.c_void_p], ctypes.c_int),
    "oscar_import_bf16_history": ([ctypes.c_void_p, ctypes.POINTER(oscar_cache), ctypes.c_void_p,
                                   ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p], ctypes.c_int),
    "oscar_quantize_rotated_f32": ([ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_float, ctypes.c_int,
                                    ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p], ctypes.c_int),
    "oscar_debug_rotate": ([ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                            ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p], ctypes.c_int),
    "oscar_get_error": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.POINTER(ctypes.c_int)], ctypes.c_int),
    "oscar_last_cuda_error": ([], ctypes.c_int),
    "oscar_decode_step": ([ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(oscar_cache), ctypes.c_void_p, ctypes.c_void_p,
                           ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                           ctypes.c_int, ctypes.c_void_p], ctypes.c_int),
    "oscar_prefill": ([ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(oscar_cache), ctypes.c_void_p, ctypes.c_void_p,
                       ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                       ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p], ctypes.c_int),
    "oscar_append_bf16_history": ([ctypes.c_void_p, ctypes.POINTER(oscar_cache), ctypes.c_void_p, ctypes.c_void_p,
                                   ctypes.c_int, ctypes.c_void_p], ctypes.c_int),
    "oscar_calibration_scratch_bytes": ([ctypes.c_int, ctypes.c_int, ctypes.c_int], ctypes.c_size_t),
    "oscar_calibrate": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                         ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                         ctypes.c_size_t, ctypes.c_void_p], ctypes.c_int),
    "oscar_clip_errors": ([ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                           ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                           ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                           ctypes.c_void_p], ctypes.c_int),
    "oscar_set_codebook": ([ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p],
                           ctypes.c_int),
    "oscar_codebook_scratch_bytes": ([ctypes.c_int], ctypes.c_size_t),
    "oscar_fit_codebook": ([ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_int,
                            ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p,
                            ctypes.POINTER(ctypes.c_int), ctypes.c_void_p], ctypes.c_int),
    "oscar_quantize_codebook_f32": ([ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_float, ctypes.c_float,
                                     ctypes.c_float, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p],
                                    ctypes.c_int),
    "oscar_check_cache_host": ([ctypes.POINTER(oscar_config), ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                ctypes.c_int, ctypes.POINTER(ctypes.c_int)], ctypes.c_int),
    "oscar_profile_enable": ([ctypes.c_void_p, ctypes.c_int], ctypes.c_int),
    "oscar_profile_read": ([ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(ctypes.c_int),
                            ctypes.POINTER(ctypes.c_double), ctypes.c_int], ctypes.c_int),
}

KERNEL_APPEND = 0
KERNEL_IMPORT = 1
KERNEL_DECODE_PREP = 2
KERNEL_DECODE_MAIN = 3
KERNEL_DECODE_MERGE = 4
KERNEL_STEP = 5
KERNEL_PREFILL_PREP = 6
KERNEL_PREFILL_ATTN = 7
KERNEL_PREFILL_MERGE = 8
KERNEL_NAMES = {0: "append", 1: "import", 2: "decode_prep", 3: "decode_main", 4: "decode_merge", 5: "step_append_prep",
                6: "prefill_prep", 7: "prefill_attn", 8: "prefill_merge"}


def exported_symbols():
    return list(_SIGS)


def lib():
    """Load liboscar.so (built in-tree by ``bit_kv_cache_int2_gb300.build``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with bit_kv_cache_int2_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in _SIGS.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def _check(st: int, where: str):
    if st != OK:
        if st == ERR_CUDA:
            where = f"{where} [cudaError {lib().oscar_last_cuda_error()}]"
        raise OscarError(st, where)


def _ptr(t):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch

        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def status_string(st: int) -> str:
    try:
        return lib().oscar_status_string(st).decode()
    except RuntimeError:
        return f"status {st}"


def oscar_version() -> int:
    return lib().oscar_version()


def make_config(num_layers=1, num_q_heads=32, num_kv_heads=8, group_size=128, max_batch=1,
                max_pages_per_req=1, num_pages=1) -> oscar_config:
    return oscar_config(num_layers, num_q_heads, num_kv_heads, HEAD_DIM, group_size, PAGE_SIZE,
                        SINK_TOKENS, RECENT_TOKENS, max_batch, max_pages_per_req, num_pages)


def oscar_layout(cfg: oscar_config) -> oscar_layout_info:
    info = oscar_layout_info()
    _check(lib().oscar_layout(ctypes.byref(cfg), ctypes.byref(info)), "oscar_layout")
    return info


def oscar_create(cfg: oscar_config) -> ctypes.c_void_p:
    h = ctypes.c_void_p()
    _check(lib().oscar_create(ctypes.byref(cfg), ctypes.byref(h)), "oscar_create")
    return h


def oscar_destroy(ctx):
    _check(lib().oscar_destroy(ctx), "oscar_destroy")


def oscar_set_option(ctx, option: int, value: int):
    _check(lib().oscar_set_option(ctx, option, value), "oscar_set_option")


def oscar_set_rotation(ctx, layer, U_K, U_V, clip_k, clip_v, rot_mode=ROT_OSCAR, stream=None):
    """U_K, U_V: host float32 [Hkv][128][128] (numpy or CPU tensor) or None; clips: host float32 [Hkv]."""
    import numpy as np

    def host(a):
        if a is None:
            return None, None
        a = np.ascontiguousarray(np.asarray(a, dtype=np.float32))
        return a, a.ctypes.data_as(ctypes.c_void_p)

    uk, puk = host(U_K)
    uv, puv = host(U_V)
    ck, pck = host(clip_k)
    cv, pcv = host(clip_v)
    _check(lib().oscar_set_rotation(ctx, layer, puk, puv, pck, pcv, rot_mode, _stream(stream)),
           "oscar_set_rotation")


def _cache_struct(c: dict) -> oscar_cache:
    return oscar_cache(*(c[k].data_ptr() if c.get(k) is not None else None for k in
                         ("pool", "page_table", "sink_k", "sink_v", "ring_k", "ring_v", "seq_lens", "hist_lens")))


def oscar_append(ctx, layer, cache: dict, k_new, v_new, batch, stream=None):
    cs = _cache_struct(cache)
    _check(lib().oscar_append(ctx, layer, ctypes.byref(cs), _ptr(k_new), _ptr(v_new), batch, _stream(stream)),
           "oscar_append")


def oscar_demote(ctx, layer, cache: dict, batch, stream=None):
    cs = _cache_struct(cache)
    _check(lib().oscar_demote(ctx, layer, ctypes.byref(cs), batch, _stream(stream)), "oscar_demote")


def oscar_import_tokens(ctx, layer, cache: dict, K, V, batch, n, stream=None):
    cs = _cache_struct(cache)
    _check(lib().oscar_import_tokens(ctx, layer, ctypes.byref(cs), _ptr(K), _ptr(V), batch, n, _stream(stream)),
           "oscar_import_tokens")


def oscar_decode(ctx, layer, cache: dict, q, out, lse, scratch, batch, stream=None):
    cs = _cache_struct(cache)
    _check(lib().oscar_decode(ctx, layer, ctypes.byref(cs), _ptr(q), _ptr(out), _ptr(lse), _ptr(scratch),
                              scratch.numel() * scratch.element_size(), batch, _stream(stream)),
           "oscar_decode")


def oscar_append_bf16_history(ctx, cache: dict, k_new, v_new, batch, stream=None):
    cs = _cache_struct(cache)
    _check(lib().oscar_append_bf16_history(ctx, ctypes.byref(cs), _ptr(k_new), _ptr(v_new), batch, _stream(stream)),
           "oscar_append_bf16_history")


def calibration_scratch(G, N, M=0, device="cuda"):
    import torch

    n = lib().oscar_calibration_scratch_bytes(G, N, M)
    return torch.empty((n + 255) // 256 * 256, dtype=torch.uint8, device=device)


def _np_ptr(a):
    return ctypes.c_void_p(a.ctypes.data)


def oscar_calibrate(ctx, Q, K, V, N, scratch, stream=None):
    """Q device bf16 [G][N][128]; K, V device bf16 [N][128].  Returns host
    (U_K, U_V) float32 [128][128] and (C_Q, C_S) float64 [128][128]."""
    import numpy as np

    U_K = np.zeros((128, 128), dtype=np.float32)
    U_V = np.zeros((128, 128), dtype=np.float32)
    C_Q = np.zeros((128, 128), dtype=np.float64)
    C_S = np.zeros((128, 128), dtype=np.float64)
    _check(lib().oscar_calibrate(ctx, _ptr(Q), _ptr(K), _ptr(V), N, _np_ptr(U_K), _np_ptr(U_V), _np_ptr(C_Q),
                                 _np_ptr(C_S), _ptr(scratch), scratch.numel() * scratch.element_size(),
                                 _stream(stream)), "oscar_calibrate")
    return U_K, U_V, C_Q, C_S


def oscar_clip_errors(ctx, layer, kv_head, Q, K, V, N, ratios, scratch, stream=None):
    """Errors of each candidate clip ratio for keys and values with the layer's
    loaded rotation.  Returns (err_k, err_v, best_k, best_v)."""
    import numpy as np

    r = np.ascontiguousarray(ratios, dtype=np.float32)
    M = len(r)
    ek = np.zeros(M, dtype=np.float64)
    ev = np.zeros(M, dtype=np.float64)
    bk, bv = ctypes.c_int(0), ctypes.c_int(0)
    _check(lib().oscar_clip_errors(ctx, layer, kv_head, _ptr(Q), _ptr(K), _ptr(V), N, _np_ptr(r), M, _np_ptr(ek),
                                   _np_ptr(ev), ctypes.byref(bk), ctypes.byref(bv), _ptr(scratch),
                                   scratch.numel() * scratch.element_size(), _stream(stream)), "oscar_clip_errors")
    return ek, ev, bk.value, bv.value


def oscar_set_codebook(ctx, layer, k_ab=None, v_ab=None, stream=None):
    """Lloyd-Max codebooks of a layer: k_ab, v_ab [Hkv][2] (a, b) pairs, or
    None for the uniform levels."""
    import numpy as np

    k = None if k_ab is None else np.ascontiguousarray(k_ab, dtype=np.float32)
    v = None if v_ab is None else np.ascontiguousarray(v_ab, dtype=np.float32)
    _check(lib().oscar_set_codebook(ctx, layer, None if k is None else _np_ptr(k), None if v is None else _np_ptr(v),
                                    _stream(stream)), "oscar_set_codebook")


def codebook_scratch(N, device="cuda"):
    import torch

    n = lib().oscar_codebook_scratch_bytes(N)
    if n == 0:
        raise OscarError(ERR_INVALID_ARG, "codebook_scratch")
    return torch.empty((n + 255) // 256 * 256, dtype=torch.uint8, device=device)


def oscar_fit_codebook(ctx, layer, kv_head, which, X, N, scratch, max_iters=100, stream=None):
    """Lloyd-Max fit of one (layer, kv head) for keys (which=0) or values
    (which=1).  Returns (a, b, updates)."""
    import numpy as np

    ab = np.zeros(2, dtype=np.float32)
    up = ctypes.c_int(0)
    _check(lib().oscar_fit_codebook(ctx, layer, kv_head, which, _ptr(X), N, max_iters, _ptr(scratch),
                                    scratch.numel() * scratch.element_size(), _np_ptr(ab), ctypes.byref(up),
                                    _stream(stream)), "oscar_fit_codebook")
    return float(ab[0]), float(ab[1]), up.value


def oscar_prefill(ctx, layer, cache: dict, q, k, v, T, out, lse, scratch, batch, stream=None):
    """Chunked prefill: T new tokens per request attend to the cache and
    causally to each other (the chunk is not stored)."""
    cs = _cache_struct(cache)
    _check(lib().oscar_prefill(ctx, layer, ctypes.byref(cs), _ptr(q), _ptr(k), _ptr(v), T, _ptr(out), _ptr(lse),
                               _ptr(scratch), scratch.numel() * scratch.element_size(), batch, _stream(stream)),
           "oscar_prefill")


def oscar_decode_step(ctx, layer, cache: dict, k_new, v_new, q, out, lse, scratch, batch, stream=None):
    """oscar_append(k_new, v_new) then oscar_decode(q), with the query rotation
    run beside the append."""
    cs = _cache_struct(cache)
    _check(lib().oscar_decode_step(ctx, layer, ctypes.byref(cs), _ptr(k_new), _ptr(v_new), _ptr(q), _ptr(out),
                                   _ptr(lse), _ptr(scratch), scratch.numel() * scratch.element_size(), batch,
                                   _stream(stream)), "oscar_decode_step")


def bind_decode_step(ctx, layer, cache: dict, q, out, lse, scratch, batch, stream=None):
    """oscar_decode_step with everything but the new tokens marshalled once:
    returns f(k_new_ptr, v_new_ptr) taking raw device addresses (ints)."""
    cs = _cache_struct(cache)
    head = (ctx, layer, ctypes.byref(cs))
    tail = (_ptr(q), _ptr(out), _ptr(lse), _ptr(scratch), scratch.numel() * scratch.element_size(), batch,
            _stream(stream))
    fn = lib().oscar_decode_step

    def call(k_ptr: int, v_ptr: int):
        _check(fn(*head, ctypes.c_void_p(k_ptr), ctypes.c_void_p(v_ptr), *tail), "oscar_decode_step")

    call._keep = cs
    return call


def bind_decode_step_ptrs(ctx, layer, cache: dict, out, lse, scratch, batch, stream=None):
    """As bind_decode_step, with q passed per call too: returns
    f(k_new_ptr, v_new_ptr, q_ptr) taking raw addresses (ints) of device or
    pinned host memory."""
    cs = _cache_struct(cache)
    head = (ctx, layer, ctypes.byref(cs))
    tail = (_ptr(out), _ptr(lse), _ptr(scratch), scratch.numel() * scratch.element_size(), batch, _stream(stream))
    fn = lib().oscar_decode_step

    def call(k_ptr: int, v_ptr: int, q_ptr: int):
        _check(fn(*head, ctypes.c_void_p(k_ptr), ctypes.c_void_p(v_ptr), ctypes.c_void_p(q_ptr), *tail),
               "oscar_decode_step")

    call._keep = cs
    return call


def bind_step_any_batch(ctx, layer, cache: dict, out, lse, scratch, bf16_history=False, stream=None):
    """One decode step with the cache and outputs marshalled once and the
    batch given per call: returns f(k_ptr, v_ptr, q_ptr, batch) taking raw
    addresses.  INT2 history: oscar_decode_step; BF16 history:
    oscar_append_bf16_history then oscar_decode_bf16_history."""
    cs = _cache_struct(cache)
    L = lib()
    st = _stream(stream)
    o, ls, sc, nb = _ptr(out), _ptr(lse), _ptr(scratch), scratch.numel() * scratch.element_size()
    P = ctypes.c_void_p
    if not bf16_history:
        fn = L.oscar_decode_step

        def call(k_ptr: int, v_ptr: int, q_ptr: int, batch: int):
            _check(fn(ctx, layer, ctypes.byref(cs), P(k_ptr), P(v_ptr), P(q_ptr), o, ls, sc, nb, batch, st),
                   "oscar_decode_step")
    else:
        fa, fd = L.oscar_append_bf16_history, L.oscar_decode_bf16_history

        def call(k_ptr: int, v_ptr: int, q_ptr: int, batch: int):
            _check(fa(ctx, ctypes.byref(cs), P(k_ptr), P(v_ptr), batch, st), "oscar_append_bf16_history")
            _check(fd(ctx, ctypes.byref(cs), P(q_ptr), o, ls, sc, nb, batch, st), "oscar_decode_bf16_history")

    call._keep = cs
    return call


def bind_append(ctx, layer, cache: dict, batch, stream=None):
    """oscar_append with the cache and stream marshalled once, for tight loops:
    returns f(k_new_ptr, v_new_ptr) taking raw device addresses (ints)."""
    cs = _cache_struct(cache)
    csr, st, fn = ctypes.byref(cs), _stream(stream), lib().oscar_append

    def call(k_ptr: int, v_ptr: int):
        _check(fn(ctx, layer, csr, ctypes.c_void_p(k_ptr), ctypes.c_void_p(v_ptr), batch, st), "oscar_append")

    call._keep = cs  # the struct must outlive the closure's byref
    return call


def bind_decode(ctx, layer, cache: dict, q, out, lse, scratch, batch, stream=None):
    """oscar_decode with every argument marshalled once, for tight loops:
    returns a no-argument callable."""
    cs = _cache_struct(cache)
    args = (ctx, layer, ctypes.byref(cs), _ptr(q), _ptr(out), _ptr(lse), _ptr(scratch),
            scratch.numel() * scratch.element_size(), batch, _stream(stream))
    fn = lib().oscar_decode

    def call():
        _check(fn(*args), "oscar_decode")

    call._keep = cs
    return call


def oscar_decode_noalloc(ctx, layer, cache: dict, q, out, lse, batch, stream=None):
    """oscar_decode with the library's own built-in working memory: the caller
    passes no scratch and nothing is allocated."""
    cs = _cache_struct(cache)
    _check(lib().oscar_decode_noalloc(ctx, layer, ctypes.byref(cs), _ptr(q), _ptr(out), _ptr(lse), batch,
                                      _stream(stream)), "oscar_decode_noalloc")


def oscar_decode_bf16_history(ctx, cache: dict, q, out, lse, scratch, batch, stream=None):
    cs = _cache_struct(cache)
    _check(lib().oscar_decode_bf16_history(ctx, ctypes.byref(cs), _ptr(q), _ptr(out), _ptr(lse), _ptr(scratch),
                                           scratch.numel() * scratch.element_size(), batch, _stream(stream)),
           "oscar_decode_bf16_history")


def oscar_import_bf16_history(ctx, cache: dict, K, V, batch, n, stream=None):
    cs = _cache_struct(cache)
    _check(lib().oscar_import_bf16_history(ctx, ctypes.byref(cs), _ptr(K), _ptr(V), batch, n, _stream(stream)),
           "oscar_import_bf16_history")


def oscar_quantize_rotated_f32(x, group_size, clip, which, codes, sz, stream=None):
    _check(lib().oscar_quantize_rotated_f32(_ptr(x), x.shape[0], group_size, float(clip), which, _ptr(codes),
                                            _ptr(sz), _stream(stream)), "oscar_quantize_rotated_f32")


def check_cache(cfg, cache: dict, batch: int):
    """Debug aid: copies the cache's lengths and page table to the host and
    checks them (oscar_check_cache_host).  Returns (status, first bad request
    or -1); status OK when the state is consistent."""
    import numpy as np

    seq = np.ascontiguousarray(cache["seq_lens"].cpu().numpy(), dtype=np.int32)
    hist = np.ascontiguousarray(cache["hist_lens"].cpu().numpy(), dtype=np.int32)
    pt = np.ascontiguousarray(cache["page_table"].cpu().numpy(), dtype=np.int32)
    bad = ctypes.c_int(-1)
    st = lib().oscar_check_cache_host(ctypes.byref(cfg), _np_ptr(seq), _np_ptr(hist), _np_ptr(pt), batch,
                                      ctypes.byref(bad))
    return st, bad.value


def oscar_quantize_codebook_f32(x, group_size, clip, a, b, which, codes, sz, stream=None):
    _check(lib().oscar_quantize_codebook_f32(_ptr(x), x.shape[0], group_size, float(clip), float(a), float(b), which,
                                             _ptr(codes), _ptr(sz), _stream(stream)), "oscar_quantize_codebook_f32")


def oscar_debug_rotate(ctx, layer, which, kv_head, x, x_rot, stream=None):
    _check(lib().oscar_debug_rotate(ctx, layer, which, kv_head, _ptr(x), _ptr(x_rot), x.shape[0], _stream(stream)),
           "oscar_debug_rotate")


def oscar_get_error(ctx, stream=None) -> int:
    code = ctypes.c_int(0)
    _check(lib().oscar_get_error(ctx, _stream(stream), ctypes.byref(code)), "oscar_get_error")
    return code.value


def oscar_profile_enable(ctx, enable: bool):
    _check(lib().oscar_profile_enable(ctx, 1 if enable else 0), "oscar_profile_enable")


def oscar_profile_read(ctx, kernel_id: int, reset: bool = False):
    """(launches, total_ms) of one kernel since the last reset."""
    n = ctypes.c_int(0)
    ms = ctypes.c_double(0.0)
    _check(lib().oscar_profile_read(ctx, kernel_id, ctypes.byref(n), ctypes.byref(ms), 1 if reset else 0),
           "oscar_profile_read")
    return n.value, ms.value


# ---------------------------------------------------------------- plumbing
def alloc_cache(cfg: oscar_config, device="cuda", bf16_history=False, zero=True):
    """Device buffers of one layer's cache (torch allocations, caller-owned)."""
    import torch

    info = oscar_layout(cfg)
    page_bytes = info.bf16_page_bytes if bf16_history else info.int2_page_bytes
    mk = torch.zeros if zero else torch.empty
    B, Hkv = cfg.max_batch, cfg.num_kv_heads
    return {
        "pool": mk(cfg.num_pages * page_bytes, dtype=torch.uint8, device=device),
        "page_table": torch.full((B, cfg.max_pages_per_req), -1, dtype=torch.int32, device=device),
        "sink_k": mk(B, Hkv, SINK_TOKENS, HEAD_DIM, dtype=torch.bfloat16, device=device),
        "sink_v": mk(B, Hkv, SINK_TOKENS, HEAD_DIM, dtype=torch.bfloat16, device=device),
        "ring_k": mk(B, Hkv, RECENT_TOKENS, HEAD_DIM, dtype=torch.bfloat16, device=device),
        "ring_v": mk(B, Hkv, RECENT_TOKENS, HEAD_DIM, dtype=torch.bfloat16, device=device),
        "seq_lens": torch.zeros(B, dtype=torch.int32, device=device),
        "hist_lens": torch.zeros(B, dtype=torch.int32, device=device),
    }


def alloc_scratch(cfg: oscar_config, device="cuda", prefill=False):
    import torch

    info = oscar_layout(cfg)
    n = info.prefill_scratch_bytes if prefill else info.decode_scratch_bytes
    return torch.empty((n + 255) // 256 * 256, dtype=torch.uint8, device=device)
