"""C-ABI checks that need no GPU: the library builds, loads, exports every
symbol include/oscar.h declares, and rejects bad arguments on the host."""
import ctypes
import os
import re
import subprocess

import pytest

from bit_kv_cache_int2_gb300 import build as B
from bit_kv_cache_int2_gb300 import oscar

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return oscar.lib()


def header_functions():
    with open(os.path.join(ROOT, "include", "oscar.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:oscar_status|int|size_t|const char\*)\s+(oscar_\w+)\s*\(", text, re.M)))


def test_header_declares_the_boundary():
    names = header_functions()
    for n in ("oscar_create", "oscar_destroy", "oscar_layout", "oscar_set_rotation", "oscar_append",
              "oscar_demote", "oscar_import_tokens", "oscar_decode", "oscar_decode_bf16_history",
              "oscar_quantize_rotated_f32", "oscar_debug_rotate", "oscar_get_error"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", oscar.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (oscar_\w+)", out))
    for n in header_functions():
        assert n in exported, n
        assert hasattr(lib, n)
    assert set(oscar.exported_symbols()) <= exported


def test_version_and_status_strings(lib):
    assert oscar.oscar_version() >= 10000
    assert oscar.status_string(oscar.OK) == "ok"
    assert "page" in oscar.status_string(oscar.ERR_NO_PAGE)


@pytest.mark.parametrize("g,head", [(128, 4608), (64, 5120), (32, 6144)])
def test_layout_sizes(lib, g, head):
    cfg = oscar.make_config(1, 32, 8, g, max_batch=4, max_pages_per_req=100, num_pages=400)
    info = oscar.oscar_layout(cfg)
    assert info.int2_head_bytes == head
    assert info.int2_page_bytes == 8 * head
    assert (info.off_k_codes, info.off_v_codes, info.off_k_sz) == (0, 2048, 4096)
    assert info.off_v_sz == 4096 + 64 * (128 // g) * 4
    assert info.bf16_head_bytes == 32768
    assert info.sink_bytes == 4 * 8 * 64 * 128 * 2
    assert info.ring_bytes == 4 * 8 * 256 * 128 * 2
    assert info.decode_scratch_bytes > 4 * 32 * 128 * 4


def test_layout_rejects_unsupported(lib):
    for kw, st in ((dict(group_size=16), oscar.ERR_UNSUPPORTED), (dict(num_q_heads=48), oscar.ERR_UNSUPPORTED),
                   (dict(num_q_heads=30), oscar.ERR_INVALID_ARG), (dict(max_batch=0), oscar.ERR_INVALID_ARG)):
        args = dict(num_layers=1, num_q_heads=32, num_kv_heads=8, group_size=128, max_batch=1,
                    max_pages_per_req=1, num_pages=1)
        args.update(kw)
        with pytest.raises(oscar.OscarError) as e:
            oscar.oscar_layout(oscar.make_config(**args))
        assert e.value.status == st
    cfg = oscar.make_config()
    cfg.head_dim = 64
    with pytest.raises(oscar.OscarError) as e:
        oscar.oscar_layout(cfg)
    assert e.value.status == oscar.ERR_UNSUPPORTED


def test_null_and_bad_arguments_rejected_on_host(lib):
    L = lib
    cs = oscar.oscar_cache()
    assert L.oscar_decode(None, 0, ctypes.byref(cs), None, None, None, None, 0, 1, None) == oscar.ERR_INVALID_ARG
    assert L.oscar_append(None, 0, ctypes.byref(cs), None, None, 1, None) == oscar.ERR_INVALID_ARG
    assert L.oscar_destroy(None) == oscar.ERR_INVALID_ARG
    assert L.oscar_get_error(None, None, None) == oscar.ERR_INVALID_ARG
    assert L.oscar_set_option(None, 0, 0) == oscar.ERR_INVALID_ARG
    # quantiser hook validation happens before any device work
    fake = ctypes.c_void_p(256)
    assert L.oscar_quantize_rotated_f32(fake, 10, 16, 1.0, 0, fake, fake, None) == oscar.ERR_UNSUPPORTED
    assert L.oscar_quantize_rotated_f32(fake, 10, 128, 1.0, 1, fake, fake, None) == oscar.ERR_INVALID_ARG
    assert L.oscar_quantize_rotated_f32(fake, 64, 128, 1.5, 1, fake, fake, None) == oscar.ERR_INVALID_ARG
    assert L.oscar_quantize_rotated_f32(fake, 64, 128, 0.0, 0, fake, fake, None) == oscar.ERR_INVALID_ARG
    assert L.oscar_quantize_rotated_f32(None, 64, 128, 1.0, 0, fake, fake, None) == oscar.ERR_INVALID_ARG
    # codebook: pairs outside 0 <= a < b <= 3 (or not finite) are refused on the host
    for a, b in ((0.6, 0.5), (0.5, 3.5), (-0.1, 1.0), (float("nan"), 1.0), (0.5, float("inf"))):
        assert L.oscar_quantize_codebook_f32(fake, 64, 128, 1.0, a, b, 0, fake, fake, None) == oscar.ERR_INVALID_ARG
    assert L.oscar_quantize_codebook_f32(fake, 64, 16, 1.0, 0.5, 1.5, 0, fake, fake, None) == oscar.ERR_UNSUPPORTED
    assert L.oscar_set_codebook(None, 0, None, None, None) == oscar.ERR_INVALID_ARG
    assert L.oscar_fit_codebook(None, 0, 0, 0, fake, 4, 10, fake, 1 << 20, fake, None, None) == oscar.ERR_INVALID_ARG
    assert L.oscar_codebook_scratch_bytes(0) == 0
    assert L.oscar_codebook_scratch_bytes(oscar.CODEBOOK_MAX_ROWS + 1) == 0
    assert L.oscar_codebook_scratch_bytes(100) >= 100 * 128 * 4 + 24


def test_create_without_gpu_reports_cuda_error(lib):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(oscar.OscarError) as e:
        oscar.oscar_create(oscar.make_config())
    assert e.value.status == oscar.ERR_CUDA


def test_binding_fails_loudly_without_library(monkeypatch):
    monkeypatch.setattr(oscar, "_lib", None)
    monkeypatch.setattr(oscar, "LIB_PATH", "/nonexistent/liboscar.so")
    with pytest.raises(RuntimeError):
        oscar.lib()


def test_header_is_plain_c_and_the_library_is_callable_from_c(lib, tmp_path):
    """A C99 program (-pedantic -Werror) built against include/oscar.h and
    linked to liboscar.so calls the host-only entry points: the boundary needs
    neither C++ nor Python."""
    import shutil

    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "abi.c"
    src.write_text(r"""
#include <stdio.h>
#include <string.h>
#include "oscar.h"
int main(void) {
  oscar_config c = {0};
  oscar_layout_info info;
  if (oscar_version() < 10000) return 1;
  if (strcmp(oscar_status_string(OSCAR_OK), "ok") != 0) return 2;
  if (oscar_codebook_scratch_bytes(0) != 0) return 3;
  if (oscar_codebook_scratch_bytes(16) < (size_t)16 * 128 * 4) return 4;
  c.num_layers = 1; c.num_q_heads = 32; c.num_kv_heads = 8; c.head_dim = 128; c.group_size = 128;
  c.page_size = 64; c.sink_tokens = 64; c.recent_tokens = 256; c.max_batch = 2;
  c.max_pages_per_req = 100; c.num_pages = 200;
  if (oscar_layout(&c, &info) != OSCAR_OK) return 5;
  if (info.int2_head_bytes != 4608 || info.int2_page_bytes != 8 * 4608) return 6;
  c.group_size = 16;
  if (oscar_layout(&c, &info) != OSCAR_ERR_UNSUPPORTED) return 7;
  puts("abi ok");
  return 0;
}
""")
    exe = tmp_path / "abi"
    libdir = os.path.dirname(oscar.LIB_PATH)
    subprocess.run([gcc, "-std=c99", "-pedantic", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                    str(src), "-o", str(exe), oscar.LIB_PATH, f"-Wl,-rpath,{libdir}"], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and "abi ok" in r.stdout, (r.returncode, r.stdout, r.stderr)


def _state(B, mpr, pages_of, L, H):
    import torch

    pt = torch.full((B, mpr), -1, dtype=torch.int32)
    for b, ids in enumerate(pages_of):
        pt[b, :len(ids)] = torch.tensor(ids, dtype=torch.int32)
    return {"seq_lens": torch.tensor(L, dtype=torch.int32), "hist_lens": torch.tensor(H, dtype=torch.int32),
            "page_table": pt}


def test_cache_state_check_on_host(lib):
    """oscar_check_cache_host: lengths within the three-region rules, page
    ids present, in range and owned by one history slot only."""
    cfg = oscar.make_config(1, 8, 2, 128, max_batch=3, max_pages_per_req=4, num_pages=8)
    ok = _state(3, 4, [[5, 1], [0], []], [320 + 100, 320 + 64, 200], [100, 64, 0])
    assert oscar.check_cache(cfg, ok, 3) == (oscar.OK, -1)
    # demotes shrink the window: history up to L - 64 is still consistent
    assert oscar.check_cache(cfg, _state(1, 4, [[2, 3, 4]], [200], [136]), 1) == (oscar.OK, -1)
    cases = [
        (_state(2, 4, [[1, 3], [2]], [420, 1000], [100, 600]), (oscar.ERR_STATE, 1)),     # history too short
        (_state(1, 4, [[1, 2, 3]], [200], [137]), (oscar.ERR_STATE, 0)),                  # more than L - 64
        (_state(1, 4, [[1, -1]], [320 + 100], [100]), (oscar.ERR_NO_PAGE, 0)),            # missing page
        (_state(1, 4, [[1, 8]], [320 + 100], [100]), (oscar.ERR_RANGE, 0)),               # id out of range
        (_state(2, 4, [[1, 2], [2]], [420, 330], [100, 10]), (oscar.ERR_RANGE, 1)),       # page shared
        (_state(1, 4, [[1, 1]], [420], [100]), (oscar.ERR_RANGE, 0)),                     # page twice
        (_state(1, 4, [[0, 1, 2, 3]], [320 + 4 * 64 + 1], [4 * 64 + 1]), (oscar.ERR_RANGE, 0)),  # > max pages
        (_state(1, 4, [[]], [-1], [0]), (oscar.ERR_STATE, 0)),
    ]
    for st, want in cases:
        assert oscar.check_cache(cfg, st, st["seq_lens"].numel()) == want, want
    # entries beyond a request's history pages are not looked at
    assert oscar.check_cache(cfg, _state(1, 4, [[1, 7, 9, 9]], [320 + 70], [70]), 1) == (oscar.OK, -1)
