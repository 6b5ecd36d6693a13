"""The C ABI on the host, without a GPU: libmqa.so loads, exports every function include/mqa.h
declares, and rejects bad arguments with the documented status before any CUDA call."""
from __future__ import annotations

import ctypes
import math
import os
import re

import pytest

from query_grouped_decode_kv_b300 import build as mqa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mqa.h")

OK, INVALID, UNSUPPORTED, CUDA_ERR, BOUNDS, TIMEOUT = range(6)


@pytest.fixture(scope="module")
def lib():
    path = mqa_build.build()
    L = ctypes.CDLL(path)
    vp, i32 = ctypes.c_void_p, ctypes.c_int
    L.mqa_kv_append.restype = i32
    L.mqa_kv_append.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, vp]
    L.mqa_decode_attention.restype = i32
    L.mqa_decode_attention.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                       ctypes.c_float, vp]
    L.mqa_status_string.restype = ctypes.c_char_p
    L.mqa_get_device_status.restype = i32
    L.mqa_get_device_status.argtypes = [vp, ctypes.POINTER(i32)]
    L.mqa_debug_override.restype = i32
    L.mqa_debug_override.argtypes = [i32, i32]
    L.mqa_kernel_launch_count.restype = ctypes.c_uint64
    L.mqa_decode_step.restype = i32
    L.mqa_decode_step.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                  ctypes.c_float, vp]
    L.mqa_debug_timeout_site.restype = i32
    L.mqa_debug_timeout_site.argtypes = [vp]
    L.mqa_kv_append_paged.restype = i32
    L.mqa_kv_append_paged.argtypes = [vp, vp, vp, vp, vp, vp] + [i32] * 6 + [vp]
    L.mqa_decode_attention_paged.restype = i32
    L.mqa_decode_attention_paged.argtypes = [vp] * 6 + [i32] * 7 + [ctypes.c_float, vp]
    L.mqa_kv_append_fp8.restype = i32
    L.mqa_kv_append_fp8.argtypes = [vp] * 5 + [i32] * 4 + [ctypes.c_float] * 2 + [vp]
    L.mqa_decode_attention_fp8.restype = i32
    L.mqa_decode_attention_fp8.argtypes = [vp] * 5 + [i32] * 5 + [ctypes.c_float] * 3 + [vp]
    L.mqa_decode_step_fp8.restype = i32
    L.mqa_decode_step_fp8.argtypes = [vp] * 8 + [i32] * 5 + [ctypes.c_float] * 3 + [vp]
    L.mqa_kv_append_multi.restype = i32
    L.mqa_kv_append_multi.argtypes = [vp] * 5 + [i32] * 5 + [vp]
    L.mqa_decode_attention_multi.restype = i32
    L.mqa_decode_attention_multi.argtypes = [vp] * 5 + [i32] * 6 + [ctypes.c_float, vp]
    L.mqa_decode_step_multi.restype = i32
    L.mqa_decode_step_multi.argtypes = [vp] * 8 + [i32] * 6 + [ctypes.c_float, vp]
    L.mqa_decode_step_paged.restype = i32
    L.mqa_decode_step_paged.argtypes = [vp] * 9 + [i32] * 7 + [ctypes.c_float, vp]
    return L


def declared_functions() -> list[str]:
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mqa_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("mqa_kv_append", "mqa_decode_attention", "mqa_decode_step",
                     "mqa_status_string", "mqa_get_device_status"):
        assert required in names


def test_library_exports_every_declared_function(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in mqa.h but not exported"


def test_library_exports_nothing_undeclared():
    # the .so is built with hidden visibility: only the extern "C" ABI is exported
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", mqa_build.build()], check=True,
                         capture_output=True, text=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    mqa = {s for s in exported if s.startswith("mqa_")}
    assert mqa == set(declared_functions())


def test_status_strings(lib):
    for code in range(6):
        assert lib.mqa_status_string(code).decode().startswith("MQA_")
    assert lib.mqa_status_string(42) == b"unknown mqa status"


# fake, well-aligned device addresses: these calls must fail in the host checks, before CUDA
A = 0x7f0000000000


def _attn(lib, q=A, k=A + 0x1000, v=A + 0x2000, lens=A + 0x3000, out=A + 0x4000, b=2, h=8, g=2,
          d_h=128, n_max=100, scale=0.088):
    return lib.mqa_decode_attention(q, k, v, lens, out, b, h, g, d_h, n_max, scale, None)


def _append(lib, kn=A, vn=A + 0x1000, kc=A + 0x2000, vc=A + 0x3000, pos=A + 0x4000, b=2, g=2,
            d_h=128, n_max=100):
    return lib.mqa_kv_append(kn, vn, kc, vc, pos, b, g, d_h, n_max, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=0), INVALID), (dict(k=0), INVALID), (dict(v=0), INVALID), (dict(lens=0), INVALID),
    (dict(out=0), INVALID),
    (dict(b=0), INVALID), (dict(h=-1), INVALID), (dict(g=0), INVALID), (dict(n_max=0), INVALID),
    (dict(h=8, g=3), INVALID),                    # heads must split evenly into groups
    (dict(scale=math.inf), INVALID), (dict(scale=math.nan), INVALID),
    (dict(q=A + 8), INVALID), (dict(k=A + 2), INVALID), (dict(out=A + 4), INVALID),
    (dict(lens=A + 2), INVALID),
    (dict(d_h=96), UNSUPPORTED), (dict(d_h=256), UNSUPPORTED),
    (dict(h=128, g=1), UNSUPPORTED),              # h/g above 64
    (dict(b=8193), UNSUPPORTED),
])
def test_attention_host_checks(lib, kw, code):
    assert _attn(lib, **kw) == code


@pytest.mark.parametrize("kw,code", [
    (dict(kn=0), INVALID), (dict(vn=0), INVALID), (dict(kc=0), INVALID), (dict(vc=0), INVALID),
    (dict(pos=0), INVALID), (dict(b=0), INVALID), (dict(g=-2), INVALID), (dict(n_max=0), INVALID),
    (dict(kc=A + 8), INVALID), (dict(pos=A + 1), INVALID),
    (dict(d_h=80), UNSUPPORTED),
])
def test_append_host_checks(lib, kw, code):
    assert _append(lib, **kw) == code


def test_debug_override_validation(lib):
    assert lib.mqa_debug_override(-1, 0) == INVALID
    assert lib.mqa_debug_override(0, 4) == INVALID     # paths are 0 (auto) .. 3 (tcgen05)
    for path in (3, 2, 1, 0):
        assert lib.mqa_debug_override(0, path) == OK


def test_forced_cuda_core_path_rejects_large_groups(lib):
    assert lib.mqa_debug_override(0, 1) == OK
    try:
        assert _attn(lib, h=8, g=1) == UNSUPPORTED   # G = 8 has no CUDA-core kernel
    finally:
        lib.mqa_debug_override(0, 0)


def test_device_status_needs_an_output(lib):
    assert lib.mqa_get_device_status(None, None) == INVALID


def _step(lib, q=A, kn=A + 0x1000, vn=A + 0x2000, k=A + 0x3000, v=A + 0x4000, pos=A + 0x5000,
          lens=A + 0x6000, out=A + 0x7000, b=2, h=8, g=2, d_h=128, n_max=100, scale=0.088):
    return lib.mqa_decode_step(q, kn, vn, k, v, pos, lens, out, b, h, g, d_h, n_max, scale, None)


@pytest.mark.parametrize("kw,code", [
    # the append's arguments ...
    (dict(kn=0), INVALID), (dict(vn=0), INVALID), (dict(pos=0), INVALID),
    (dict(kn=A + 8), INVALID), (dict(vn=A + 2), INVALID), (dict(pos=A + 0x5002), INVALID),
    # ... and the attention's, checked the same way as mqa_decode_attention
    (dict(q=0), INVALID), (dict(k=0), INVALID), (dict(lens=0), INVALID), (dict(out=0), INVALID),
    (dict(b=0), INVALID), (dict(h=8, g=3), INVALID), (dict(scale=math.nan), INVALID),
    (dict(k=A + 4), INVALID),
    (dict(d_h=96), UNSUPPORTED), (dict(h=128, g=1), UNSUPPORTED), (dict(b=8193), UNSUPPORTED),
])
def test_fused_step_host_checks(lib, kw, code):
    assert _step(lib, **kw) == code


def test_timeout_site_rejects_null(lib):
    assert lib.mqa_debug_timeout_site(None) == INVALID


# ---- paged caches: the page table and the pool geometry are checked on the host too ----------
PAGED_GEOMETRY_CASES = [
    (dict(table=0), INVALID), (dict(table=A + 0x8002), INVALID),
    (dict(page_size=0), INVALID), (dict(max_pages=0), INVALID), (dict(num_pages=-1), INVALID),
    (dict(page_size=24), UNSUPPORTED), (dict(page_size=48), UNSUPPORTED),
    (dict(page_size=4), UNSUPPORTED), (dict(page_size=192), UNSUPPORTED),
    (dict(page_size=64, max_pages=1 << 26), UNSUPPORTED),   # 2^32 addressable rows
    (dict(num_pages=1 << 30), UNSUPPORTED),                 # num_pages * g past int32
    (dict(d_h=96), UNSUPPORTED), (dict(b=0), INVALID), (dict(g=0), INVALID),
]


def _attn_paged(lib, q=A, k=A + 0x1000, v=A + 0x2000, table=A + 0x8000, lens=A + 0x3000,
                out=A + 0x4000, b=2, h=8, g=2, d_h=128, page_size=16, max_pages=8, num_pages=20,
                scale=0.088):
    return lib.mqa_decode_attention_paged(q, k, v, table, lens, out, b, h, g, d_h, page_size,
                                          max_pages, num_pages, scale, None)


def _step_paged(lib, q=A, kn=A + 0x1000, vn=A + 0x2000, k=A + 0x3000, v=A + 0x4000,
                pos=A + 0x5000, table=A + 0x8000, lens=A + 0x6000, out=A + 0x7000, b=2, h=8, g=2,
                d_h=128, page_size=16, max_pages=8, num_pages=20, scale=0.088):
    return lib.mqa_decode_step_paged(q, kn, vn, k, v, pos, table, lens, out, b, h, g, d_h,
                                     page_size, max_pages, num_pages, scale, None)


def _append_paged(lib, kn=A, vn=A + 0x1000, kc=A + 0x2000, vc=A + 0x3000, pos=A + 0x4000,
                  table=A + 0x8000, b=2, g=2, d_h=128, page_size=16, max_pages=8, num_pages=20):
    return lib.mqa_kv_append_paged(kn, vn, kc, vc, pos, table, b, g, d_h, page_size, max_pages,
                                   num_pages, None)


@pytest.mark.parametrize("kw,code", PAGED_GEOMETRY_CASES + [
    (dict(q=0), INVALID), (dict(k=0), INVALID), (dict(lens=0), INVALID), (dict(out=A + 4), INVALID),
    (dict(h=8, g=3), INVALID), (dict(scale=math.inf), INVALID), (dict(h=128, g=1), UNSUPPORTED),
])
def test_paged_attention_host_checks(lib, kw, code):
    assert _attn_paged(lib, **kw) == code


@pytest.mark.parametrize("kw,code", PAGED_GEOMETRY_CASES + [
    (dict(kn=0), INVALID), (dict(vn=A + 0x2002), INVALID), (dict(pos=0), INVALID),
    (dict(pos=A + 0x5001), INVALID), (dict(q=0), INVALID), (dict(k=A + 0x3008), INVALID),
    (dict(h=8, g=3), INVALID),
])
def test_paged_step_host_checks(lib, kw, code):
    assert _step_paged(lib, **kw) == code


@pytest.mark.parametrize("kw,code", PAGED_GEOMETRY_CASES + [
    (dict(kn=0), INVALID), (dict(vc=0), INVALID), (dict(pos=0), INVALID),
    (dict(kc=A + 0x2008), INVALID), (dict(pos=A + 0x4001), INVALID),
])
def test_paged_append_host_checks(lib, kw, code):
    assert _append_paged(lib, **kw) == code


# ---- fp8 caches: the scales and the head dimension are checked on the host too ---------------
FP8_SCALE_CASES = [
    (dict(ks=0.0), INVALID), (dict(vs=-1.0), INVALID), (dict(ks=math.inf), INVALID),
    (dict(vs=math.nan), INVALID), (dict(d_h=64), UNSUPPORTED), (dict(d_h=256), UNSUPPORTED),
]


def _attn_fp8(lib, q=A, k=A + 0x1000, v=A + 0x2000, lens=A + 0x3000, out=A + 0x4000, b=2, h=8,
              g=2, d_h=128, n_max=100, scale=0.088, ks=0.01, vs=0.02):
    return lib.mqa_decode_attention_fp8(q, k, v, lens, out, b, h, g, d_h, n_max, scale, ks, vs,
                                        None)


def _step_fp8(lib, q=A, kn=A + 0x1000, vn=A + 0x2000, k=A + 0x3000, v=A + 0x4000, pos=A + 0x5000,
              lens=A + 0x6000, out=A + 0x7000, b=2, h=8, g=2, d_h=128, n_max=100, scale=0.088,
              ks=0.01, vs=0.02):
    return lib.mqa_decode_step_fp8(q, kn, vn, k, v, pos, lens, out, b, h, g, d_h, n_max, scale,
                                   ks, vs, None)


def _append_fp8(lib, kn=A, vn=A + 0x1000, kc=A + 0x2000, vc=A + 0x3000, pos=A + 0x4000, b=2, g=2,
                d_h=128, n_max=100, ks=0.01, vs=0.02):
    return lib.mqa_kv_append_fp8(kn, vn, kc, vc, pos, b, g, d_h, n_max, ks, vs, None)


@pytest.mark.parametrize("kw,code", FP8_SCALE_CASES + [
    (dict(q=0), INVALID), (dict(k=0), INVALID), (dict(lens=0), INVALID), (dict(out=A + 4), INVALID),
    (dict(k=A + 0x1008), INVALID), (dict(b=0), INVALID), (dict(h=8, g=3), INVALID),
    (dict(scale=math.nan), INVALID), (dict(h=128, g=1), UNSUPPORTED), (dict(b=8193), UNSUPPORTED),
])
def test_fp8_attention_host_checks(lib, kw, code):
    assert _attn_fp8(lib, **kw) == code


@pytest.mark.parametrize("kw,code", FP8_SCALE_CASES + [
    (dict(kn=0), INVALID), (dict(vn=A + 0x2002), INVALID), (dict(pos=0), INVALID),
    (dict(pos=A + 0x5001), INVALID), (dict(q=0), INVALID), (dict(v=A + 0x4008), INVALID),
    (dict(h=8, g=3), INVALID),
])
def test_fp8_step_host_checks(lib, kw, code):
    assert _step_fp8(lib, **kw) == code


@pytest.mark.parametrize("kw,code", FP8_SCALE_CASES + [
    (dict(kn=0), INVALID), (dict(vc=0), INVALID), (dict(pos=0), INVALID), (dict(b=0), INVALID),
    (dict(n_max=0), INVALID), (dict(kc=A + 0x2008), INVALID), (dict(pos=A + 0x4001), INVALID),
])
def test_fp8_append_host_checks(lib, kw, code):
    assert _append_fp8(lib, **kw) == code


# ---- several tokens per sequence ----------------------------------------------------------------
def _attn_multi(lib, q=A, k=A + 0x1000, v=A + 0x2000, lens=A + 0x3000, out=A + 0x4000, b=2, T=4,
                h=8, g=2, d_h=128, n_max=100, scale=0.088):
    return lib.mqa_decode_attention_multi(q, k, v, lens, out, b, T, h, g, d_h, n_max, scale, None)


def _step_multi(lib, q=A, kn=A + 0x1000, vn=A + 0x2000, k=A + 0x3000, v=A + 0x4000,
                pos=A + 0x5000, lens=A + 0x6000, out=A + 0x7000, b=2, T=4, h=8, g=2, d_h=128,
                n_max=100, scale=0.088):
    return lib.mqa_decode_step_multi(q, kn, vn, k, v, pos, lens, out, b, T, h, g, d_h, n_max,
                                     scale, None)


def _append_multi(lib, kn=A, vn=A + 0x1000, kc=A + 0x2000, vc=A + 0x3000, pos=A + 0x4000, b=2,
                  T=4, g=2, d_h=128, n_max=100):
    return lib.mqa_kv_append_multi(kn, vn, kc, vc, pos, b, T, g, d_h, n_max, None)


MULTI_CASES = [
    (dict(T=0), INVALID), (dict(T=-3), INVALID), (dict(q=0), INVALID), (dict(out=A + 4), INVALID),
    (dict(h=8, g=3), INVALID), (dict(d_h=96), UNSUPPORTED),
    (dict(T=1 << 21, h=8, g=2), UNSUPPORTED),      # 2^21 tokens x 4 heads: past the prefill rows
]


@pytest.mark.parametrize("kw,code", MULTI_CASES)
def test_multi_attention_host_checks(lib, kw, code):
    assert _attn_multi(lib, **kw) == code


@pytest.mark.parametrize("kw,code", MULTI_CASES + [
    (dict(kn=0), INVALID), (dict(pos=A + 0x5001), INVALID), (dict(vn=A + 0x2008), INVALID),
])
def test_multi_step_host_checks(lib, kw, code):
    assert _step_multi(lib, **kw) == code


@pytest.mark.parametrize("kw,code", [
    (dict(T=0), INVALID), (dict(kn=0), INVALID), (dict(pos=0), INVALID), (dict(b=0), INVALID),
    (dict(kc=A + 0x2008), INVALID), (dict(d_h=80), UNSUPPORTED),
])
def test_multi_append_host_checks(lib, kw, code):
    assert _append_multi(lib, **kw) == code


def test_multi_rejects_forced_cuda_cores_and_mma_sync_past_one_tile_of_rows(lib):
    # several tokens: CUDA cores never; mma.sync up to 64 rows per KV head; more rows (17 tokens x
    # 4 heads = 68) only on the tcgen05 prefill kernel, automatic or forced
    for path, kw in ((1, dict(h=4, g=4)), (2, dict(T=17, h=8, g=2))):
        assert lib.mqa_debug_override(0, path) == OK
        try:
            assert _attn_multi(lib, **kw) == UNSUPPORTED
        finally:
            lib.mqa_debug_override(0, 0)
    for path in (0, 3):
        assert lib.mqa_debug_override(0, path) == OK
        try:
            # past the host checks (with no GPU here the launch itself then fails)
            assert _attn_multi(lib, T=17, h=8, g=2) not in (INVALID, UNSUPPORTED)
            assert _attn_multi(lib, T=2, h=64, g=1) not in (INVALID, UNSUPPORTED)
        finally:
            lib.mqa_debug_override(0, 0)
