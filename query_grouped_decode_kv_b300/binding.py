"""ctypes binding over ``libmqa.so`` (declared in ``include/mqa.h``).

Argument marshalling only: shapes are read off the torch tensors, pointers and the current CUDA
stream are handed to the C ABI, and a non-zero status becomes :class:`MqaError`. Every step of the
computation runs in the library's CUDA kernels; there is no fallback path. Importing this module
raises ``ImportError`` if the library has not been built (``python -m
query_grouped_decode_kv_b300.build``).
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libmqa.so")

if not os.path.exists(_LIB_PATH):
    raise ImportError(f"libmqa.so is not built ({_LIB_PATH}); run "
                      "`python -m query_grouped_decode_kv_b300.build`")

_lib = ctypes.CDLL(_LIB_PATH)
_vp, _i32, _f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float

_lib.mqa_kv_append.restype = _i32
_lib.mqa_kv_append.argtypes = [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _vp]
_lib.mqa_decode_attention.restype = _i32
_lib.mqa_decode_attention.argtypes = [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32,
                                      _f32, _vp]
_lib.mqa_decode_step.restype = _i32
_lib.mqa_decode_step.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32,
                                 _i32, _f32, _vp]
_lib.mqa_kv_append_paged.restype = _i32
_lib.mqa_kv_append_paged.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32,
                                     _i32, _vp]
_lib.mqa_decode_attention_paged.restype = _i32
_lib.mqa_decode_attention_paged.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32,
                                            _i32, _i32, _i32, _f32, _vp]
_lib.mqa_decode_step_paged.restype = _i32
_lib.mqa_decode_step_paged.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32,
                                       _i32, _i32, _i32, _i32, _i32, _f32, _vp]
_lib.mqa_kv_append_fp8.restype = _i32
_lib.mqa_kv_append_fp8.argtypes = [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _f32, _f32,
                                   _vp]
_lib.mqa_decode_attention_fp8.restype = _i32
_lib.mqa_decode_attention_fp8.argtypes = [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32,
                                          _f32, _f32, _f32, _vp]
_lib.mqa_decode_step_fp8.restype = _i32
_lib.mqa_decode_step_fp8.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32,
                                     _i32, _i32, _f32, _f32, _f32, _vp]
_lib.mqa_kv_append_multi.restype = _i32
_lib.mqa_kv_append_multi.argtypes = [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _vp]
_lib.mqa_decode_attention_multi.restype = _i32
_lib.mqa_decode_attention_multi.argtypes = [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32,
                                            _i32, _f32, _vp]
_lib.mqa_decode_step_multi.restype = _i32
_lib.mqa_decode_step_multi.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32,
                                       _i32, _i32, _i32, _f32, _vp]
_lib.mqa_kv_append_paged_fp8.restype = _i32
_lib.mqa_kv_append_paged_fp8.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32,
                                         _i32, _i32, _f32, _f32, _vp]
_lib.mqa_decode_attention_paged_fp8.restype = _i32
_lib.mqa_decode_attention_paged_fp8.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32,
                                                _i32, _i32, _i32, _i32, _f32, _f32, _f32, _vp]
_lib.mqa_decode_step_paged_fp8.restype = _i32
_lib.mqa_decode_step_paged_fp8.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32,
                                           _i32, _i32, _i32, _i32, _i32, _i32, _f32, _f32, _f32,
                                           _vp]
_lib.mqa_kv_append_paged_multi.restype = _i32
_lib.mqa_kv_append_paged_multi.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32,
                                           _i32, _i32, _i32, _vp]
_lib.mqa_decode_attention_paged_multi.restype = _i32
_lib.mqa_decode_attention_paged_multi.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32,
                                                  _i32, _i32, _i32, _i32, _i32, _f32, _vp]
_lib.mqa_decode_step_paged_multi.restype = _i32
_lib.mqa_decode_step_paged_multi.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32,
                                             _i32, _i32, _i32, _i32, _i32, _i32, _i32, _f32, _vp]
_lib.mqa_status_string.restype = ctypes.c_char_p
_lib.mqa_status_string.argtypes = [_i32]
_lib.mqa_get_device_status.restype = _i32
_lib.mqa_get_device_status.argtypes = [_vp, ctypes.POINTER(_i32)]
_lib.mqa_kernel_launch_count.restype = ctypes.c_uint64
_lib.mqa_kernel_launch_count.argtypes = []
_lib.mqa_debug_timeout_site.restype = _i32
_lib.mqa_debug_timeout_site.argtypes = [ctypes.POINTER(_i32)]
_lib.mqa_debug_stall.restype = _i32
_lib.mqa_debug_stall.argtypes = [_i32]
_lib.mqa_debug_set_wait_limit_ns.restype = _i32
_lib.mqa_debug_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
_lib.mqa_debug_override.restype = _i32
_lib.mqa_debug_override.argtypes = [_i32, _i32]
_lib.mqa_set_launch_overlap.restype = _i32
_lib.mqa_set_launch_overlap.argtypes = [_vp, _i32]

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_DEVICE_BOUNDS, ERR_TIMEOUT = range(6)


class MqaError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {status_string(status)}" if what else status_string(status))


def library_path() -> str:
    return _LIB_PATH


def raw() -> ctypes.CDLL:
    """The loaded library, for callers that pass raw pointers themselves."""
    return _lib


def status_string(status: int) -> str:
    return _lib.mqa_status_string(int(status)).decode()


def kernel_launch_count() -> int:
    return int(_lib.mqa_kernel_launch_count())


def debug_override(num_ctas: int = 0, path: int = 0) -> None:
    st = _lib.mqa_debug_override(int(num_ctas), int(path))
    if st:
        raise MqaError(st, "mqa_debug_override")


def debug_timeout_site() -> tuple[int, int, int, int]:
    """(site, tile, block, thread) of the first in-kernel wait that timed out since the last
    call; site 0 means none. Synchronises the current device."""
    out = (_i32 * 4)()
    st = _lib.mqa_debug_timeout_site(out)
    if st:
        raise MqaError(st, "mqa_debug_timeout_site")
    return tuple(int(x) for x in out)


def debug_set_wait_limit_ns(ns: int = 0) -> None:
    """Testing hook: in-kernel wait limit in nanoseconds (0 = the default of one second)."""
    st = _lib.mqa_debug_set_wait_limit_ns(int(ns))
    if st:
        raise MqaError(st, "mqa_debug_set_wait_limit_ns")


def debug_stall(on: bool | int) -> None:
    """Testing hook: make the consumer warps of following launches wait on a barrier nothing
    completes, so each launch times out after the wait limit: before their first tile (True or
    1), or right after counting their first arrival at a split sequence (2), which leaves arrival
    counters non-zero."""
    mode = int(on) if not isinstance(on, bool) else (1 if on else 0)
    st = _lib.mqa_debug_stall(mode)
    if st:
        raise MqaError(st, "mqa_debug_stall")


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _check(t: torch.Tensor, name: str, dtype: torch.dtype, ndim: int) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda or t.dtype != dtype or t.dim() != ndim or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA {dtype} tensor with {ndim} dims, "
                         f"got {t.dtype} {tuple(t.shape)} on {t.device}")


def set_launch_overlap(on: bool, stream=None) -> None:
    """Allow (or forbid) the attention launches on ``stream`` to start before the kernel ahead
    of them on it has finished (programmatic dependent launch). The caller guarantees that the
    kernel preceding each call writes none of the call's inputs (q, new rows, positions,
    lengths, page table, the cache rows it reads besides the ones it appends); see
    ``mqa_set_launch_overlap`` in ``include/mqa.h``."""
    st = _lib.mqa_set_launch_overlap(_vp(_stream_handle(stream)), 1 if on else 0)
    if st:
        raise MqaError(st, "mqa_set_launch_overlap")


def get_device_status(stream=None) -> int:
    """Synchronise the stream, then read and clear the latched device status (0 = ok)."""
    out = _i32(0)
    st = _lib.mqa_get_device_status(_vp(_stream_handle(stream)), ctypes.byref(out))
    if st:
        raise MqaError(st, "mqa_get_device_status")
    return int(out.value)


def kv_append(k_new: torch.Tensor, v_new: torch.Tensor, k_cache: torch.Tensor,
              v_cache: torch.Tensor, pos: torch.Tensor, stream=None) -> None:
    """``k_cache[b, j, pos[b]] = k_new[b, j]`` (and V) for every sequence b and KV head j."""
    for t, n in ((k_new, "k_new"), (v_new, "v_new")):
        _check(t, n, torch.bfloat16, 3)
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _check(t, n, torch.bfloat16, 4)
    _check(pos, "pos", torch.int32, 1)
    b, g, n_max, d_h = k_cache.shape
    if v_cache.shape != k_cache.shape or k_new.shape != (b, g, d_h) or v_new.shape != (b, g, d_h) \
            or pos.shape != (b,):
        raise ValueError("kv_append: inconsistent shapes")
    st = _lib.mqa_kv_append(k_new.data_ptr(), v_new.data_ptr(), k_cache.data_ptr(),
                            v_cache.data_ptr(), pos.data_ptr(), b, g, d_h, n_max,
                            _vp(_stream_handle(stream)))
    if st:
        raise MqaError(st, "mqa_kv_append")


def decode_attention(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                     seq_lens: torch.Tensor, out: torch.Tensor | None = None,
                     scale: float | None = None, stream=None) -> torch.Tensor:
    """Grouped decode attention: ``out[b, i] = softmax(scale q[b,i] K_j^T) V_j``, j = i // (h/g),
    over the first ``seq_lens[b]`` cache rows. ``scale`` defaults to ``1/sqrt(d_h)``."""
    _check(q, "q", torch.bfloat16, 3)
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _check(t, n, torch.bfloat16, 4)
    _check(seq_lens, "seq_lens", torch.int32, 1)
    b, h, d_h = q.shape
    bk, g, n_max, dk = k_cache.shape
    if bk != b or dk != d_h or v_cache.shape != k_cache.shape or seq_lens.shape != (b,):
        raise ValueError("decode_attention: inconsistent shapes")
    if out is None:
        out = torch.empty_like(q)
    else:
        _check(out, "out", torch.bfloat16, 3)
        if out.shape != q.shape:
            raise ValueError("decode_attention: out must have q's shape")
    if scale is None:
        scale = 1.0 / math.sqrt(d_h)
    st = _lib.mqa_decode_attention(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                   seq_lens.data_ptr(), out.data_ptr(), b, h, g, d_h, n_max,
                                   float(scale), _vp(_stream_handle(stream)))
    if st:
        raise MqaError(st, "mqa_decode_attention")
    return out


def decode_step(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor, k_cache: torch.Tensor,
                v_cache: torch.Tensor, pos: torch.Tensor, seq_lens: torch.Tensor,
                out: torch.Tensor | None = None, scale: float | None = None,
                stream=None) -> torch.Tensor:
    """One launch doing :func:`kv_append` then :func:`decode_attention`: writes ``k_new``/``v_new``
    at row ``pos[b]`` of the caches and attends over the first ``seq_lens[b]`` rows."""
    _check(q, "q", torch.bfloat16, 3)
    for t, n in ((k_new, "k_new"), (v_new, "v_new")):
        _check(t, n, torch.bfloat16, 3)
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _check(t, n, torch.bfloat16, 4)
    _check(pos, "pos", torch.int32, 1)
    _check(seq_lens, "seq_lens", torch.int32, 1)
    b, h, d_h = q.shape
    bk, g, n_max, dk = k_cache.shape
    if bk != b or dk != d_h or v_cache.shape != k_cache.shape or seq_lens.shape != (b,) \
            or pos.shape != (b,) or k_new.shape != (b, g, d_h) or v_new.shape != (b, g, d_h):
        raise ValueError("decode_step: inconsistent shapes")
    if out is None:
        out = torch.empty_like(q)
    else:
        _check(out, "out", torch.bfloat16, 3)
        if out.shape != q.shape:
            raise ValueError("decode_step: out must have q's shape")
    if scale is None:
        scale = 1.0 / math.sqrt(d_h)
    st = _lib.mqa_decode_step(q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(),
                              k_cache.data_ptr(), v_cache.data_ptr(), pos.data_ptr(),
                              seq_lens.data_ptr(), out.data_ptr(), b, h, g, d_h, n_max,
                              float(scale), _vp(_stream_handle(stream)))
    if st:
        raise MqaError(st, "mqa_decode_step")
    return out


def _pool_shape(k_pool: torch.Tensor, v_pool: torch.Tensor, page_table: torch.Tensor, b: int,
                what: str) -> tuple[int, int, int, int, int]:
    for t, n in ((k_pool, "k_pool"), (v_pool, "v_pool")):
        _check(t, n, torch.bfloat16, 4)
    _check(page_table, "page_table", torch.int32, 2)
    num_pages, g, page_size, d_h = k_pool.shape
    if v_pool.shape != k_pool.shape or page_table.shape[0] != b:
        raise ValueError(f"{what}: inconsistent shapes")
    return num_pages, g, page_size, d_h, page_table.shape[1]


def kv_append_paged(k_new: torch.Tensor, v_new: torch.Tensor, k_pool: torch.Tensor,
                    v_pool: torch.Tensor, pos: torch.Tensor, page_table: torch.Tensor,
                    stream=None) -> None:
    """:func:`kv_append` into paged caches: pools ``[num_pages, g, page_size, d_h]`` and a page
    table ``[b, max_pages]``; row ``pos[b]`` lives in page ``page_table[b, pos[b] // page_size]``."""
    for t, n in ((k_new, "k_new"), (v_new, "v_new")):
        _check(t, n, torch.bfloat16, 3)
    _check(pos, "pos", torch.int32, 1)
    b = pos.shape[0]
    num_pages, g, page_size, d_h, max_pages = _pool_shape(k_pool, v_pool, page_table, b,
                                                          "kv_append_paged")
    if k_new.shape != (b, g, d_h) or v_new.shape != (b, g, d_h):
        raise ValueError("kv_append_paged: inconsistent shapes")
    st = _lib.mqa_kv_append_paged(k_new.data_ptr(), v_new.data_ptr(), k_pool.data_ptr(),
                                  v_pool.data_ptr(), pos.data_ptr(), page_table.data_ptr(), b, g,
                                  d_h, page_size, max_pages, num_pages,
                                  _vp(_stream_handle(stream)))
    if st:
        raise MqaError(st, "mqa_kv_append_paged")


def decode_attention_paged(q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                           page_table: torch.Tensor, seq_lens: torch.Tensor,
                           out: torch.Tensor | None = None, scale: float | None = None,
                           stream=None) -> torch.Tensor:
    """:func:`decode_attention` over paged caches (see :func:`kv_append_paged` for the layout)."""
    _check(q, "q", torch.bfloat16, 3)
    _check(seq_lens, "seq_lens", torch.int32, 1)
    b, h, d_h = q.shape
    num_pages, g, page_size, dk, max_pages = _pool_shape(k_pool, v_pool, page_table, b,
                                                         "decode_attention_paged")
    if dk != d_h or seq_lens.shape != (b,):
        raise ValueError("decode_attention_paged: inconsistent shapes")
    if out is None:
        out = torch.empty_like(q)
    else:
        _check(out, "out", torch.bfloat16, 3)
        if out.shape != q.shape:
            raise ValueError("decode_attention_paged: out must have q's shape")
    if scale is None:
        scale = 1.0 / math.sqrt(d_h)
    st = _lib.mqa_decode_attention_paged(q.data_ptr(), k_pool.data_ptr(), v_pool.data_ptr(),
                                         page_table.data_ptr(), seq_lens.data_ptr(),
                                         out.data_ptr(), b, h, g, d_h, page_size, max_pages,
                                         num_pages, float(scale), _vp(_stream_handle(stream)))
    if st:
        raise MqaError(st, "mqa_decode_attention_paged")
    return out


def decode_step_paged(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                      k_pool: torch.Tensor, v_pool: torch.Tensor, pos: torch.Tensor,
                      page_table: torch.Tensor, seq_lens: torch.Tensor,
                      out: torch.Tensor | None = None, scale: float | None = None,
                      stream=None) -> torch.Tensor:
    """:func:`decode_step` over paged caches: one launch that appends through the page table and
    attends over the first ``seq_lens[b]`` rows the table maps."""
    _check(q, "q", torch.bfloat16, 3)
    for t, n in ((k_new, "k_new"), (v_new, "v_new")):
        _check(t, n, torch.bfloat16, 3)
    _check(pos, "pos", torch.int32, 1)
    _check(seq_lens, "seq_lens", torch.int32, 1)
    b, h, d_h = q.shape
    num_pages, g, page_size, dk, max_pages = _pool_shape(k_pool, v_pool, page_table, b,
                                                         "decode_step_paged")
    if dk != d_h or seq_lens.shape != (b,) or pos.shape != (b,) or k_new.shape != (b, g, d_h) \
            or v_new.shape != (b, g, d_h):
        raise ValueError("decode_step_paged: inconsistent shapes")
    if out is None:
        out = torch.empty_like(q)
    else:
        _check(out, "out", torch.bfloat16, 3)
        if out.shape != q.shape:
            raise ValueError("decode_step_paged: out must have q's shape")
    if scale is None:
        scale = 1.0 / math.sqrt(d_h)
    st = _lib.mqa_decode_step_paged(q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(),
                                    k_pool.data_ptr(), v_pool.data_ptr(), pos.data_ptr(),
                                    page_table.data_ptr(), seq_lens.data_ptr(), out.data_ptr(), b,
                                    h, g, d_h, page_size, max_pages, num_pages, float(scale),
                                    _vp(_stream_handle(stream)))
    if st:
        raise MqaError(st, "mqa_decode_step_paged")
    return out


_FP8_DTYPES = (torch.uint8, torch.float8_e4m3fn)


def _check_fp8_cache(t: torch.Tensor, name: str) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda or t.dtype not in _FP8_DTYPES or t.dim() != 4 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA uint8 / float8_e4m3fn tensor with 4 "
                         f"dims, got {t.dtype} {tuple(t.shape)} on {t.device}")


def kv_append_fp8(k_new: torch.Tensor, v_new: torch.Tensor, k_cache: torch.Tensor,
                  v_cache: torch.Tensor, pos: torch.Tensor, k_scale: float, v_scale: float,
                  stream=None) -> None:
    """:func:`kv_append` into fp8 E4M3 caches ``[b, g, n_max, d_h]`` (uint8 codes): row
    ``pos[b]`` receives ``e4m3(k_new / k_scale)`` (and V with ``v_scale``)."""
    for t, n in ((k_new, "k_new"), (v_new, "v_new")):
        _check(t, n, torch.bfloat16, 3)
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _check_fp8_cache(t, n)
    _check(pos, "pos", torch.int32, 1)
    b, g, n_max, d_h = k_cache.shape
    if v_cache.shape != k_cache.shape or k_new.shape != (b, g, d_h) or v_new.shape != (b, g, d_h) \
            or pos.shape != (b,):
        raise ValueError("kv_append_fp8: inconsistent shapes")
    st = _lib.mqa_kv_append_fp8(k_new.data_ptr(), v_new.data_ptr(), k_cache.data_ptr(),
                                v_cache.data_ptr(), pos.data_ptr(), b, g, d_h, n_max,
                                float(k_scale), float(v_scale), _vp(_stream_handle(stream)))
    if st:
        raise MqaError(st, "mqa_kv_append_fp8")


def decode_attention_fp8(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                         seq_lens: torch.Tensor, k_scale: float, v_scale: float,
                         out: torch.Tensor | None = None, scale: float | None = None,
                         stream=None) -> torch.Tensor:
    """:func:`decode_attention` over fp8 E4M3 caches whose values are ``code * k_scale`` and
    ``code * v_scale``."""
    _check(q, "q", torch.bfloat16, 3)
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _check_fp8_cache(t, n)
    _check(seq_lens, "seq_lens", torch.int32, 1)
    b, h, d_h = q.shape
    bk, g, n_max, dk = k_cache.shape
    if bk != b or dk != d_h or v_cache.shape != k_cache.shape or seq_lens.shape != (b,):
        raise ValueError("decode_attention_fp8: inconsistent shapes")
    if out is None:
        out = torch.empty_like(q)
    else:
        _check(out, "out", torch.bfloat16, 3)
        if out.shape != q.shape:
            raise ValueError("decode_attention_fp8: out must have q's shape")
    if scale is None:
        scale = 1.0 / math.sqrt(d_h)
    st = _lib.mqa_decode_attention_fp8(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                       seq_lens.data_ptr(), out.data_ptr(), b, h, g, d_h, n_max,
                                       float(scale), float(k_scale), float(v_scale),
                                       _vp(_stream_handle(stream)))
    if st:
        raise MqaError(st, "mqa_decode_attention_fp8")
    return out


def decode_step_fp8(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                    k_cache: torch.Tensor, v_cache: torch.Tensor, pos: torch.Tensor,
                    seq_lens: torch.Tensor, k_scale: float, v_scale: float,
                    out: torch.Tensor | None = None, scale: float | None = None,
                    stream=None) -> torch.Tensor:
    """:func:`decode_step` over fp8 E4M3 caches: one launch that quantizes and appends the new
    rows and attends over the first ``seq_lens[b]`` rows."""
    _check(q, "q", torch.bfloat16, 3)
    for t, n in ((k_new, "k_new"), (v_new, "v_new")):
        _check(t, n, torch.bfloat16, 3)
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _check_fp8_cache(t, n)
    _check(pos, "pos", torch.int32, 1)
    _check(seq_lens, "seq_lens", torch.int32, 1)
    b, h, d_h = q.shape
    bk, g, n_max, dk = k_cache.shape
    if bk != b or dk != d_h or v_cache.shape != k_cache.shape or seq_lens.shape != (b,) \
            or pos.shape != (b,) or k_new.shape != (b, g, d_h) or v_new.shape != (b, g, d_h):
        raise ValueError("decode_step_fp8: inconsistent shapes")
    if out is None:
        out = torch.empty_like(q)
    else:
        _check(out, "out", torch.bfloat16, 3)
        if out.shape != q.shape:
            raise ValueError("decode_step_fp8: out must have q's shape")
    if scale is None:
        scale = 1.0 / math.sqrt(d_h)
    st = _lib.mqa_decode_step_fp8(q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(),
                                  k_cache.data_ptr(), v_cache.data_ptr(), pos.data_ptr(),
                                  seq_lens.data_ptr(), out.data_ptr(), b, h, g, d_h, n_max,
                                  float(scale), float(k_scale), float(v_scale),
                                  _vp(_stream_handle(stream)))
    if st:
        raise MqaError(st, "mqa_decode_step_fp8")
    return out


def kv_append_multi(k_new: torch.Tensor, v_new: torch.Tensor, k_cache: torch.Tensor,
                    v_cache: torch.Tensor, pos: torch.Tensor, stream=None) -> None:
    """Append T rows per sequence: ``k_new`` [b, T, g, d_h]; token t goes to row ``pos[b] + t``."""
    for t, n in ((k_new, "k_new"), (v_new, "v_new")):
        _check(t, n, torch.bfloat16, 4)
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _check(t, n, torch.bfloat16, 4)
    _check(pos, "pos", torch.int32, 1)
    b, g, n_max, d_h = k_cache.shape
    T = k_new.shape[1]
    if v_cache.shape != k_cache.shape or k_new.shape != (b, T, g, d_h) \
            or v_new.shape != (b, T, g, d_h) or pos.shape != (b,):
        raise ValueError("kv_append_multi: inconsistent shapes")
    st = _lib.mqa_kv_append_multi(k_new.data_ptr(), v_new.data_ptr(), k_cache.data_ptr(),
                                  v_cache.data_ptr(), pos.data_ptr(), b, T, g, d_h, n_max,
                                  _vp(_stream_handle(stream)))
    if st:
        raise MqaError(st, "mqa_kv_append_multi")


def decode_attention_multi(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                           seq_lens: torch.Tensor, out: torch.Tensor | None = None,
                           scale: float | None = None, stream=None) -> torch.Tensor:
    """Causal attention of T tokens per sequence: ``q`` [b, T, h, d_h]; token t attends the first
    ``seq_lens[b] - T + 1 + t`` cache rows. Returns [b, T, h, d_h]."""
    _check(q, "q", torch.bfloat16, 4)
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _check(t, n, torch.bfloat16, 4)
    _check(seq_lens, "seq_lens", torch.int32, 1)
    b, T, h, d_h = q.shape
    bk, g, n_max, dk = k_cache.shape
    if bk != b or dk != d_h or v_cache.shape != k_cache.shape or seq_lens.shape != (b,):
        raise ValueError("decode_attention_multi: inconsistent shapes")
    if out is None:
        out = torch.empty_like(q)
    else:
        _check(out, "out", torch.bfloat16, 4)
        if out.shape != q.shape:
            raise ValueError("decode_attention_multi: out must have q's shape")
    if scale is None:
        scale = 1.0 / math.sqrt(d_h)
    st = _lib.mqa_decode_attention_multi(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                         seq_lens.data_ptr(), out.data_ptr(), b, T, h, g, d_h,
                                         n_max, float(scale), _vp(_stream_handle(stream)))
    if st:
        raise MqaError(st, "mqa_decode_attention_multi")
    return out


def decode_step_multi(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                      k_cache: torch.Tensor, v_cache: torch.Tensor, pos: torch.Tensor,
                      seq_lens: torch.Tensor, out: torch.Tensor | None = None,
                      scale: float | None = None, stream=None) -> torch.Tensor:
    """One launch doing :func:`kv_append_multi` then :func:`decode_attention_multi`."""
    _check(q, "q", torch.bfloat16, 4)
    for t, n in ((k_new, "k_new"), (v_new, "v_new")):
        _check(t, n, torch.bfloat16, 4)
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _check(t, n, torch.bfloat16, 4)
    _check(pos, "pos", torch.int32, 1)
    _check(seq_lens, "seq_lens", torch.int32, 1)
    b, T, h, d_h = q.shape
    bk, g, n_max, dk = k_cache.shape
    if bk != b or dk != d_h or v_cache.shape != k_cache.shape or seq_lens.shape != (b,) \
            or pos.shape != (b,) or k_new.shape != (b, T, g, d_h) or v_new.shape != (b, T, g, d_h):
        raise ValueError("decode_step_multi: inconsistent shapes")
    if out is None:
        out = torch.empty_like(q)
    else:
        _check(out, "out", torch.bfloat16, 4)
        if out.shape != q.shape:
            raise ValueError("decode_step_multi: out must have q's shape")
    if scale is None:
        scale = 1.0 / math.sqrt(d_h)
    st = _lib.mqa_decode_step_multi(q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(),
                                    k_cache.data_ptr(), v_cache.data_ptr(), pos.data_ptr(),
                                    seq_lens.data_ptr(), out.data_ptr(), b, T, h, g, d_h, n_max,
                                    float(scale), _vp(_stream_handle(stream)))
    if st:
        raise MqaError(st, "mqa_decode_step_multi")
    return out


def _fp8_pool_shape(k_pool: torch.Tensor, v_pool: torch.Tensor, page_table: torch.Tensor, b: int,
                    what: str) -> tuple[int, int, int, int, int]:
    for t, n in ((k_pool, "k_pool"), (v_pool, "v_pool")):
        _check_fp8_cache(t, n)
    _check(page_table, "page_table", torch.int32, 2)
    num_pages, g, page_size, d_h = k_pool.shape
    if v_pool.shape != k_pool.shape or page_table.shape[0] != b:
        raise ValueError(f"{what}: inconsistent shapes")
    return num_pages, g, page_size, d_h, page_table.shape[1]


def _out_like(q: torch.Tensor, out: torch.Tensor | None, ndim: int, what: str) -> torch.Tensor:
    if out is None:
        return torch.empty_like(q)
    _check(out, "out", torch.bfloat16, ndim)
    if out.shape != q.shape:
        raise ValueError(f"{what}: out must have q's shape")
    return out


def kv_append_paged_fp8(k_new: torch.Tensor, v_new: torch.Tensor, k_pool: torch.Tensor,
                        v_pool: torch.Tensor, pos: torch.Tensor, page_table: torch.Tensor,
                        k_scale: float, v_scale: float, stream=None) -> None:
    """:func:`kv_append_fp8` into paged fp8 pools ``[num_pages, g, page_size, d_h]`` (uint8
    codes) through ``page_table`` ``[b, max_pages]``."""
    for t, n in ((k_new, "k_new"), (v_new, "v_new")):
        _check(t, n, torch.bfloat16, 3)
    _check(pos, "pos", torch.int32, 1)
    b = pos.shape[0]
    num_pages, g, page_size, d_h, max_pages = _fp8_pool_shape(k_pool, v_pool, page_table, b,
                                                              "kv_append_paged_fp8")
    if k_new.shape != (b, g, d_h) or v_new.shape != (b, g, d_h):
        raise ValueError("kv_append_paged_fp8: inconsistent shapes")
    st = _lib.mqa_kv_append_paged_fp8(k_new.data_ptr(), v_new.data_ptr(), k_pool.data_ptr(),
                                      v_pool.data_ptr(), pos.data_ptr(), page_table.data_ptr(), b,
                                      g, d_h, page_size, max_pages, num_pages, float(k_scale),
                                      float(v_scale), _vp(_stream_handle(stream)))
    if st:
        raise MqaError(st, "mqa_kv_append_paged_fp8")


def decode_attention_paged_fp8(q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                               page_table: torch.Tensor, seq_lens: torch.Tensor, k_scale: float,
                               v_scale: float, out: torch.Tensor | None = None,
                               scale: float | None = None, stream=None) -> torch.Tensor:
    """:func:`decode_attention_fp8` over paged fp8 pools."""
    _check(q, "q", torch.bfloat16, 3)
    _check(seq_lens, "seq_lens", torch.int32, 1)
    b, h, d_h = q.shape
    num_pages, g, page_size, dk, max_pages = _fp8_pool_shape(k_pool, v_pool, page_table, b,
                                                             "decode_attention_paged_fp8")
    if dk != d_h or seq_lens.shape != (b,):
        raise ValueError("decode_attention_paged_fp8: inconsistent shapes")
    out = _out_like(q, out, 3, "decode_attention_paged_fp8")
    if scale is None:
        scale = 1.0 / math.sqrt(d_h)
    st = _lib.mqa_decode_attention_paged_fp8(q.data_ptr(), k_pool.data_ptr(), v_pool.data_ptr(),
                                             page_table.data_ptr(), seq_lens.data_ptr(),
                                             out.data_ptr(), b, h, g, d_h, page_size, max_pages,
                                             num_pages, float(scale), float(k_scale),
                                             float(v_scale), _vp(_stream_handle(stream)))
    if st:
        raise MqaError(st, "mqa_decode_attention_paged_fp8")
    return out


def decode_step_paged_fp8(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                          k_pool: torch.Tensor, v_pool: torch.Tensor, pos: torch.Tensor,
                          page_table: torch.Tensor, seq_lens: torch.Tensor, k_scale: float,
                          v_scale: float, out: torch.Tensor | None = None,
                          scale: float | None = None, stream=None) -> torch.Tensor:
    """:func:`decode_step_fp8` over paged fp8 pools: one launch that quantizes and appends the
    new rows through the table and attends."""
    _check(q, "q", torch.bfloat16, 3)
    for t, n in ((k_new, "k_new"), (v_new, "v_new")):
        _check(t, n, torch.bfloat16, 3)
    _check(pos, "pos", torch.int32, 1)
    _check(seq_lens, "seq_lens", torch.int32, 1)
    b, h, d_h = q.shape
    num_pages, g, page_size, dk, max_pages = _fp8_pool_shape(k_pool, v_pool, page_table, b,
                                                             "decode_step_paged_fp8")
    if dk != d_h or seq_lens.shape != (b,) or pos.shape != (b,) or k_new.shape != (b, g, d_h) \
            or v_new.shape != (b, g, d_h):
        raise ValueError("decode_step_paged_fp8: inconsistent shapes")
    out = _out_like(q, out, 3, "decode_step_paged_fp8")
    if scale is None:
        scale = 1.0 / math.sqrt(d_h)
    st = _lib.mqa_decode_step_paged_fp8(q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(),
                                        k_pool.data_ptr(), v_pool.data_ptr(), pos.data_ptr(),
                                        page_table.data_ptr(), seq_lens.data_ptr(),
                                        out.data_ptr(), b, h, g, d_h, page_size, max_pages,
                                        num_pages, float(scale), float(k_scale), float(v_scale),
                                        _vp(_stream_handle(stream)))
    if st:
        raise MqaError(st, "mqa_decode_step_paged_fp8")
    return out


def kv_append_paged_multi(k_new: torch.Tensor, v_new: torch.Tensor, k_pool: torch.Tensor,
                          v_pool: torch.Tensor, pos: torch.Tensor, page_table: torch.Tensor,
                          stream=None) -> None:
    """T rows per sequence (``k_new`` [b, T, g, d_h]) through the page table: token t goes to
    row ``pos[b] + t``."""
    for t, n in ((k_new, "k_new"), (v_new, "v_new")):
        _check(t, n, torch.bfloat16, 4)
    _check(pos, "pos", torch.int32, 1)
    b, T = k_new.shape[0], k_new.shape[1]
    num_pages, g, page_size, d_h, max_pages = _pool_shape(k_pool, v_pool, page_table, b,
                                                          "kv_append_paged_multi")
    if k_new.shape != (b, T, g, d_h) or v_new.shape != (b, T, g, d_h) or pos.shape != (b,):
        raise ValueError("kv_append_paged_multi: inconsistent shapes")
    st = _lib.mqa_kv_append_paged_multi(k_new.data_ptr(), v_new.data_ptr(), k_pool.data_ptr(),
                                        v_pool.data_ptr(), pos.data_ptr(), page_table.data_ptr(),
                                        b, T, g, d_h, page_size, max_pages, num_pages,
                                        _vp(_stream_handle(stream)))
    if st:
        raise MqaError(st, "mqa_kv_append_paged_multi")


def decode_attention_paged_multi(q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                                 page_table: torch.Tensor, seq_lens: torch.Tensor,
                                 out: torch.Tensor | None = None, scale: float | None = None,
                                 stream=None) -> torch.Tensor:
    """:func:`decode_attention_multi` over paged caches (q [b, T, h, d_h])."""
    _check(q, "q", torch.bfloat16, 4)
    _check(seq_lens, "seq_lens", torch.int32, 1)
    b, T, h, d_h = q.shape
    num_pages, g, page_size, dk, max_pages = _pool_shape(k_pool, v_pool, page_table, b,
                                                         "decode_attention_paged_multi")
    if dk != d_h or seq_lens.shape != (b,):
        raise ValueError("decode_attention_paged_multi: inconsistent shapes")
    out = _out_like(q, out, 4, "decode_attention_paged_multi")
    if scale is None:
        scale = 1.0 / math.sqrt(d_h)
    st = _lib.mqa_decode_attention_paged_multi(q.data_ptr(), k_pool.data_ptr(), v_pool.data_ptr(),
                                               page_table.data_ptr(), seq_lens.data_ptr(),
                                               out.data_ptr(), b, T, h, g, d_h, page_size,
                                               max_pages, num_pages, float(scale),
                                               _vp(_stream_handle(stream)))
    if st:
        raise MqaError(st, "mqa_decode_attention_paged_multi")
    return out


def decode_step_paged_multi(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                            k_pool: torch.Tensor, v_pool: torch.Tensor, pos: torch.Tensor,
                            page_table: torch.Tensor, seq_lens: torch.Tensor,
                            out: torch.Tensor | None = None, scale: float | None = None,
                            stream=None) -> torch.Tensor:
    """One launch doing :func:`kv_append_paged_multi` then :func:`decode_attention_paged_multi`."""
    _check(q, "q", torch.bfloat16, 4)
    for t, n in ((k_new, "k_new"), (v_new, "v_new")):
        _check(t, n, torch.bfloat16, 4)
    _check(pos, "pos", torch.int32, 1)
    _check(seq_lens, "seq_lens", torch.int32, 1)
    b, T, h, d_h = q.shape
    num_pages, g, page_size, dk, max_pages = _pool_shape(k_pool, v_pool, page_table, b,
                                                         "decode_step_paged_multi")
    if dk != d_h or seq_lens.shape != (b,) or pos.shape != (b,) \
            or k_new.shape != (b, T, g, d_h) or v_new.shape != (b, T, g, d_h):
        raise ValueError("decode_step_paged_multi: inconsistent shapes")
    out = _out_like(q, out, 4, "decode_step_paged_multi")
    if scale is None:
        scale = 1.0 / math.sqrt(d_h)
    st = _lib.mqa_decode_step_paged_multi(q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(),
                                          k_pool.data_ptr(), v_pool.data_ptr(), pos.data_ptr(),
                                          page_table.data_ptr(), seq_lens.data_ptr(),
                                          out.data_ptr(), b, T, h, g, d_h, page_size, max_pages,
                                          num_pages, float(scale), _vp(_stream_handle(stream)))
    if st:
        raise MqaError(st, "mqa_decode_step_paged_multi")
    return out
