"""CPU oracle for MQA/GQA incremental decode attention (fp64, plain C behind ctypes).

TEST INFRASTRUCTURE, NOT THE PRODUCT. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference leg of ``bench.py`` may import this package. It shares no code with the
CUDA library and never imports it; the library never imports this.

What each function computes, and the passage it follows:

* :func:`kv_cache_bytes` -- ``2 x layers x kv_heads x seq_len x head_dim x dtype_bytes``
  ("GQA与MQA深度实战", ybb.press, §一 and §七).
* :func:`kv_append` -- write the new token's K/V row of every KV head at position ``pos[b]``
  (same page, §八; nanhubrain.csdn.net MQA article §2.2, concatenation along the sequence axis).
* :func:`decode_attention` -- for every sequence ``b`` and query head ``i`` with
  ``j = i // (h/g)``: ``softmax_t(scale * q_i . K_{j,t}) . V_{j,t}`` over ``t < seq_lens[b]``
  (ybb.press page §五).
* :func:`attention_partial` / :func:`lse_merge` -- per-range softmax states and their
  log-sum-exp combination (not on the pages; the identity that makes splitting a sequence exact).
* :func:`bf16_to_f64` / :func:`f64_to_bf16` -- bfloat16 conversions from the bit layout
  (round to nearest, ties to even).
* :func:`gather_pages` / :func:`kv_append_paged` -- the paged cache: a pool of fixed-size pages
  found through a per-sequence page table (nanhubrain.csdn.net MQA article §3.3 on vLLM's
  16-token blocks; ybb.press page §十 item 12); attention over it is attention over the gathered
  rows.

* :func:`e4m3_to_f64` / :func:`f64_to_e4m3` -- the 8-bit float format E4M3 from its bit layout
  (round to nearest, ties to even, saturating at +-448); :func:`kv_append_fp8` quantizes the new
  rows into fp8 caches with one scale per tensor, :func:`dequantize_e4m3` undoes it, and
  :func:`decode_attention_fp8` is attention over the dequantized caches (quantized K/V caches:
  ybb.press page §十 item 7, nanhubrain.csdn.net MQA article §4.3).

* :func:`kv_append_multi` / :func:`decode_attention_multi` -- T new tokens per sequence
  (ybb.press page §八: ``forward(x, start)`` writes T rows and attends over ``start + T`` rows;
  §十 item 10: the causal mask still applies per query position): token t attends the first
  ``seq_lens[b] - T + 1 + t`` rows.

Every function is pinned by ``tests/test_oracle_pins.py`` against closed forms, the pages' printed
numbers, invariants and library routines.
"""
from __future__ import annotations

import ctypes

import numpy as np

from . import build as _build

OK = 0
ERR_INVALID_ARG = 1
ERR_BOUNDS = 4

_lib = None


def _configure(lib):
    u64, i32, dbl, vp = ctypes.c_uint64, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
    lib.oracle_kv_cache_bytes.restype = u64
    lib.oracle_kv_cache_bytes.argtypes = [u64] * 5
    lib.oracle_bf16_to_double.restype = dbl
    lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_double_to_bf16.restype = ctypes.c_uint16
    lib.oracle_double_to_bf16.argtypes = [dbl]
    lib.oracle_kv_append.restype = i32
    lib.oracle_kv_append.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32]
    for name in ("oracle_decode_attention_bf16", "oracle_decode_attention_f64"):
        fn = getattr(lib, name)
        fn.restype = i32
        fn.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, dbl, i32]
    lib.oracle_attention_partial_f64.restype = i32
    lib.oracle_attention_partial_f64.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, dbl,
                                                 i32, i32, vp, vp, vp]
    lib.oracle_lse_merge.restype = i32
    lib.oracle_lse_merge.argtypes = [vp, vp, vp, i32, i32, vp]
    lib.oracle_gather_pages.restype = i32
    lib.oracle_gather_pages.argtypes = [vp, vp, i32, i32, i32, i32, i32, i32, vp]
    lib.oracle_kv_append_paged.restype = i32
    lib.oracle_kv_append_paged.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32]
    lib.oracle_e4m3_to_double.restype = dbl
    lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
    lib.oracle_double_to_e4m3.restype = ctypes.c_uint8
    lib.oracle_double_to_e4m3.argtypes = [dbl]
    lib.oracle_kv_append_fp8.restype = i32
    lib.oracle_kv_append_fp8.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, ctypes.c_float,
                                         ctypes.c_float]
    lib.oracle_dequantize_e4m3.restype = i32
    lib.oracle_dequantize_e4m3.argtypes = [vp, ctypes.c_size_t, dbl, vp]
    lib.oracle_kv_append_multi.restype = i32
    lib.oracle_kv_append_multi.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32]
    lib.oracle_decode_attention_multi_bf16.restype = i32
    lib.oracle_decode_attention_multi_bf16.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32,
                                                       i32, i32, dbl, i32]
    lib.oracle_gather_pages_u8.restype = i32
    lib.oracle_gather_pages_u8.argtypes = [vp, vp, i32, i32, i32, i32, i32, i32, vp]
    lib.oracle_kv_append_paged_multi.restype = i32
    lib.oracle_kv_append_paged_multi.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                                 i32, i32]
    lib.oracle_kv_append_paged_fp8.restype = i32
    lib.oracle_kv_append_paged_fp8.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                               i32, ctypes.c_float, ctypes.c_float]
    lib.oracle_num_threads.restype = i32
    lib.oracle_num_threads.argtypes = []
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = _configure(ctypes.CDLL(_build.build()))
    return _lib


def _swap_library(path):
    """Load another build of the oracle source (used by the mutation tests, which compile a
    deliberately broken copy to show that the pins catch it). Returns the previous handle."""
    global _lib
    prev = _load()
    _lib = _configure(ctypes.CDLL(path)) if path is not None else None
    return prev


def _restore_library(handle):
    global _lib
    _lib = handle


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


def num_threads() -> int:
    """OpenMP threads the oracle uses by default (the host's logical cores)."""
    return int(_load().oracle_num_threads())


def kv_cache_bytes(num_layers: int, num_kv_heads: int, seq_len: int, head_dim: int,
                   dtype_bytes: int) -> int:
    return int(_load().oracle_kv_cache_bytes(num_layers, num_kv_heads, seq_len, head_dim,
                                             dtype_bytes))


def bf16_to_f64(bits) -> np.ndarray:
    """Widen bfloat16 bit patterns (uint16) to float64, exactly."""
    lib = _load()
    b = _c(bits, np.uint16)
    out = np.empty(b.shape, dtype=np.float64)
    flat_in, flat_out = b.reshape(-1), out.reshape(-1)
    for k in range(flat_in.size):
        flat_out[k] = lib.oracle_bf16_to_double(int(flat_in[k]))
    return out


def f64_to_bf16(x) -> np.ndarray:
    """Round float64 values to bfloat16 bit patterns (nearest, ties to even)."""
    lib = _load()
    a = _c(x, np.float64)
    out = np.empty(a.shape, dtype=np.uint16)
    flat_in, flat_out = a.reshape(-1), out.reshape(-1)
    for k in range(flat_in.size):
        flat_out[k] = lib.oracle_double_to_bf16(float(flat_in[k]))
    return out


def kv_append(k_new, v_new, k_cache, v_cache, pos, n_max: int | None = None) -> int:
    """Append in place. ``k_new``/``v_new``: uint16 [b, g, d_h]; caches: uint16
    [b, g, n_max, d_h] (modified in place, must be C-contiguous uint16 arrays); ``pos``: int32 [b].
    Returns the oracle status (0 ok, 4 if some ``pos`` is outside ``[0, n_max)``)."""
    lib = _load()
    for c in (k_cache, v_cache):
        if not (isinstance(c, np.ndarray) and c.dtype == np.uint16 and c.flags.c_contiguous):
            raise TypeError("caches must be C-contiguous uint16 numpy arrays (updated in place)")
    b, g, nm, d_h = k_cache.shape
    kn, vn = _c(k_new, np.uint16), _c(v_new, np.uint16)
    p = _c(pos, np.int32)
    return int(lib.oracle_kv_append(_ptr(kn), _ptr(vn), _ptr(k_cache), _ptr(v_cache), _ptr(p),
                                    b, g, d_h, nm))


def decode_attention(q, k_cache, v_cache, seq_lens, scale: float, threads: int = 0,
                     return_status: bool = False):
    """fp64 grouped decode attention.

    ``q`` [b, h, d_h]; caches [b, g, n_max, d_h]; either all uint16 (bfloat16 bit patterns,
    widened exactly) or all float64. ``seq_lens`` int32 [b]. Returns float64 [b, h, d_h].
    """
    lib = _load()
    q = np.asarray(q)
    if q.dtype == np.uint16:
        fn, dt = lib.oracle_decode_attention_bf16, np.uint16
    else:
        fn, dt = lib.oracle_decode_attention_f64, np.float64
    qq, kk, vv = _c(q, dt), _c(k_cache, dt), _c(v_cache, dt)
    lens = _c(seq_lens, np.int32)
    b, h, d_h = qq.shape
    _, g, n_max, d_k = kk.shape
    if d_k != d_h or vv.shape != kk.shape or lens.shape != (b,):
        raise ValueError("shape mismatch")
    out = np.empty((b, h, d_h), dtype=np.float64)
    st = int(fn(_ptr(qq), _ptr(kk), _ptr(vv), _ptr(lens), _ptr(out), b, h, g, d_h, n_max,
                float(scale), int(threads)))
    if st == ERR_INVALID_ARG:
        raise ValueError("oracle rejected the arguments")
    return (out, st) if return_status else out


def attention_partial(q, k_cache, v_cache, scale: float, t_begin: int, t_end: int):
    """Per-range softmax state over rows ``[t_begin, t_end)`` (float64 inputs).
    Returns ``(m [b,h], l [b,h], o [b,h,d_h])`` with ``o`` un-normalised."""
    lib = _load()
    qq = _c(q, np.float64)
    kk, vv = _c(k_cache, np.float64), _c(v_cache, np.float64)
    b, h, d_h = qq.shape
    _, g, n_max, _ = kk.shape
    m = np.empty((b, h)); l = np.empty((b, h)); o = np.empty((b, h, d_h))
    st = int(lib.oracle_attention_partial_f64(_ptr(qq), _ptr(kk), _ptr(vv), b, h, g, d_h, n_max,
                                              float(scale), t_begin, t_end, _ptr(m), _ptr(l),
                                              _ptr(o)))
    if st:
        raise ValueError(f"oracle partial failed with status {st}")
    return m, l, o


def lse_merge(m, l, o) -> np.ndarray:
    """Merge S partial states of one row: ``m`` [S], ``l`` [S], ``o`` [S, d_h] -> [d_h]."""
    lib = _load()
    mm, ll, oo = _c(m, np.float64), _c(l, np.float64), _c(o, np.float64)
    S, d_h = oo.shape
    out = np.empty(d_h)
    st = int(lib.oracle_lse_merge(_ptr(mm), _ptr(ll), _ptr(oo), S, d_h, _ptr(out)))
    if st == ERR_INVALID_ARG:
        raise ValueError("bad merge arguments")
    return out


def gather_pages(pool, table, page_size: int):
    """Contiguous cache [b, g, max_pages * page_size, d_h] (uint16) from a page pool
    [num_pages, g, page_size, d_h] and a page table [b, max_pages] (int32). Rows of pages whose
    index is out of range come back zero and the status is 4. Returns (cache, status)."""
    lib = _load()
    pl = _c(pool, np.uint16)
    tb = _c(table, np.int32)
    num_pages, g, ps, d_h = pl.shape
    if ps != page_size:
        raise ValueError("page size mismatch")
    b, max_pages = tb.shape
    out = np.empty((b, g, max_pages * page_size, d_h), dtype=np.uint16)
    st = int(lib.oracle_gather_pages(_ptr(pl), _ptr(tb), b, g, d_h, page_size, max_pages,
                                     num_pages, _ptr(out)))
    if st == ERR_INVALID_ARG:
        raise ValueError("oracle rejected the arguments")
    return out, st


def kv_append_paged(k_new, v_new, k_pool, v_pool, pos, table) -> int:
    """Append through the page table, in place (pools: C-contiguous uint16 numpy arrays)."""
    lib = _load()
    for c in (k_pool, v_pool):
        if not (isinstance(c, np.ndarray) and c.dtype == np.uint16 and c.flags.c_contiguous):
            raise TypeError("pools must be C-contiguous uint16 numpy arrays (updated in place)")
    num_pages, g, page_size, d_h = k_pool.shape
    kn, vn = _c(k_new, np.uint16), _c(v_new, np.uint16)
    p = _c(pos, np.int32)
    tb = _c(table, np.int32)
    b, max_pages = tb.shape
    return int(lib.oracle_kv_append_paged(_ptr(kn), _ptr(vn), _ptr(k_pool), _ptr(v_pool), _ptr(p),
                                          _ptr(tb), b, g, d_h, page_size, max_pages, num_pages))


def gather_pages_u8(pool, table, page_size: int):
    """gather_pages for a pool of one-byte codes [num_pages, g, page_size, d_h] (uint8): the
    contiguous codes [b, g, max_pages * page_size, d_h]; rows of out-of-range pages are code 0 and
    the status is 4. Returns (cache, status)."""
    lib = _load()
    pl = _c(pool, np.uint8)
    tb = _c(table, np.int32)
    num_pages, g, ps, d_h = pl.shape
    if ps != page_size:
        raise ValueError("page size mismatch")
    b, max_pages = tb.shape
    out = np.empty((b, g, max_pages * page_size, d_h), dtype=np.uint8)
    st = int(lib.oracle_gather_pages_u8(_ptr(pl), _ptr(tb), b, g, d_h, page_size, max_pages,
                                        num_pages, _ptr(out)))
    if st == ERR_INVALID_ARG:
        raise ValueError("oracle rejected the arguments")
    return out, st


def kv_append_paged_multi(k_new, v_new, k_pool, v_pool, pos, table) -> int:
    """T new rows per sequence through the page table, in place (k_new [b, T, g, d_h]; pools
    C-contiguous uint16 numpy arrays)."""
    lib = _load()
    for c in (k_pool, v_pool):
        if not (isinstance(c, np.ndarray) and c.dtype == np.uint16 and c.flags.c_contiguous):
            raise TypeError("pools must be C-contiguous uint16 numpy arrays (updated in place)")
    num_pages, g, page_size, d_h = k_pool.shape
    kn, vn = _c(k_new, np.uint16), _c(v_new, np.uint16)
    b, T = kn.shape[0], kn.shape[1]
    p = _c(pos, np.int32)
    tb = _c(table, np.int32)
    max_pages = tb.shape[1]
    return int(lib.oracle_kv_append_paged_multi(_ptr(kn), _ptr(vn), _ptr(k_pool), _ptr(v_pool),
                                                _ptr(p), _ptr(tb), b, T, g, d_h, page_size,
                                                max_pages, num_pages))


def kv_append_paged_fp8(k_new, v_new, k_pool, v_pool, pos, table, k_scale: float,
                        v_scale: float) -> int:
    """The quantized append through the page table, in place (pools of codes: C-contiguous uint8
    numpy arrays [num_pages, g, page_size, d_h])."""
    lib = _load()
    for c in (k_pool, v_pool):
        if not (isinstance(c, np.ndarray) and c.dtype == np.uint8 and c.flags.c_contiguous):
            raise TypeError("pools must be C-contiguous uint8 numpy arrays (updated in place)")
    num_pages, g, page_size, d_h = k_pool.shape
    kn, vn = _c(k_new, np.uint16), _c(v_new, np.uint16)
    p = _c(pos, np.int32)
    tb = _c(table, np.int32)
    b, max_pages = tb.shape
    return int(lib.oracle_kv_append_paged_fp8(_ptr(kn), _ptr(vn), _ptr(k_pool), _ptr(v_pool),
                                              _ptr(p), _ptr(tb), b, g, d_h, page_size, max_pages,
                                              num_pages, float(k_scale), float(v_scale)))


def e4m3_to_f64(codes) -> np.ndarray:
    """E4M3 codes (uint8) -> float64 values (NaN for the two NaN codes)."""
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8)
    return np.array([lib.oracle_e4m3_to_double(int(x)) for x in c.ravel()],
                    dtype=np.float64).reshape(c.shape)


def f64_to_e4m3(x) -> np.ndarray:
    """float64 -> E4M3 codes: nearest, ties to even, saturating at +-448."""
    lib = _load()
    a = np.asarray(x, dtype=np.float64)
    return np.array([lib.oracle_double_to_e4m3(float(v)) for v in a.ravel()],
                    dtype=np.uint8).reshape(a.shape)


def dequantize_e4m3(codes, scale: float) -> np.ndarray:
    """codes * scale in float64 (any shape)."""
    lib = _load()
    c = _c(codes, np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    st = int(lib.oracle_dequantize_e4m3(_ptr(c), c.size, float(scale), _ptr(out)))
    if st:
        raise ValueError("oracle rejected the arguments")
    return out


def kv_append_fp8(k_new, v_new, k_cache, v_cache, pos, k_scale: float, v_scale: float) -> int:
    """Quantize this step's rows (bf16 bit patterns) into fp8 caches, in place (caches:
    C-contiguous uint8 numpy arrays [b, g, n_max, d_h])."""
    lib = _load()
    for c in (k_cache, v_cache):
        if not (isinstance(c, np.ndarray) and c.dtype == np.uint8 and c.flags.c_contiguous):
            raise TypeError("caches must be C-contiguous uint8 numpy arrays (updated in place)")
    b, g, n_max, d_h = k_cache.shape
    kn, vn = _c(k_new, np.uint16), _c(v_new, np.uint16)
    p = _c(pos, np.int32)
    st = int(lib.oracle_kv_append_fp8(_ptr(kn), _ptr(vn), _ptr(k_cache), _ptr(v_cache), _ptr(p),
                                      b, g, d_h, n_max, float(k_scale), float(v_scale)))
    if st == ERR_INVALID_ARG:
        raise ValueError("oracle rejected the arguments")
    return st


def decode_attention_fp8(q, k_codes, v_codes, seq_lens, k_scale: float, v_scale: float,
                         scale: float, threads: int = 0, return_status: bool = False):
    """Attention over fp8 caches: the caches dequantized (codes * scale, exact in float64), then
    :func:`decode_attention` on them with ``q`` (bf16 bit patterns) widened exactly."""
    qf = bf16_to_f64(np.asarray(q, dtype=np.uint16))
    kf = dequantize_e4m3(k_codes, k_scale)
    vf = dequantize_e4m3(v_codes, v_scale)
    return decode_attention(qf, kf, vf, seq_lens, scale, threads=threads,
                            return_status=return_status)


def kv_append_multi(k_new, v_new, k_cache, v_cache, pos) -> int:
    """Append T rows per sequence (``k_new`` [b, T, g, d_h]) at rows ``pos[b] .. pos[b]+T-1``,
    in place (caches: C-contiguous uint16 numpy arrays)."""
    lib = _load()
    for c in (k_cache, v_cache):
        if not (isinstance(c, np.ndarray) and c.dtype == np.uint16 and c.flags.c_contiguous):
            raise TypeError("caches must be C-contiguous uint16 numpy arrays (updated in place)")
    b, g, n_max, d_h = k_cache.shape
    kn, vn = _c(k_new, np.uint16), _c(v_new, np.uint16)
    T = kn.shape[1]
    p = _c(pos, np.int32)
    st = int(lib.oracle_kv_append_multi(_ptr(kn), _ptr(vn), _ptr(k_cache), _ptr(v_cache), _ptr(p),
                                        b, T, g, d_h, n_max))
    if st == ERR_INVALID_ARG:
        raise ValueError("oracle rejected the arguments")
    return st


def decode_attention_multi(q, k_cache, v_cache, seq_lens, scale: float, threads: int = 0,
                           return_status: bool = False):
    """Causal attention of T query tokens per sequence (``q`` [b, T, h, d_h], bf16 bit
    patterns) over bf16 caches; token t sees the first ``seq_lens[b] - T + 1 + t`` rows.
    Returns float64 [b, T, h, d_h]."""
    lib = _load()
    qq = _c(q, np.uint16)
    kk, vv = _c(k_cache, np.uint16), _c(v_cache, np.uint16)
    lens = _c(seq_lens, np.int32)
    b, T, h, d_h = qq.shape
    _, g, n_max, _ = kk.shape
    out = np.empty((b, T, h, d_h), dtype=np.float64)
    st = int(lib.oracle_decode_attention_multi_bf16(_ptr(qq), _ptr(kk), _ptr(vv), _ptr(lens),
                                                    _ptr(out), b, T, h, g, d_h, n_max,
                                                    float(scale), int(threads)))
    if st == ERR_INVALID_ARG:
        raise ValueError("oracle rejected the arguments")
    return (out, st) if return_status else out
