"""fp64 CPU oracle for attention over a paged KV cache.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference arm are the only callers.  The product
path (``paged_kv_cache_174_gb300``) never imports this package, and this
package never imports the product.  Arrays are numpy; bfloat16 tensors are
passed as their raw 16-bit patterns (``np.uint16``), which the C code decodes
itself.

What it computes, and which page passage each function follows, is stated in
``oracle.c``.  Every function here is a thin ctypes marshaller over it.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_LIB = None


def lib() -> ctypes.CDLL:
    global _LIB
    if _LIB is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        i32, i64, dbl, vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
        L.oracle_num_threads.restype = ctypes.c_int
        L.oracle_slot_of.argtypes = [vp, i32, i32]
        L.oracle_slot_of.restype = i64
        L.oracle_reshape_and_cache.argtypes = [vp, vp, i32, vp, vp, i32, i32, i32, i32, vp]
        L.oracle_reshape_and_cache.restype = ctypes.c_int
        L.oracle_copy_blocks.argtypes = [vp, vp, i32, i32, i32, i32, vp, i32]
        L.oracle_copy_blocks.restype = ctypes.c_int
        L.oracle_swap_out.argtypes = [vp, vp, i32, i32, i32, i32, vp, i32, vp, vp]
        L.oracle_swap_out.restype = ctypes.c_int
        L.oracle_swap_in.argtypes = [vp, vp, i32, i32, i32, i32, vp, i32, vp, vp]
        L.oracle_swap_in.restype = ctypes.c_int
        L.oracle_paged_attention.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32,
                                             vp, i32, vp, vp, i32, dbl, vp, i32]
        L.oracle_paged_attention.restype = ctypes.c_int
        L.oracle_paged_attention_rows.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32,
                                                  vp, i32, vp, vp, i32, dbl, vp, i32,
                                                  vp, i32]
        L.oracle_paged_attention_rows.restype = ctypes.c_int
        L.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
        L.oracle_e4m3_to_double.restype = dbl
        L.oracle_e4m3_from_float.argtypes = [ctypes.c_float]
        L.oracle_e4m3_from_float.restype = ctypes.c_uint8
        L.oracle_reshape_and_cache_fp8.argtypes = [vp, vp, i32, vp, vp, vp, vp, i32, i32, i32,
                                                   i32, vp]
        L.oracle_reshape_and_cache_fp8.restype = ctypes.c_int
        L.oracle_paged_attention_fp8.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                                 vp, i32, vp, vp, i32, dbl, vp, i32]
        L.oracle_paged_attention_fp8.restype = ctypes.c_int
        _LIB = L
    return _LIB


class OracleError(RuntimeError):
    pass


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _c(a, dtype) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def num_threads() -> int:
    return int(lib().oracle_num_threads())


def slot_of(block_table_row, pos: int, block_size: int) -> int:
    row = _c(block_table_row, np.int32)
    return int(lib().oracle_slot_of(_ptr(row), int(pos), int(block_size)))


def reshape_and_cache(k, v, k_cache: np.ndarray, v_cache: np.ndarray, slot_mapping) -> None:
    """In place on k_cache / v_cache ([num_blocks, block_size, n_kv, d] uint16)."""
    assert k_cache.dtype == np.uint16 and k_cache.flags.c_contiguous
    assert v_cache.dtype == np.uint16 and v_cache.flags.c_contiguous
    k = _c(k, np.uint16)
    v = _c(v, np.uint16)
    sm = _c(slot_mapping, np.int32)
    nb, bs, nkv, d = k_cache.shape
    st = lib().oracle_reshape_and_cache(_ptr(k), _ptr(v), int(sm.shape[0]), _ptr(k_cache),
                                        _ptr(v_cache), nb, bs, nkv, d, _ptr(sm))
    if st:
        raise OracleError(f"oracle_reshape_and_cache status {st}")


def copy_blocks(k_cache: np.ndarray, v_cache: np.ndarray, pairs) -> None:
    """In place; pairs is [n, 2] int (src, dst)."""
    assert k_cache.dtype == np.uint16 and k_cache.flags.c_contiguous
    p = _c(pairs, np.int32).reshape(-1, 2)
    nb, bs, nkv, d = k_cache.shape
    st = lib().oracle_copy_blocks(_ptr(k_cache), _ptr(v_cache), nb, bs, nkv, d, _ptr(p),
                                  int(p.shape[0]))
    if st:
        raise OracleError(f"oracle_copy_blocks status {st}")


def swap_out(k_cache: np.ndarray, v_cache: np.ndarray, block_ids):
    """Returns (host_k, host_v), each [n, block_size, n_kv, d] uint16: the blocks
    block_ids[i] of the caches, in list order."""
    kc = _c(k_cache, np.uint16)
    vc = _c(v_cache, np.uint16)
    ids = _c(block_ids, np.int32).reshape(-1)
    nb, bs, nkv, d = kc.shape
    hk = np.empty((ids.shape[0], bs, nkv, d), np.uint16)
    hv = np.empty_like(hk)
    st = lib().oracle_swap_out(_ptr(kc), _ptr(vc), nb, bs, nkv, d, _ptr(ids), int(ids.shape[0]),
                               _ptr(hk), _ptr(hv))
    if st:
        raise OracleError(f"oracle_swap_out status {st}")
    return hk, hv


def swap_in(k_cache: np.ndarray, v_cache: np.ndarray, block_ids, host_k, host_v) -> None:
    """In place: block block_ids[i] of the caches <- host_k[i], host_v[i]."""
    assert k_cache.dtype == np.uint16 and k_cache.flags.c_contiguous
    assert v_cache.dtype == np.uint16 and v_cache.flags.c_contiguous
    ids = _c(block_ids, np.int32).reshape(-1)
    hk = _c(host_k, np.uint16)
    hv = _c(host_v, np.uint16)
    nb, bs, nkv, d = k_cache.shape
    assert hk.shape == (ids.shape[0], bs, nkv, d) and hv.shape == hk.shape
    st = lib().oracle_swap_in(_ptr(k_cache), _ptr(v_cache), nb, bs, nkv, d, _ptr(ids),
                              int(ids.shape[0]), _ptr(hk), _ptr(hv))
    if st:
        raise OracleError(f"oracle_swap_in status {st}")


def paged_attention(q, k_cache, v_cache, block_tables, seq_lens, query_start_loc,
                    scale: float, threads: int = 0) -> np.ndarray:
    """Returns fp64 out [num_tokens, n_q, d]; rows owned by no sequence are NaN."""
    q = _c(q, np.uint16)
    kc = _c(k_cache, np.uint16)
    vc = _c(v_cache, np.uint16)
    bt = _c(block_tables, np.int32)
    sl = _c(seq_lens, np.int32)
    qsl = _c(query_start_loc, np.int32)
    T, nq, d = q.shape
    nb, bs, nkv, d2 = kc.shape
    assert d == d2
    S = int(sl.shape[0])
    maxb = int(bt.shape[1]) if bt.ndim == 2 else 0
    out = np.full((T, nq, d), np.nan, dtype=np.float64)
    st = lib().oracle_paged_attention(_ptr(q), _ptr(kc), _ptr(vc), nb, bs, nq, nkv, d,
                                      _ptr(bt), maxb, _ptr(sl), _ptr(qsl), S, float(scale),
                                      _ptr(out), int(threads))
    if st:
        raise OracleError(f"oracle_paged_attention status {st}")
    return out


def paged_attention_rows(q, k_cache, v_cache, block_tables, seq_lens, query_start_loc,
                         scale: float, samples, threads: int = 0) -> np.ndarray:
    """samples: [n, 3] (sequence, row within the sequence, q head) -> fp64 [n, d]."""
    q = _c(q, np.uint16)
    kc = _c(k_cache, np.uint16)
    vc = _c(v_cache, np.uint16)
    bt = _c(block_tables, np.int32)
    sl = _c(seq_lens, np.int32)
    qsl = _c(query_start_loc, np.int32)
    smp = _c(samples, np.int32).reshape(-1, 3)
    T, nq, d = q.shape
    nb, bs, nkv, _ = kc.shape
    out = np.full((smp.shape[0], d), np.nan, dtype=np.float64)
    st = lib().oracle_paged_attention_rows(_ptr(q), _ptr(kc), _ptr(vc), nb, bs, nq, nkv, d,
                                           _ptr(bt), int(bt.shape[1]), _ptr(sl), _ptr(qsl),
                                           int(sl.shape[0]), float(scale), _ptr(smp),
                                           int(smp.shape[0]), _ptr(out), int(threads))
    if st:
        raise OracleError(f"oracle_paged_attention_rows status {st}")
    return out


# ---------------------------------------------------------------------------
# The 8-bit (FP8 E4M3) cache variant, defined in oracle.c's header comment.
# ---------------------------------------------------------------------------

def e4m3_to_double(codes) -> np.ndarray:
    """Values of E4M3 codes (uint8 array), exact, as fp64."""
    c = np.asarray(codes, np.uint8)
    f = lib().oracle_e4m3_to_double
    return np.array([f(int(x)) for x in c.reshape(-1)], np.float64).reshape(c.shape)


def e4m3_from_float(values) -> np.ndarray:
    """fp32 values -> E4M3 codes (nearest, ties to even, saturating at 448)."""
    v = np.asarray(values, np.float32)
    f = lib().oracle_e4m3_from_float
    return np.array([f(float(x)) for x in v.reshape(-1)], np.uint8).reshape(v.shape)


def fp8_cache(num_blocks: int, block_size: int, num_kv_heads: int, head_dim: int,
              fill_code: int = 0x7F):
    """Empty 8-bit cache: (k codes, v codes, k scales, v scales); codes filled
    with fill_code (NaN by default), scales with NaN."""
    shape = (num_blocks, block_size, num_kv_heads, head_dim)
    kc = np.full(shape, fill_code, np.uint8)
    vc = np.full(shape, fill_code, np.uint8)
    ks = np.full(shape[:3], np.nan, np.float32)
    vs = np.full(shape[:3], np.nan, np.float32)
    return kc, vc, ks, vs


def reshape_and_cache_fp8(k, v, k_cache, v_cache, k_scale, v_scale, slot_mapping) -> None:
    """In place: quantise each new (token, kv head) row into the 8-bit cache."""
    for a, dt in ((k_cache, np.uint8), (v_cache, np.uint8), (k_scale, np.float32),
                  (v_scale, np.float32)):
        assert a.dtype == dt and a.flags.c_contiguous
    k = _c(k, np.uint16)
    v = _c(v, np.uint16)
    sm = _c(slot_mapping, np.int32)
    nb, bs, nkv, d = k_cache.shape
    st = lib().oracle_reshape_and_cache_fp8(_ptr(k), _ptr(v), int(sm.shape[0]), _ptr(k_cache),
                                            _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), nb,
                                            bs, nkv, d, _ptr(sm))
    if st:
        raise OracleError(f"oracle_reshape_and_cache_fp8 status {st}")


def paged_attention_fp8(q, k_cache, v_cache, k_scale, v_scale, block_tables, seq_lens,
                        query_start_loc, scale: float, threads: int = 0) -> np.ndarray:
    """oracle paged attention with every cached value = code * row scale."""
    q = _c(q, np.uint16)
    kc = _c(k_cache, np.uint8)
    vc = _c(v_cache, np.uint8)
    ks = _c(k_scale, np.float32)
    vs = _c(v_scale, np.float32)
    bt = _c(block_tables, np.int32)
    sl = _c(seq_lens, np.int32)
    qsl = _c(query_start_loc, np.int32)
    T, nq, d = q.shape
    nb, bs, nkv, d2 = kc.shape
    assert d == d2 and ks.shape == (nb, bs, nkv) and vs.shape == ks.shape
    S = int(sl.shape[0])
    maxb = int(bt.shape[1]) if bt.ndim == 2 else 0
    out = np.full((T, nq, d), np.nan, dtype=np.float64)
    st = lib().oracle_paged_attention_fp8(_ptr(q), _ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs), nb,
                                          bs, nq, nkv, d, _ptr(bt), maxb, _ptr(sl), _ptr(qsl),
                                          S, float(scale), _ptr(out), int(threads))
    if st:
        raise OracleError(f"oracle_paged_attention_fp8 status {st}")
    return out
