"""Python binding of libpagedattn.so (C ABI in include/pagedattn.h).

Argument marshalling only: every function checks dtypes, devices and
contiguity, then passes raw device pointers and sizes to the library, which
runs all of the work in its own CUDA kernels on the current torch stream.
torch provides device memory and streams, nothing else.

There is no fallback: if the library is missing or fails to load, every call
raises :class:`PagedAttnError`.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libpagedattn.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "pagedattn.h")

PA_OK = 0
STATUS_NAMES = {0: "PA_OK", 1: "PA_ERR_INVALID_ARG", 2: "PA_ERR_UNSUPPORTED", 3: "PA_ERR_CUDA",
                4: "PA_ERR_DEVICE_BOUNDS", 5: "PA_ERR_TIMEOUT", 6: "PA_ERR_WORKSPACE"}


class PagedAttnError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(code, code)}: {msg}")
        self.code = code


_lib = None


class StepBuffers(ctypes.Structure):
    """struct pa_step_buffers of include/pagedattn.h."""
    _vp, _i32 = ctypes.c_void_p, ctypes.c_int32
    _fields_ = [("k_cache", _vp), ("v_cache", _vp),
                ("num_blocks", _i32), ("block_size", _i32), ("num_q_heads", _i32),
                ("num_kv_heads", _i32), ("head_dim", _i32),
                ("max_tokens", _i32), ("max_seqs", _i32), ("max_blocks", _i32),
                ("max_pairs", _i32), ("max_q_len", _i32), ("max_seq_len", _i32),
                ("scale", ctypes.c_float),
                ("q", _vp), ("k_new", _vp), ("v_new", _vp), ("out", _vp),
                ("slot_mapping", _vp), ("block_tables", _vp), ("seq_lens", _vp),
                ("query_start_loc", _vp), ("copy_pairs", _vp),
                ("workspace", _vp), ("workspace_bytes", ctypes.c_size_t),
                ("host_meta", _vp), ("dev_meta", _vp), ("meta_bytes", ctypes.c_size_t),
                ("host_out", _vp), ("out_copy_bytes", ctypes.c_size_t)]


def _load() -> ctypes.CDLL:
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise PagedAttnError(-1, f"{LIB_PATH} is missing; build it with "
                                 "`python -m paged_kv_cache_174_gb300.build`")
    try:
        L = ctypes.CDLL(LIB_PATH)
    except OSError as e:  # pragma: no cover - depends on the machine
        raise PagedAttnError(-1, f"cannot load {LIB_PATH}: {e}") from e
    i32, vp, sz, f32 = ctypes.c_int32, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_float
    L.pa_version.restype = ctypes.c_int
    L.pa_get_last_error.restype = ctypes.c_char_p
    L.pa_reshape_and_cache.argtypes = [vp, vp, i32, vp, vp, i32, i32, i32, i32, vp, vp]
    L.pa_reshape_and_cache.restype = ctypes.c_int
    L.pa_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32, i32]
    L.pa_workspace_size.restype = sz
    L.pa_prefill_splits.argtypes = [i32, i32, i32, i32, i32, i32]
    L.pa_prefill_splits.restype = ctypes.c_int
    L.pa_paged_attention.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, vp, i32, vp, vp, i32,
                                     i32, i32, i32, f32, vp, vp, sz, vp]
    L.pa_paged_attention.restype = ctypes.c_int
    L.pa_paged_attention_qrange.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, vp, i32, vp, vp,
                                            i32, i32, i32, i32, i32, f32, vp, vp, sz, vp]
    L.pa_paged_attention_qrange.restype = ctypes.c_int
    L.pa_decode_step.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp, i32, vp, vp,
                                 i32, i32, i32, vp, f32, vp, vp, sz, vp]
    L.pa_decode_step.restype = ctypes.c_int
    L.pa_paged_attention_step.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp, i32,
                                          vp, vp, i32, i32, i32, i32, vp, f32, vp, vp, sz, vp]
    L.pa_paged_attention_step.restype = ctypes.c_int
    L.pa_copy_blocks.argtypes = [vp, vp, i32, i32, i32, i32, vp, i32, vp]
    L.pa_swap_staging_bytes.argtypes = [i32, i32, i32, i32]
    L.pa_swap_staging_bytes.restype = sz
    L.pa_swap_out.argtypes = [vp, vp, i32, i32, i32, i32, vp, i32, vp, vp, vp, vp]
    L.pa_swap_in.argtypes = [vp, vp, i32, i32, i32, i32, vp, i32, vp, vp, vp, vp]
    L.pa_copy_blocks.restype = ctypes.c_int
    L.pa_selftest_wait_timeout.argtypes = [ctypes.c_uint64, vp]
    L.pa_selftest_wait_timeout.restype = ctypes.c_int
    L.pa_check_device_errors.argtypes = [vp]
    L.pa_check_device_errors.restype = ctypes.c_int
    L.pa_fp8_page_bytes.argtypes = [i32, i32]
    L.pa_fp8_page_bytes.restype = sz
    L.pa_reshape_and_cache_fp8.argtypes = [vp, vp, i32, vp, vp, i32, i32, i32, i32, vp, vp]
    L.pa_reshape_and_cache_fp8.restype = ctypes.c_int
    L.pa_paged_attention_fp8.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, vp, i32,
                                         vp, vp, i32, i32, i32, i32, f32, vp, vp, sz, vp]
    L.pa_paged_attention_fp8.restype = ctypes.c_int
    L.pa_copy_blocks_fp8.argtypes = [vp, vp, i32, i32, i32, i32, vp, i32, vp]
    L.pa_copy_blocks_fp8.restype = ctypes.c_int
    L.pa_step_graph_create.argtypes = [ctypes.POINTER(StepBuffers), ctypes.POINTER(vp)]
    L.pa_step_graph_create.restype = ctypes.c_int
    L.pa_step_graph_launch.argtypes = [vp, vp]
    L.pa_step_graph_launch.restype = ctypes.c_int
    L.pa_step_graph_destroy.argtypes = [vp]
    L.pa_step_graph_destroy.restype = ctypes.c_int
    _lib = L
    return L


def lib() -> ctypes.CDLL:
    """The loaded ctypes library (raises if it is missing)."""
    return _load()


def declared_symbols() -> list:
    """Names of the functions include/pagedattn.h declares."""
    with open(HEADER_PATH) as f:
        text = f.read()
    return sorted(set(re.findall(r"\b(pa_[a-z_0-9]+)\s*\(", text)))


def _check(code: int) -> None:
    if code != PA_OK:
        msg = _load().pa_get_last_error()
        raise PagedAttnError(code, msg.decode() if msg else "")


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, dim: Optional[int] = None) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dim is not None and t.dim() != dim:
        raise ValueError(f"{name} must have {dim} dimensions, got {t.dim()}")


def _attention_shapes(q, k_cache, v_cache, block_tables, seq_lens, query_start_loc,
                      out=None):
    """Shape agreement of an attention call's tensors (the library only sees
    pointers, so a mismatch here would be an out-of-bounds access there).
    Returns (T, n_q, d, num_blocks, block_size, n_kv, S)."""
    if q.dim() != 3 or k_cache.dim() != 4:
        raise ValueError("q must be [T, n_q, d] and k_cache [num_blocks, block_size, n_kv, d]")
    T, nq, d = q.shape
    nb, bs, nkv, d2 = k_cache.shape
    if d2 != d or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("q / k_cache / v_cache head_dim or shapes disagree")
    if nkv <= 0 or nq % nkv != 0:
        raise ValueError(f"num_q_heads {nq} must be a multiple of num_kv_heads {nkv}")
    if seq_lens.dim() != 1 or query_start_loc.dim() != 1 or block_tables.dim() != 2:
        raise ValueError("seq_lens [S], query_start_loc [S+1], block_tables [S, maxb] expected")
    S = seq_lens.shape[0]
    if query_start_loc.shape[0] != S + 1 or block_tables.shape[0] != S:
        raise ValueError("seq_lens [S], query_start_loc [S+1], block_tables [S, maxb] disagree")
    if out is not None and tuple(out.shape) != tuple(q.shape):
        raise ValueError("out must have q's shape")
    return T, nq, d, nb, bs, nkv, S


def _new_rows_shapes(k, v, nkv, d, slot_mapping, name="k"):
    """k, v [T, n_kv, d] and slot_mapping [T] against a cache's n_kv, d."""
    if tuple(v.shape) != tuple(k.shape) or k.dim() != 3 or tuple(k.shape[1:]) != (nkv, d):
        raise ValueError(f"{name} / v{name[1:]} must be [T, n_kv, d] matching the cache")
    if slot_mapping.dim() != 1 or slot_mapping.shape[0] != k.shape[0]:
        raise ValueError(f"slot_mapping must be [T] with T = {name}.shape[0]")


def _need_workspace(workspace: torch.Tensor) -> None:
    if workspace.dtype != torch.uint8 or not workspace.is_cuda or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA uint8 tensor")


def _need_pairs(pairs: torch.Tensor) -> None:
    _need(pairs, "src_dst_pairs", torch.int32, 2)
    if pairs.shape[1] != 2:
        raise ValueError("src_dst_pairs must be [n, 2]")


def version() -> int:
    return int(_load().pa_version())


def reshape_and_cache(k: torch.Tensor, v: torch.Tensor, k_cache: torch.Tensor,
                      v_cache: torch.Tensor, slot_mapping: torch.Tensor, stream=None) -> None:
    """Scatter new K/V rows [T, n_kv, d] into their slots (see pa_reshape_and_cache)."""
    L = _load()
    _need(k, "k", torch.bfloat16, 3)
    _need(v, "v", torch.bfloat16, 3)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need(slot_mapping, "slot_mapping", torch.int32, 1)
    if v_cache.shape != k_cache.shape:
        raise ValueError("k_cache and v_cache shapes must match")
    nb, bs, nkv, d = k_cache.shape
    _new_rows_shapes(k, v, nkv, d, slot_mapping)
    _check(L.pa_reshape_and_cache(k.data_ptr(), v.data_ptr(), k.shape[0], k_cache.data_ptr(),
                                  v_cache.data_ptr(), nb, bs, nkv, d, slot_mapping.data_ptr(),
                                  _stream(stream)))


def workspace_size(num_seqs: int, num_tokens: int, num_q_heads: int, num_kv_heads: int,
                   head_dim: int, max_q_len: int, max_seq_len: int) -> int:
    n = int(_load().pa_workspace_size(num_seqs, num_tokens, num_q_heads, num_kv_heads, head_dim,
                                      max_q_len, max_seq_len))
    if n == 0:
        raise PagedAttnError(1, "pa_workspace_size rejected the arguments or found no device")
    return n


def prefill_splits(num_tokens: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                   max_q_len: int, max_seq_len: int) -> int:
    """Key pieces the prefill kernel uses for these sizes (1 = no split)."""
    n = int(_load().pa_prefill_splits(num_tokens, num_q_heads, num_kv_heads, head_dim,
                                      max_q_len, max_seq_len))
    if n == 0:
        raise PagedAttnError(1, "pa_prefill_splits rejected the arguments or found no device")
    return n


def alloc_workspace(num_seqs: int, num_tokens: int, num_q_heads: int, num_kv_heads: int,
                    head_dim: int, max_q_len: int, max_seq_len: int,
                    device=None) -> torch.Tensor:
    n = workspace_size(num_seqs, num_tokens, num_q_heads, num_kv_heads, head_dim, max_q_len,
                       max_seq_len)
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def paged_attention(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                    block_tables: torch.Tensor, seq_lens: torch.Tensor,
                    query_start_loc: torch.Tensor, scale: float, *, max_q_len: int,
                    max_seq_len: int, out: Optional[torch.Tensor] = None,
                    workspace: Optional[torch.Tensor] = None, stream=None,
                    min_q_len: int = 0) -> torch.Tensor:
    """Causal GQA varlen attention over the paged cache (see pa_paged_attention).

    ``max_q_len`` / ``max_seq_len`` are host-side bounds that size the launch
    without reading device memory; ``min_q_len`` >= 2 promises that no
    request has a single query row (pa_paged_attention_qrange: no decode
    launch).  Returns ``out``.
    """
    L = _load()
    _need(q, "q", torch.bfloat16, 3)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    _need(query_start_loc, "query_start_loc", torch.int32, 1)
    T, nq, d, nb, bs, nkv, S = _attention_shapes(q, k_cache, v_cache, block_tables, seq_lens,
                                                 query_start_loc, out)
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16, 3)
    if workspace is None:
        workspace = alloc_workspace(S, T, nq, nkv, d, max_q_len, max_seq_len, q.device)
    _need_workspace(workspace)
    if min_q_len >= 2:
        _check(L.pa_paged_attention_qrange(
            q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), nb, bs, nq, nkv, d,
            block_tables.data_ptr(), block_tables.shape[1], seq_lens.data_ptr(),
            query_start_loc.data_ptr(), S, T, int(min_q_len), int(max_q_len), int(max_seq_len),
            float(scale), out.data_ptr(), workspace.data_ptr(), workspace.numel(),
            _stream(stream)))
        return out
    _check(L.pa_paged_attention(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), nb, bs,
                                nq, nkv, d, block_tables.data_ptr(), block_tables.shape[1],
                                seq_lens.data_ptr(), query_start_loc.data_ptr(), S, T,
                                int(max_q_len), int(max_seq_len), float(scale), out.data_ptr(),
                                workspace.data_ptr(), workspace.numel(), _stream(stream)))
    return out


def decode_step(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
                seq_lens: torch.Tensor, query_start_loc: torch.Tensor,
                slot_mapping: torch.Tensor, scale: float, *, max_seq_len: int,
                out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                stream=None) -> torch.Tensor:
    """reshape_and_cache + paged_attention of a decode-only step in one kernel
    (pa_decode_step).  Returns ``out``."""
    L = _load()
    for name, t, dim in (("q", q, 3), ("k_new", k_new, 3), ("v_new", v_new, 3),
                         ("k_cache", k_cache, 4), ("v_cache", v_cache, 4)):
        _need(t, name, torch.bfloat16, dim)
    for name, t in (("block_tables", block_tables), ("seq_lens", seq_lens),
                    ("query_start_loc", query_start_loc), ("slot_mapping", slot_mapping)):
        _need(t, name, torch.int32)
    T, nq, d, nb, bs, nkv, S = _attention_shapes(q, k_cache, v_cache, block_tables, seq_lens,
                                                 query_start_loc, out)
    _new_rows_shapes(k_new, v_new, nkv, d, slot_mapping, name="k_new")
    if k_new.shape[0] != T:
        raise ValueError("k_new / v_new must have one row per query token")
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16, 3)
    if workspace is None:
        workspace = alloc_workspace(S, T, nq, nkv, d, 1, max_seq_len, q.device)
    _need_workspace(workspace)
    _check(L.pa_decode_step(q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(),
                            k_cache.data_ptr(), v_cache.data_ptr(), nb, bs, nq, nkv, d,
                            block_tables.data_ptr(), block_tables.shape[1], seq_lens.data_ptr(),
                            query_start_loc.data_ptr(), S, T, int(max_seq_len),
                            slot_mapping.data_ptr(), float(scale), out.data_ptr(),
                            workspace.data_ptr(), workspace.numel(), _stream(stream)))
    return out


def attention_step(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                   k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
                   seq_lens: torch.Tensor, query_start_loc: torch.Tensor,
                   slot_mapping: torch.Tensor, scale: float, *, max_q_len: int, max_seq_len: int,
                   out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                   stream=None) -> torch.Tensor:
    """reshape_and_cache + paged_attention of a step with any mix of decode and
    chunked-prefill rows, the scatter done inside the attention kernels
    (pa_paged_attention_step).  Returns ``out``."""
    L = _load()
    for name, t, dim in (("q", q, 3), ("k_new", k_new, 3), ("v_new", v_new, 3),
                         ("k_cache", k_cache, 4), ("v_cache", v_cache, 4)):
        _need(t, name, torch.bfloat16, dim)
    for name, t in (("block_tables", block_tables), ("seq_lens", seq_lens),
                    ("query_start_loc", query_start_loc), ("slot_mapping", slot_mapping)):
        _need(t, name, torch.int32)
    T, nq, d, nb, bs, nkv, S = _attention_shapes(q, k_cache, v_cache, block_tables, seq_lens,
                                                 query_start_loc, out)
    _new_rows_shapes(k_new, v_new, nkv, d, slot_mapping, name="k_new")
    if k_new.shape[0] != T:
        raise ValueError("k_new / v_new must have one row per query token")
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16, 3)
    if workspace is None:
        workspace = alloc_workspace(S, T, nq, nkv, d, max_q_len, max_seq_len, q.device)
    _need_workspace(workspace)
    _check(L.pa_paged_attention_step(q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(),
                                     k_cache.data_ptr(), v_cache.data_ptr(), nb, bs, nq, nkv, d,
                                     block_tables.data_ptr(), block_tables.shape[1],
                                     seq_lens.data_ptr(), query_start_loc.data_ptr(), S, T,
                                     int(max_q_len), int(max_seq_len), slot_mapping.data_ptr(),
                                     float(scale), out.data_ptr(), workspace.data_ptr(),
                                     workspace.numel(), _stream(stream)))
    return out


def copy_blocks(k_cache: torch.Tensor, v_cache: torch.Tensor, src_dst_pairs: torch.Tensor,
                stream=None) -> None:
    """Copy-on-write: block dst <- block src for each (src, dst) row."""
    L = _load()
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need_pairs(src_dst_pairs)
    if v_cache.shape != k_cache.shape:
        raise ValueError("k_cache and v_cache shapes must match")
    nb, bs, nkv, d = k_cache.shape
    _check(L.pa_copy_blocks(k_cache.data_ptr(), v_cache.data_ptr(), nb, bs, nkv, d,
                            src_dst_pairs.data_ptr(), src_dst_pairs.shape[0], _stream(stream)))


def _swap(out: bool, k_cache, v_cache, block_ids, host_k, host_v, staging, stream):
    L = _load()
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need(block_ids, "block_ids", torch.int32, 1)
    nb, bs, nkv, d = k_cache.shape
    n = int(block_ids.shape[0])
    for name, h in (("host_k", host_k), ("host_v", host_v)):
        if h.device.type != "cpu" or h.dtype != torch.bfloat16 or not h.is_contiguous():
            raise TypeError(f"{name} must be a contiguous bf16 CPU tensor (pinned for overlap)")
        if tuple(h.shape) != (n, bs, nkv, d):
            raise ValueError(f"{name} must be [{n}, {bs}, {nkv}, {d}]")
    need = int(L.pa_swap_staging_bytes(n, bs, nkv, d))
    if staging is None:
        staging = torch.empty(need // 2, dtype=torch.bfloat16, device=k_cache.device)
    elif staging.numel() * staging.element_size() < need or staging.device != k_cache.device:
        raise ValueError(f"staging must be a device buffer of >= {need} bytes")
    fn = L.pa_swap_out if out else L.pa_swap_in
    _check(fn(k_cache.data_ptr(), v_cache.data_ptr(), nb, bs, nkv, d, block_ids.data_ptr(), n,
              staging.data_ptr(), host_k.data_ptr(), host_v.data_ptr(), _stream(stream)))
    return staging


def swap_out(k_cache: torch.Tensor, v_cache: torch.Tensor, block_ids: torch.Tensor,
             host_k: torch.Tensor, host_v: torch.Tensor, staging: Optional[torch.Tensor] = None,
             stream=None) -> torch.Tensor:
    """Blocks block_ids of both caches -> host_k / host_v ([n, bs, n_kv, d] bf16 CPU
    tensors, pinned for the copy to be asynchronous); valid once the stream has
    synchronised.  Returns the device staging buffer (reusable)."""
    return _swap(True, k_cache, v_cache, block_ids, host_k, host_v, staging, stream)


def swap_in(k_cache: torch.Tensor, v_cache: torch.Tensor, block_ids: torch.Tensor,
            host_k: torch.Tensor, host_v: torch.Tensor, staging: Optional[torch.Tensor] = None,
            stream=None) -> torch.Tensor:
    """host_k / host_v -> blocks block_ids (distinct) of both caches."""
    return _swap(False, k_cache, v_cache, block_ids, host_k, host_v, staging, stream)


# ---------------------------------------------------------------------------
# 8-bit (FP8 E4M3) cache: uint8 [num_blocks, block_size // 16, page bytes],
# each 16-token page its codes [16, n_kv, d], then their fp32 scales
# [16, n_kv] (one per cached row).
# ---------------------------------------------------------------------------

FP8_PAGE_TOKENS = 16


def fp8_page_bytes(num_kv_heads: int, head_dim: int) -> int:
    """Bytes of one 16-token page of the 8-bit cache (codes, then scales)."""
    return FP8_PAGE_TOKENS * num_kv_heads * (head_dim + 4)


def empty_fp8_cache(num_blocks: int, block_size: int, num_kv_heads: int, head_dim: int,
                    device=None):
    """(k cache, v cache): uint8 [num_blocks, block_size // 16, page bytes],
    zero-filled, on the device."""
    if block_size % FP8_PAGE_TOKENS:
        raise ValueError(f"block_size {block_size} is not a multiple of {FP8_PAGE_TOKENS}")
    dev = device or "cuda"
    shape = (num_blocks, block_size // FP8_PAGE_TOKENS, fp8_page_bytes(num_kv_heads, head_dim))
    return (torch.zeros(shape, dtype=torch.uint8, device=dev),
            torch.zeros(shape, dtype=torch.uint8, device=dev))


def fp8_cache_views(cache: torch.Tensor, num_kv_heads: int, head_dim: int):
    """(codes, scales) views of an 8-bit cache: codes uint8 [num_blocks,
    block_size // 16, 16, n_kv, d] and scales fp32 [num_blocks,
    block_size // 16, 16, n_kv]; token row r of page p of block b is slot
    b * block_size + 16 p + r."""
    nb, npg, pb = cache.shape
    if pb != fp8_page_bytes(num_kv_heads, head_dim):
        raise ValueError(f"page of {pb} bytes is not one of n_kv {num_kv_heads}, d {head_dim}")
    cb = FP8_PAGE_TOKENS * num_kv_heads * head_dim
    codes = cache[:, :, :cb].view(nb, npg, FP8_PAGE_TOKENS, num_kv_heads, head_dim)
    scales = cache[:, :, cb:].view(torch.float32).view(nb, npg, FP8_PAGE_TOKENS, num_kv_heads)
    return codes, scales


def _fp8_geometry(k_cache, v_cache, num_kv_heads: int, head_dim: int):
    """(num_blocks, block_size) of a pair of 8-bit caches."""
    _need(k_cache, "k_cache", torch.uint8, 3)
    _need(v_cache, "v_cache", torch.uint8, 3)
    if v_cache.shape != k_cache.shape or \
            k_cache.shape[2] != fp8_page_bytes(num_kv_heads, head_dim):
        raise ValueError("caches must be alike, uint8 [num_blocks, block_size // 16, "
                         f"{fp8_page_bytes(num_kv_heads, head_dim)}] for n_kv {num_kv_heads}, "
                         f"d {head_dim}")
    return k_cache.shape[0], k_cache.shape[1] * FP8_PAGE_TOKENS


def reshape_and_cache_fp8(k: torch.Tensor, v: torch.Tensor, k_cache: torch.Tensor,
                          v_cache: torch.Tensor, slot_mapping: torch.Tensor, stream=None) -> None:
    """Quantise each new (token, kv head) row of k / v into its slot."""
    L = _load()
    _need(k, "k", torch.bfloat16, 3)
    _need(v, "v", torch.bfloat16, 3)
    _need(slot_mapping, "slot_mapping", torch.int32, 1)
    nkv, d = k.shape[1], k.shape[2]
    nb, bs = _fp8_geometry(k_cache, v_cache, nkv, d)
    _new_rows_shapes(k, v, nkv, d, slot_mapping)
    _check(L.pa_reshape_and_cache_fp8(k.data_ptr(), v.data_ptr(), k.shape[0], k_cache.data_ptr(),
                                      v_cache.data_ptr(), nb, bs, nkv, d,
                                      slot_mapping.data_ptr(), _stream(stream)))


def paged_attention_fp8(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                        block_tables: torch.Tensor, seq_lens: torch.Tensor,
                        query_start_loc: torch.Tensor, scale: float, *, max_q_len: int,
                        max_seq_len: int, out: Optional[torch.Tensor] = None,
                        workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """paged_attention over the 8-bit cache (decode and prefill rows); n_kv
    follows from the page size and q's head_dim."""
    L = _load()
    _need(q, "q", torch.bfloat16, 3)
    T, nq, d = q.shape
    _need(k_cache, "k_cache", torch.uint8, 3)
    nkv = k_cache.shape[2] // fp8_page_bytes(1, d)
    nb, bs = _fp8_geometry(k_cache, v_cache, nkv, d)
    if nkv <= 0 or nq % nkv != 0:
        raise ValueError(f"num_q_heads {nq} must be a multiple of num_kv_heads {nkv}")
    for name, t in (("block_tables", block_tables), ("seq_lens", seq_lens),
                    ("query_start_loc", query_start_loc)):
        _need(t, name, torch.int32)
    if block_tables.dim() != 2 or seq_lens.dim() != 1 or query_start_loc.dim() != 1:
        raise ValueError("block_tables must be 2-D, seq_lens and query_start_loc 1-D")
    S = seq_lens.shape[0]
    if block_tables.shape[0] != S or query_start_loc.shape[0] != S + 1:
        raise ValueError("block_tables [S, max_blocks], seq_lens [S], query_start_loc [S + 1]")
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16, 3)
    if out.shape != q.shape:
        raise ValueError("out must have q's shape")
    if workspace is None:
        workspace = alloc_workspace(S, T, nq, nkv, d, max_q_len, max_seq_len, q.device)
    _need_workspace(workspace)
    _check(L.pa_paged_attention_fp8(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                    nb, bs, nq, nkv, d, block_tables.data_ptr(),
                                    block_tables.shape[1], seq_lens.data_ptr(),
                                    query_start_loc.data_ptr(), S, T, int(max_q_len),
                                    int(max_seq_len), float(scale), out.data_ptr(),
                                    workspace.data_ptr(), workspace.numel(), _stream(stream)))
    return out


def copy_blocks_fp8(k_cache, v_cache, src_dst_pairs: torch.Tensor, *, num_kv_heads: int,
                    head_dim: int, stream=None) -> None:
    """Copy-on-write on the 8-bit cache: the pages (codes and scales) of block
    dst <- block src."""
    L = _load()
    nb, bs = _fp8_geometry(k_cache, v_cache, num_kv_heads, head_dim)
    _need_pairs(src_dst_pairs)
    _check(L.pa_copy_blocks_fp8(k_cache.data_ptr(), v_cache.data_ptr(), nb, bs, num_kv_heads,
                                head_dim, src_dst_pairs.data_ptr(), src_dst_pairs.shape[0],
                                _stream(stream)))


def selftest_wait_timeout(limit_ns: int = 5_000_000, stream=None) -> None:
    """Run the kernels' bounded wait on a barrier nothing completes (see
    pa_selftest_wait_timeout); check_device_errors then raises PA_ERR_TIMEOUT."""
    _check(_load().pa_selftest_wait_timeout(int(limit_ns), _stream(stream)))


def check_device_errors(stream=None) -> None:
    """Synchronise the stream and raise if a kernel flagged an error."""
    _check(_load().pa_check_device_errors(_stream(stream)))


class StepGraph:
    """One serving step (block copies, slot scatter, attention) captured as a
    CUDA graph by the library (pa_step_graph_create) over fixed buffers sized
    for the largest step.

    Per step: write the step's q / k_new / v_new rows (first num_tokens rows),
    then call :meth:`launch` with the step's integer inputs as host arrays (or
    :meth:`stage` them first and call :meth:`launch` with none); they are
    padded to the maxima in a pinned buffer.  ``stream`` is a
    torch.cuda.Stream or None (the current stream).

    * ``host_io=False``: q / k_new / v_new / out are device tensors
      (``self.q`` ...); the graph's own first node copies the integer inputs
      from the pinned buffer.  Two graphs alternate over two pinned buffers,
      so the host fills one while the GPU may still read the other.
    * ``host_io=True``: a step's whole input (integer arrays and q / k_new /
      v_new) sits in one pinned region (fill the views :meth:`inputs_host`
      returns) and its output comes back into pinned memory
      (:meth:`output_host`, after :meth:`wait_output`).  Two graphs
      alternate over two device copies of the region; each launch copies its
      region in on one side stream and its output out on another, so the copy
      of step i+1's inputs and of step i's output overlap step i's kernels.
      :meth:`fork` / :meth:`join` order the side streams after / before a
      point of the launching stream (to time a run of launches).
    """

    def __init__(self, k_cache: torch.Tensor, v_cache: torch.Tensor, *, num_q_heads: int,
                 max_tokens: int, max_seqs: int, max_blocks: int, max_pairs: int,
                 max_q_len: int, max_seq_len: int, scale: float, host_io: bool = False):
        import numpy as np
        L = _load()
        _need(k_cache, "k_cache", torch.bfloat16, 4)
        _need(v_cache, "v_cache", torch.bfloat16, 4)
        if v_cache.shape != k_cache.shape:
            raise ValueError("k_cache and v_cache shapes differ")
        nb, bs, nkv, d = k_cache.shape
        dev = k_cache.device
        self.device = dev
        T, S, MB, P = int(max_tokens), int(max_seqs), int(max_blocks), int(max_pairs)
        self.max_tokens, self.max_seqs, self.max_blocks, self.max_pairs = T, S, MB, P
        # int32 metadata: slots [T] | tables [S*MB] | seq_lens [S] | qsl [S+1] | pairs [2P]
        self._off = np.cumsum([0, T, S * MB, S, S + 1, 2 * P])
        n = int(self._off[-1])
        meta_bytes = -(-4 * n // 256) * 256
        q_bytes, kv_bytes = T * num_q_heads * d * 2, T * nkv * d * 2
        total = meta_bytes + (q_bytes + 2 * kv_bytes if host_io else 0)
        self.host_io = host_io

        def bf16_views(region):
            q0, k0, v0 = meta_bytes, meta_bytes + q_bytes, meta_bytes + q_bytes + kv_bytes
            return (region[q0:k0].view(torch.bfloat16).view(T, num_q_heads, d),
                    region[k0:v0].view(torch.bfloat16).view(T, nkv, d),
                    region[v0:v0 + kv_bytes].view(torch.bfloat16).view(T, nkv, d))

        self._host_region = [torch.zeros(total, dtype=torch.uint8).pin_memory() for _ in range(2)]
        self._host = [h[:4 * n].view(torch.int32) for h in self._host_region]
        self.workspace = alloc_workspace(S, T, num_q_heads, nkv, d, max_q_len, max_seq_len, dev)
        if host_io:
            self._dev_region = [torch.zeros(total, dtype=torch.uint8, device=dev)
                                for _ in range(2)]
            self._dev_in = [bf16_views(r) for r in self._dev_region]
            self._host_inputs = [bf16_views(h) for h in self._host_region]
            self._out = [torch.zeros(T, num_q_heads, d, dtype=torch.bfloat16, device=dev)
                         for _ in range(2)]
            self._out_host = [torch.zeros(T, num_q_heads, d, dtype=torch.bfloat16).pin_memory()
                              for _ in range(2)]
            self._h2d = torch.cuda.Stream(dev)
            self._d2h = torch.cuda.Stream(dev)
            self._in_ready = [None, None]
            self._comp_done = [None, None]
            self._out_ready = [None, None]
        else:
            self._dev_region = [torch.zeros(total, dtype=torch.uint8, device=dev)] * 2
            self.q = torch.zeros(T, num_q_heads, d, dtype=torch.bfloat16, device=dev)
            self.k_new = torch.zeros(T, nkv, d, dtype=torch.bfloat16, device=dev)
            self.v_new = torch.zeros(T, nkv, d, dtype=torch.bfloat16, device=dev)
            self.out = torch.zeros(T, num_q_heads, d, dtype=torch.bfloat16, device=dev)
            self._dev_in = [(self.q, self.k_new, self.v_new)] * 2
            self._out = [self.out] * 2
            self._events = [None, None]
        self._graphs = []
        for i in range(2):
            base = self._dev_region[i].data_ptr()
            o = [base + 4 * int(x) for x in self._off]
            q, k, v = self._dev_in[i]
            b = StepBuffers(k_cache.data_ptr(), v_cache.data_ptr(), nb, bs, num_q_heads, nkv, d,
                            T, S, MB, P, int(max_q_len), int(max_seq_len), float(scale),
                            q.data_ptr(), k.data_ptr(), v.data_ptr(), self._out[i].data_ptr(),
                            o[0], o[1], o[2], o[3], o[4] if P else None,
                            self.workspace.data_ptr(), self.workspace.numel(),
                            None if host_io else self._host_region[i].data_ptr(),
                            base, 4 * n, None, 0)
            g = ctypes.c_void_p()
            _check(L.pa_step_graph_create(ctypes.byref(b), ctypes.byref(g)))
            self._graphs.append(g)
        self.input_bytes = total if host_io else 4 * n   # copied in by every launch
        self.output_bytes = q_bytes if host_io else 0    # copied out by every launch
        self._last = None
        self._next = 0
        self._staged = False
        self._filled = [False, False]    # buffer i holds a staged step
        self._keep = (k_cache, v_cache)  # the graphs hold their pointers

    def _free_host_buffer(self, i: int) -> None:
        """Block until buffer i's pinned input region may be rewritten."""
        ev = self._in_ready[i] if self.host_io else self._events[i]
        if ev is not None:
            ev.synchronize()

    def launch(self, slot_mapping=None, block_tables=None, seq_lens=None, query_start_loc=None,
               copy_pairs=None, stream=None, copy_in: bool = True,
               copy_out: bool = True) -> None:
        """Launch the staged step.  With host_io, copy_in=False reuses the
        device copy of the buffer's inputs from its last launch (inputs
        already resident) and copy_out=False leaves out on the device."""
        if slot_mapping is not None:
            self.stage(slot_mapping, block_tables, seq_lens, query_start_loc, copy_pairs)
        if not self._staged:
            raise ValueError("no step staged")
        i = self._next
        main = torch.cuda.current_stream(self.device) if stream is None else stream
        if self.host_io and copy_in:
            if self._comp_done[i] is not None:
                self._h2d.wait_event(self._comp_done[i])  # its last graph is done with it
            with torch.cuda.stream(self._h2d):
                self._dev_region[i].copy_(self._host_region[i], non_blocking=True)
                self._in_ready[i] = torch.cuda.Event()
                self._in_ready[i].record(self._h2d)
        if self.host_io and self._in_ready[i] is not None:
            main.wait_event(self._in_ready[i])
        _check(_load().pa_step_graph_launch(self._graphs[i], main.cuda_stream))
        done = torch.cuda.Event()
        done.record(main)
        if self.host_io:
            self._comp_done[i] = done
            if copy_out:
                self._d2h.wait_event(done)
                with torch.cuda.stream(self._d2h):
                    self._out_host[i].copy_(self._out[i], non_blocking=True)
                    self._out_ready[i] = torch.cuda.Event()
                    self._out_ready[i].record(self._d2h)
        else:
            self._events[i] = done
        self._last = i
        self._next = 1 - i
        self._staged = False

    def relaunch(self, stream=None, copy_in: bool = True, copy_out: bool = True) -> None:
        """Launch the next buffer's inputs as they stand (the step it last
        held, with whatever the caller rewrote in place since)."""
        if not self._filled[self._next]:
            raise ValueError("the next buffer has never been staged")
        if copy_in:
            self._free_host_buffer(self._next)
        self._staged = True
        self.launch(stream=stream, copy_in=copy_in, copy_out=copy_out)

    def inputs_host(self):
        """(q, k_new, v_new) pinned views for the next launch (host_io)."""
        if not self.host_io:
            raise ValueError("the graph was built without host_io")
        self._free_host_buffer(self._next)
        return self._host_inputs[self._next]

    def wait_output(self) -> None:
        """Block until the last launch's output is in pinned memory (host_io)."""
        if self.host_io and self._last is not None and self._out_ready[self._last] is not None:
            self._out_ready[self._last].synchronize()

    def output_host(self) -> torch.Tensor:
        """Pinned copy of out from the last launch (host_io; call wait_output
        first)."""
        if not self.host_io or self._last is None:
            raise ValueError("no host_io launch yet")
        return self._out_host[self._last]

    def output(self) -> torch.Tensor:
        """Device out of the last launch."""
        return self._out[self._last if self._last is not None else 0]

    def fork(self, stream=None) -> None:
        """Order the side copy streams after everything issued so far on stream."""
        if self.host_io:
            main = torch.cuda.current_stream(self.device) if stream is None else stream
            ev = torch.cuda.Event()
            ev.record(main)
            self._h2d.wait_event(ev)
            self._d2h.wait_event(ev)

    def join(self, stream=None) -> None:
        """Make stream wait for the last launch's output copy."""
        if self.host_io and self._last is not None:
            main = torch.cuda.current_stream(self.device) if stream is None else stream
            main.wait_event(self._out_ready[self._last])

    def stage(self, slot_mapping, block_tables, seq_lens, query_start_loc,
              copy_pairs=None) -> None:
        """Pad the step's integer inputs into the pinned buffer of the next launch."""
        import numpy as np
        T, S, MB, P = self.max_tokens, self.max_seqs, self.max_blocks, self.max_pairs
        sm = np.asarray(slot_mapping, np.int32).reshape(-1)
        bt = np.asarray(block_tables, np.int32)
        sl = np.asarray(seq_lens, np.int32).reshape(-1)
        qsl = np.asarray(query_start_loc, np.int32).reshape(-1)
        cp = np.zeros((0, 2), np.int32) if copy_pairs is None else \
            np.asarray(copy_pairs, np.int32).reshape(-1, 2)
        ns = sl.shape[0]
        if (sm.shape[0] > T or ns > S or bt.shape[0] != ns or bt.shape[1] > MB
                or qsl.shape[0] != ns + 1 or cp.shape[0] > P):
            raise ValueError(f"step beyond the graph's maxima (tokens {sm.shape[0]}/{T}, "
                             f"seqs {ns}/{S}, table columns {bt.shape[1]}/{MB}, "
                             f"pairs {cp.shape[0]}/{P}) or inconsistent shapes")
        i = self._next
        self._free_host_buffer(i)
        h = self._host[i].numpy()
        o = self._off
        h[o[0]:o[1]] = -1
        h[o[0]:o[0] + sm.shape[0]] = sm
        tab = h[o[1]:o[2]].reshape(S, MB)
        tab[:] = -1
        tab[:ns, :bt.shape[1]] = bt
        h[o[2]:o[3]] = 0
        h[o[2]:o[2] + ns] = sl
        h[o[3]:o[4]] = qsl[-1] if ns else 0
        h[o[3]:o[3] + ns + 1] = qsl
        if P:
            pr = h[o[4]:o[5]].reshape(P, 2)
            pr[:] = -1
            pr[:cp.shape[0]] = cp
        self._staged = True
        self._filled[i] = True

    def close(self) -> None:
        for g in getattr(self, "_graphs", []):
            _load().pa_step_graph_destroy(g)
        self._graphs = []

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
