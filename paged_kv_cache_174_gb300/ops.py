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
    L.pa_copy_blocks.argtypes = [vp, vp, i32, i32, i32, i32, vp, i32, vp]
    L.pa_swap_staging_bytes.argtypes = [i32, i32, i32, i32]
    L.pa_swap_staging_bytes.restype = sz
    L.pa_swap_out.argtypes = [vp, vp, i32, i32, i32, i32, vp, i32, vp, vp, vp, vp]
    L.pa_swap_in.argtypes = [vp, vp, i32, i32, i32, i32, vp, i32, vp, vp, vp, vp]
    L.pa_copy_blocks.restype = ctypes.c_int
    L.pa_check_device_errors.argtypes = [vp]
    L.pa_check_device_errors.restype = ctypes.c_int
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
    if v.shape != k.shape or v_cache.shape != k_cache.shape:
        raise ValueError("k/v and k_cache/v_cache shapes must match")
    nb, bs, nkv, d = k_cache.shape
    if k.shape[1:] != (nkv, d) or slot_mapping.shape[0] != k.shape[0]:
        raise ValueError("k [T, n_kv, d] / slot_mapping [T] do not match the cache")
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
                    workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Causal GQA varlen attention over the paged cache (see pa_paged_attention).

    ``max_q_len`` / ``max_seq_len`` are host-side bounds that size the launch
    without reading device memory.  Returns ``out``.
    """
    L = _load()
    _need(q, "q", torch.bfloat16, 3)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    _need(query_start_loc, "query_start_loc", torch.int32, 1)
    T, nq, d = q.shape
    nb, bs, nkv, d2 = k_cache.shape
    if d2 != d or v_cache.shape != k_cache.shape:
        raise ValueError("q / k_cache / v_cache head_dim or shapes disagree")
    S = seq_lens.shape[0]
    if query_start_loc.shape[0] != S + 1 or block_tables.shape[0] != S:
        raise ValueError("seq_lens [S], query_start_loc [S+1], block_tables [S, maxb] disagree")
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16, 3)
    if out.shape != q.shape:
        raise ValueError("out must have q's shape")
    if workspace is None:
        workspace = alloc_workspace(S, T, nq, nkv, d, max_q_len, max_seq_len, q.device)
    if workspace.dtype != torch.uint8 or not workspace.is_cuda or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA uint8 tensor")
    _check(L.pa_paged_attention(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), nb, bs,
                                nq, nkv, d, block_tables.data_ptr(), block_tables.shape[1],
                                seq_lens.data_ptr(), query_start_loc.data_ptr(), S, T,
                                int(max_q_len), int(max_seq_len), float(scale), out.data_ptr(),
                                workspace.data_ptr(), workspace.numel(), _stream(stream)))
    return out


def copy_blocks(k_cache: torch.Tensor, v_cache: torch.Tensor, src_dst_pairs: torch.Tensor,
                stream=None) -> None:
    """Copy-on-write: block dst <- block src for each (src, dst) row."""
    L = _load()
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need(src_dst_pairs, "src_dst_pairs", torch.int32, 2)
    if src_dst_pairs.shape[1] != 2:
        raise ValueError("src_dst_pairs must be [n, 2]")
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


def check_device_errors(stream=None) -> None:
    """Synchronise the stream and raise if a kernel flagged an error."""
    _check(_load().pa_check_device_errors(_stream(stream)))
