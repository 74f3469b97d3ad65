"""The allocation-free attention entry point, called through the C ABI.

pa_paged_attention_noalloc serves callers that cannot allocate device memory
where they run attention (inside a stream capture, plugins whose host owns all
device memory, serving loops that must not allocate): it takes no workspace
and uses an array built into the library.  Its results must match
pa_paged_attention with a caller-provided workspace, call after call, whatever
an earlier call left in the shared array.

This file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

from paged_kv_cache_174_gb300 import ops
from paged_kv_cache_174_gb300 import workloads as W

from gpu_util import MAX_ABS, REL_L2, attn_errors, to_f64

pytestmark = pytest.mark.gpu


def _noalloc_fn():
    L = ops.lib()
    f = L.pa_paged_attention_noalloc
    i32, vp = ctypes.c_int32, ctypes.c_void_p
    f.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, vp, i32, vp, vp, i32, i32, i32, i32,
                  ctypes.c_float, vp, vp]
    f.restype = ctypes.c_int
    L.pa_noalloc_scratch_bytes.restype = ctypes.c_size_t
    return L, f


def _call_noalloc(f, b, d, out):
    nb, bs, nkv, hd = d.k_cache.shape
    return f(d.q.data_ptr(), d.k_cache.data_ptr(), d.v_cache.data_ptr(), nb, bs,
             b.num_q_heads, nkv, hd, d.block_tables.data_ptr(), d.block_tables.shape[1],
             d.seq_lens.data_ptr(), d.query_start_loc.data_ptr(), b.num_seqs, b.num_tokens,
             b.max_q_len, b.max_seq_len, ctypes.c_float(b.scale), out.data_ptr(),
             torch.cuda.current_stream().cuda_stream)


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls():
    L, f = _noalloc_fn()
    assert L.pa_noalloc_scratch_bytes() == 8 << 20
    batches = [W.decode_batch(), W.tiny_decode(), W.decode_batch(num_seqs=17, seed=77)]
    for b in batches:
        d = W.to_device(b, "cuda")
        ops.reshape_and_cache(d.k_new, d.v_new, d.k_cache, d.v_cache, d.slot_mapping)
        ref = ops.paged_attention(d.q, d.k_cache, d.v_cache, d.block_tables, d.seq_lens,
                                  d.query_start_loc, b.scale, max_q_len=b.max_q_len,
                                  max_seq_len=b.max_seq_len)
        outs = []
        for _ in range(2):  # two calls in a row on the same shared scratch
            out = torch.full_like(d.q, float("nan"))
            code = _call_noalloc(f, b, d, out)
            assert code == 0, L.pa_get_last_error()
            outs.append(out)
        ops.check_device_errors()
        for out in outs:
            mx, rel = attn_errors(to_f64(out), to_f64(ref))
            assert mx <= MAX_ABS and rel <= REL_L2, (b.name, mx, rel)
            assert torch.isfinite(out.float()).all()


def test_noalloc_rejects_calls_beyond_the_builtin_scratch():
    L, f = _noalloc_fn()
    # 64 q heads of 128 on every SM need more split-KV scratch than 8 MiB
    b = W.make_batch("big", [64, 64], [1, 1], num_q_heads=64, num_kv_heads=8, head_dim=128,
                     block_size=16, num_blocks=16, seed=3)
    need = ops.workspace_size(b.num_seqs, b.num_tokens, 64, 8, 128, 1, 64)
    assert need > L.pa_noalloc_scratch_bytes()
    d = W.to_device(b, "cuda")
    out = torch.empty_like(d.q)
    code = _call_noalloc(f, b, d, out)
    assert ops.STATUS_NAMES[code] == "PA_ERR_WORKSPACE"
    assert b"built-in array" in L.pa_get_last_error()
