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

from gpu_util import MAX_ABS, REL_L2, attn_errors, run_oracle_step, to_f64

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


def _split_bytes(num_tokens, num_q_heads, head_dim, pieces):
    """Workspace the prefill key pieces take: per (token, q head, piece) an
    fp32 row of head_dim partial outputs and an fp32 (max, sum) pair, each
    array rounded up to 256 bytes."""
    if pieces <= 1:
        return 0
    rows = num_tokens * num_q_heads * pieces
    up = lambda x: -(-x // 256) * 256
    return up(rows * head_dim * 4) + up(rows * 2 * 4)


def _prefill_case(name, nq, nkv, d, seed):
    """One 64-row chunk at cached offset 4032 (seq_len 4096) plus three decode
    requests, unused slots NaN-poisoned."""
    return W.make_batch(name, [300, 4096, 77, 1500], [1, 64, 1, 1], num_q_heads=nq,
                        num_kv_heads=nkv, head_dim=d, block_size=16, num_blocks=600, seed=seed)


@pytest.mark.parametrize("nq,nkv,d", [(8, 2, 64), (32, 8, 128)])
def test_noalloc_prefill_key_pieces_match_oracle(nq, nkv, d):
    """A mixed batch whose chunk's keys split into pieces.  At 8 q / 2 kv
    heads, d 64, every piece the plan wants fits in what the decode scratch
    leaves of the built-in array; at 32 q / 8 kv heads, d 128, it does not and
    the call uses fewer pieces.  Either way: two calls in a row agree with
    the oracle and, bit for bit, with pa_paged_attention given a workspace of
    the array's size (the same plan), and the full-workspace call (all the
    pieces) agrees with the oracle too."""
    L, f = _noalloc_fn()
    cap = L.pa_noalloc_scratch_bytes()
    b = _prefill_case(f"chunk_{nq}_{nkv}_{d}", nq, nkv, d, seed=40 + nq)
    pieces = ops.prefill_splits(b.num_tokens, nq, nkv, d, b.max_q_len, b.max_seq_len)
    assert pieces >= 2, "the case must split keys"
    need = ops.workspace_size(b.num_seqs, b.num_tokens, nq, nkv, d, 1, b.max_seq_len)
    fit = max(n for n in range(1, pieces + 1)
              if _split_bytes(b.num_tokens, nq, d, n) <= cap - need)
    if nq == 8:
        assert fit == pieces
    else:
        assert fit < pieces, "the case must cut the pieces back"
    d_ = W.to_device(b, "cuda")
    ops.reshape_and_cache(d_.k_new, d_.v_new, d_.k_cache, d_.v_cache, d_.slot_mapping)
    _, _, ref = run_oracle_step(b)
    full = ops.paged_attention(d_.q, d_.k_cache, d_.v_cache, d_.block_tables, d_.seq_lens,
                               d_.query_start_loc, b.scale, max_q_len=b.max_q_len,
                               max_seq_len=b.max_seq_len)
    capped_ws = torch.empty(cap, dtype=torch.uint8, device="cuda")
    capped = ops.paged_attention(d_.q, d_.k_cache, d_.v_cache, d_.block_tables, d_.seq_lens,
                                 d_.query_start_loc, b.scale, max_q_len=b.max_q_len,
                                 max_seq_len=b.max_seq_len, workspace=capped_ws)
    outs = []
    for _ in range(2):  # the second call starts from what the first left in the array
        out = torch.full_like(d_.q, float("nan"))
        code = _call_noalloc(f, b, d_, out)
        assert code == 0, L.pa_get_last_error()
        outs.append(out)
    ops.check_device_errors()
    for what, out in (("workspace", full), ("noalloc 1", outs[0]), ("noalloc 2", outs[1])):
        got = to_f64(out)
        assert np.isfinite(got).all(), what
        mx, rel = attn_errors(got, ref)
        assert mx <= MAX_ABS and rel <= REL_L2, (what, mx, rel)
    for out in outs:
        assert torch.equal(out.view(torch.int16), capped.view(torch.int16))


def test_noalloc_empty_call_prepares_the_device():
    """A call with no requests launches nothing and returns PA_OK after
    looking up the built-in array on the current device (the set-up a caller
    makes before capturing a stream)."""
    L, f = _noalloc_fn()
    b = W.tiny_decode()
    d_ = W.to_device(b, "cuda")
    out = torch.empty_like(d_.q)
    nb, bs, nkv, hd = d_.k_cache.shape
    code = f(d_.q.data_ptr(), d_.k_cache.data_ptr(), d_.v_cache.data_ptr(), nb, bs,
             b.num_q_heads, nkv, hd, d_.block_tables.data_ptr(), d_.block_tables.shape[1],
             d_.seq_lens.data_ptr(), d_.query_start_loc.data_ptr(), 0, 0, 0, 0,
             ctypes.c_float(b.scale), out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert code == 0, L.pa_get_last_error()
