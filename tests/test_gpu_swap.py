"""Block swap-out / swap-in through the C ABI against the oracle: bit-exact
block copies to pinned host memory and back, on a side stream while
attention runs on another, and a preempted request swapped back in at other
physical blocks giving bit-identical attention output."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_174_gb300 import ops
from paged_kv_cache_174_gb300 import workloads as W

from gpu_util import assert_attn_close, run_oracle_step, to_f64

pytestmark = pytest.mark.gpu


def _random_cache(rng, nb, nkv, d, bs=16):
    return (rng.integers(0, 65536, size=(nb, bs, nkv, d), dtype=np.uint16),
            rng.integers(0, 65536, size=(nb, bs, nkv, d), dtype=np.uint16))


def _host(n, bs, nkv, d):
    return (torch.empty(n, bs, nkv, d, dtype=torch.bfloat16).pin_memory(),
            torch.empty(n, bs, nkv, d, dtype=torch.bfloat16).pin_memory())


@pytest.mark.parametrize("nkv,d,nb,n,bs", [(2, 64, 16, 1, 16), (8, 128, 600, 37, 16),
                                           (8, 128, 4096, 512, 16), (8, 128, 300, 45, 32)])
def test_swap_out_then_in_bit_exact(nkv, d, nb, n, bs):
    rng = np.random.default_rng(nb + n)
    kc, vc = _random_cache(rng, nb, nkv, d, bs)
    ids = rng.choice(nb, size=n, replace=False).astype(np.int32)
    dk, dv = W.bf16_tensor(kc, "cuda"), W.bf16_tensor(vc, "cuda")
    hk, hv = _host(n, bs, nkv, d)
    staging = ops.swap_out(dk, dv, W.int32_tensor(ids, "cuda"), hk, hv)
    ops.check_device_errors()
    ok, ov = oracle.swap_out(kc, vc, ids)
    assert np.array_equal(W.bits_of(hk), ok) and np.array_equal(W.bits_of(hv), ov)
    # back in at other ids (a permutation of the pool), reusing the staging buffer
    dst = rng.permutation(nb)[:n].astype(np.int32)
    ops.swap_in(dk, dv, W.int32_tensor(dst, "cuda"), hk, hv, staging=staging)
    ops.check_device_errors()
    oracle.swap_in(kc, vc, dst, ok, ov)
    assert np.array_equal(W.bits_of(dk), kc) and np.array_equal(W.bits_of(dv), vc)


def test_swap_out_bad_id_flagged():
    kc = torch.zeros(4, 16, 2, 64, dtype=torch.bfloat16, device="cuda")
    hk, hv = _host(2, 16, 2, 64)
    ops.swap_out(kc, kc.clone(), torch.tensor([1, 4], dtype=torch.int32, device="cuda"), hk, hv)
    with pytest.raises(ops.PagedAttnError) as ei:
        ops.check_device_errors()
    assert ei.value.code == 4


def test_swap_on_side_stream_while_attention_runs():
    """Swap-out of blocks no request of the step reads, on its own stream,
    overlapping the step's attention on the current stream."""
    b = W.decode_batch(num_seqs=16, seed=31)
    used = set(int(x) for x in b.block_tables.reshape(-1) if x >= 0)
    free_ids = np.array([i for i in range(b.num_blocks) if i not in used][:256], np.int32)
    d = W.to_device(b, "cuda")
    ops.reshape_and_cache(d.k_new, d.v_new, d.k_cache, d.v_cache, d.slot_mapping)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    hk, hv = _host(len(free_ids), 16, b.num_kv_heads, b.head_dim)
    ids_dev = W.int32_tensor(free_ids, "cuda")
    out = torch.empty_like(d.q)
    with torch.cuda.stream(side):
        ops.swap_out(d.k_cache, d.v_cache, ids_dev, hk, hv, stream=side.cuda_stream)
    ops.paged_attention(d.q, d.k_cache, d.v_cache, d.block_tables, d.seq_lens,
                        d.query_start_loc, b.scale, max_q_len=b.max_q_len,
                        max_seq_len=b.max_seq_len, out=out)
    side.synchronize()
    torch.cuda.synchronize()
    ops.check_device_errors()
    kc, vc, ref = run_oracle_step(b)
    ok, ov = oracle.swap_out(kc, vc, free_ids)
    assert np.array_equal(W.bits_of(hk), ok) and np.array_equal(W.bits_of(hv), ov)
    assert_attn_close(to_f64(out), ref, "attention next to a swap")


def test_preempted_request_swapped_back_gives_identical_bits():
    """Swap a request's blocks out, give them to other requests (overwritten),
    swap it back into different physical blocks with a rewritten Block Table:
    attention output is bit-identical (it depends only on logical positions)."""
    b = W.make_batch("swap", [700, 300], [1, 40], num_q_heads=32, num_kv_heads=8,
                     head_dim=128, block_size=16, num_blocks=120, seed=41)
    d = W.to_device(b, "cuda")
    ops.reshape_and_cache(d.k_new, d.v_new, d.k_cache, d.v_cache, d.slot_mapping)
    kw = dict(max_q_len=b.max_q_len, max_seq_len=b.max_seq_len)
    out1 = torch.empty_like(d.q)
    ops.paged_attention(d.q, d.k_cache, d.v_cache, d.block_tables, d.seq_lens,
                        d.query_start_loc, b.scale, out=out1, **kw)
    nblk = -(-700 // 16)
    table0 = b.block_tables[0, :nblk].copy()
    hk, hv = _host(nblk, 16, 8, 128)
    ops.swap_out(d.k_cache, d.v_cache, W.int32_tensor(table0, "cuda"), hk, hv)
    torch.cuda.synchronize()
    # the freed blocks are reused by someone else
    d.k_cache[torch.from_numpy(table0.astype(np.int64)).cuda()] = 0
    d.v_cache[torch.from_numpy(table0.astype(np.int64)).cuda()] = 0
    # readmitted into other free blocks
    used = set(int(x) for x in b.block_tables.reshape(-1) if x >= 0)
    free = np.array([i for i in range(b.num_blocks) if i not in used], np.int32)
    new_ids = free[:nblk]
    assert len(new_ids) == nblk
    ops.swap_in(d.k_cache, d.v_cache, W.int32_tensor(new_ids, "cuda"), hk, hv)
    bt = b.block_tables.copy()
    bt[0, :nblk] = new_ids
    out2 = torch.empty_like(d.q)
    ops.paged_attention(d.q, d.k_cache, d.v_cache, W.int32_tensor(bt, "cuda"), d.seq_lens,
                        d.query_start_loc, b.scale, out=out2, **kw)
    ops.check_device_errors()
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
