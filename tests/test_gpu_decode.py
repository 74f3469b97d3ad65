"""Split-KV decode attention on the GPU against the fp64 oracle, on the named
decode workloads and on edge cases, plus the invariants the method fixes."""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_174_gb300 import ops
from paged_kv_cache_174_gb300 import workloads as W

from gpu_util import assert_attn_close, run_gpu_step, run_oracle_step, to_f64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["tiny_decode", "decode_batch", "long_decode"])
def test_named_decode_workloads(name):
    b = W.by_name(name)
    d, out = run_gpu_step(b)
    kc, vc, ref = run_oracle_step(b)
    assert np.array_equal(W.bits_of(d.k_cache), kc), "scatter not bit-exact"
    assert np.array_equal(W.bits_of(d.v_cache), vc), "scatter not bit-exact"
    assert_attn_close(to_f64(out), ref, name)


def _decode(lens, nq=32, nkv=8, d=128, seed=0, nb=None, q_lens=None, poison=True):
    q_lens = [1] * len(lens) if q_lens is None else q_lens
    nb = nb or sum(-(-L // 16) for L in lens) + 7
    return W.make_batch("edge", lens, q_lens, num_q_heads=nq, num_kv_heads=nkv, head_dim=d,
                        block_size=16, num_blocks=nb, seed=seed, poison=poison)


@pytest.mark.parametrize("lens,nq,nkv,d", [
    ([1], 32, 8, 128),                        # single key
    ([1, 2, 15, 16, 17, 31, 33], 32, 8, 128),  # ragged page tails
    (list(range(1, 700, 7)), 8, 8, 128),       # 100 requests, group 1
    ([5000, 3, 900], 16, 8, 128),              # group 2
    ([4096, 4095, 1], 64, 8, 128),             # group 8 (tensor-core warps)
    ([300, 77, 1], 32, 4, 64),                 # group 8, d 64
    ([130, 7, 64], 8, 1, 128),                 # group 8, one kv head
    ([257, 1000], 8, 2, 64),                   # 2 kv heads, d 64
    ([130, 7, 64], 4, 1, 128),                 # multi-query
    ([64, 3000], 16, 4, 64),
    ([20] * 600, 32, 8, 128),                  # more requests than threads of a CTA
])
def test_decode_edge_shapes(lens, nq, nkv, d):
    b = _decode(lens, nq, nkv, d, seed=len(lens))
    _, out = run_gpu_step(b)
    _, _, ref = run_oracle_step(b)
    assert_attn_close(to_f64(out), ref, f"lens={lens[:5]} nq={nq} nkv={nkv} d={d}")


def test_length_one_returns_v_bit_exact():
    b = _decode([1, 1, 1, 1], nq=32, nkv=8, d=128, seed=3)
    _, out = run_gpu_step(b)
    got = W.bits_of(out)  # [T, nq, d]
    for h in range(32):
        assert np.array_equal(got[:, h], b.v_new[:, h // 4])


def test_identical_keys_give_mean_of_v():
    b = _decode([40, 77], nq=8, nkv=2, d=64, seed=4)
    key = W.randn_bf16(np.random.default_rng(0), (2, 64))
    for s in range(2):
        L = int(b.seq_lens[s])
        for pos in range(L - 1):
            b.k_cache[b.block_tables[s, pos // 16], pos % 16] = key
    b.k_new[:] = key
    _, out = run_gpu_step(b)
    kc, vc, ref = run_oracle_step(b)
    got = to_f64(out)
    assert_attn_close(got, ref, "identical keys")


def test_physical_permutation_gives_identical_bits():
    b = _decode([300, 17, 1025, 64], seed=5, nb=200)
    _, out1 = run_gpu_step(b)
    rng = np.random.default_rng(9)
    pi = rng.permutation(b.num_blocks).astype(np.int32)
    b2 = W.PagedBatch(**{**b.__dict__})
    b2.k_cache = np.empty_like(b.k_cache)
    b2.v_cache = np.empty_like(b.v_cache)
    b2.k_cache[pi] = b.k_cache
    b2.v_cache[pi] = b.v_cache
    b2.block_tables = np.where(b.block_tables >= 0, pi[np.maximum(b.block_tables, 0)],
                               -1).astype(np.int32)
    b2.slot_mapping = (pi[b.slot_mapping // 16] * 16 + b.slot_mapping % 16).astype(np.int32)
    _, out2 = run_gpu_step(b2)
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))


def test_same_request_in_different_batches_agrees():
    """Split positions depend on the batch; results agree within tolerance
    (split-KV merge invariance)."""
    alone = _decode([3001], seed=6)
    _, out_a = run_gpu_step(alone)
    # the same request (same K/V/q bits) placed among others
    many = _decode([3001] + [1500] * 40, seed=6)
    _, _, ref = run_oracle_step(alone)
    _, out_m = run_gpu_step(many)
    ga = to_f64(out_a)
    assert_attn_close(ga, ref, "alone")
    # request 0 of `many` has the same bits only if drawn first with the same
    # seed: compare it against its own oracle instead
    _, _, ref_m = run_oracle_step(many)
    assert_attn_close(to_f64(out_m), ref_m, "in a batch")


def test_zero_length_queries_and_empty_batch():
    b = _decode([50, 20, 70], q_lens=[1, 0, 1], seed=8)
    d, out = run_gpu_step(b)
    _, _, ref = run_oracle_step(b)
    assert_attn_close(to_f64(out), ref, "q_len 0 request")
    # no tokens at all
    e = torch.empty(0, 32, 128, dtype=torch.bfloat16, device="cuda")
    ops.paged_attention(e, d.k_cache, d.v_cache, d.block_tables, d.seq_lens,
                        torch.zeros(4, dtype=torch.int32, device="cuda"), 0.1, max_q_len=0,
                        max_seq_len=70, out=e)
    ops.check_device_errors()


def test_invalid_block_id_is_flagged():
    b = _decode([40, 40], seed=10)
    b.block_tables[1, 1] = b.num_blocks + 5
    d = W.to_device(b, "cuda")
    ops.paged_attention(d.q, d.k_cache, d.v_cache, d.block_tables, d.seq_lens,
                        d.query_start_loc, b.scale, max_q_len=1, max_seq_len=40)
    with pytest.raises(ops.PagedAttnError) as ei:
        ops.check_device_errors()
    assert ei.value.code == 4


def test_seq_len_beyond_table_is_flagged():
    b = _decode([40, 40], seed=11)
    d = W.to_device(b, "cuda")
    d.seq_lens[1] = 16 * b.block_tables.shape[1] + 1  # one past what the table can hold
    ops.paged_attention(d.q, d.k_cache, d.v_cache, d.block_tables, d.seq_lens,
                        d.query_start_loc, b.scale, max_q_len=1,
                        max_seq_len=16 * b.block_tables.shape[1])
    with pytest.raises(ops.PagedAttnError) as ei:
        ops.check_device_errors()
    assert ei.value.code == 4


def test_workspace_too_small_is_rejected():
    b = _decode([40], seed=12)
    d = W.to_device(b, "cuda")
    ws = torch.empty(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(ops.PagedAttnError) as ei:
        ops.paged_attention(d.q, d.k_cache, d.v_cache, d.block_tables, d.seq_lens,
                            d.query_start_loc, b.scale, max_q_len=1, max_seq_len=40,
                            workspace=ws)
    assert ei.value.code == 6


def test_repeated_calls_are_deterministic():
    b = W.decode_batch()
    d, out = run_gpu_step(b)
    outs = []
    for _ in range(3):
        o = ops.paged_attention(d.q, d.k_cache, d.v_cache, d.block_tables, d.seq_lens,
                                d.query_start_loc, b.scale, max_q_len=1,
                                max_seq_len=b.max_seq_len)
        outs.append(o)
    torch.cuda.synchronize()
    for o in outs:
        assert torch.equal(o.view(torch.int16), out.view(torch.int16))


@pytest.mark.parametrize("lens", [[4096], [32768], [40000, 16], [300, 200, 100]])
def test_one_long_request_over_every_cta(lens):
    """A request longer than the grid's pages per CTA is cut into a piece per
    CTA (up to all of them) and merged; few pages leave CTAs without any."""
    b = _decode(lens, seed=len(lens) + lens[0] % 7, nb=sum(-(-L // 16) for L in lens) + 3)
    _, out = run_gpu_step(b)
    if sum(lens) > 20000:
        rng = np.random.default_rng(1)
        samples = np.array([(s, 0, int(h)) for s in range(len(lens))
                            for h in rng.choice(32, size=6, replace=False)], np.int32)
        kc, vc, _ = run_oracle_step(b, attention=False)
        ref = oracle.paged_attention_rows(b.q, kc, vc, b.block_tables, b.seq_lens,
                                          b.query_start_loc, b.scale, samples)
        got = to_f64(out)[b.query_start_loc[samples[:, 0]], samples[:, 2]]
        assert_attn_close(got, ref, f"lens={lens} sampled heads")
    else:
        _, _, ref = run_oracle_step(b)
        assert_attn_close(to_f64(out), ref, f"lens={lens}")


@pytest.mark.parametrize("lens,nq,nkv,d,bs", [
    ([1, 2, 15, 16, 17, 33, 300], 32, 8, 128, 16),   # first row of a page, page edges
    (None, 32, 8, 128, 16),                          # the decode batch
    ([257, 1000, 40], 8, 2, 64, 16),
    ([31, 32, 33, 500], 32, 8, 128, 32),              # 32-token blocks
    ([1, 2, 15, 16, 17, 33, 300], 64, 8, 128, 16),   # group 8 (tensor-core warps)
    ([257, 1000, 40], 16, 2, 64, 32),                # group 8, d 64, 32-token blocks
])
def test_fused_decode_step_equals_scatter_then_attention(lens, nq, nkv, d, bs):
    """pa_decode_step (the new rows taken into the page in shared memory and
    stored from there) gives the same output bits and the same cache bits as
    pa_reshape_and_cache followed by pa_paged_attention."""
    if lens is None:
        b = W.decode_batch(seed=21)
    else:
        nb = sum(-(-L // bs) for L in lens) + 5
        b = W.make_batch("fused", lens, [1] * len(lens), num_q_heads=nq, num_kv_heads=nkv,
                         head_dim=d, block_size=bs, num_blocks=nb, seed=len(lens))
    d1, out1 = run_gpu_step(b)
    d2 = W.to_device(b)
    out2 = torch.full_like(d2.q, float("nan"))
    ops.decode_step(d2.q, d2.k_new, d2.v_new, d2.k_cache, d2.v_cache, d2.block_tables,
                    d2.seq_lens, d2.query_start_loc, d2.slot_mapping, b.scale,
                    max_seq_len=b.max_seq_len, out=out2)
    ops.check_device_errors()
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(d1.k_cache.view(torch.int16), d2.k_cache.view(torch.int16))
    assert torch.equal(d1.v_cache.view(torch.int16), d2.v_cache.view(torch.int16))
    kc, vc, ref = run_oracle_step(b)
    assert np.array_equal(W.bits_of(d2.k_cache), kc) and np.array_equal(W.bits_of(d2.v_cache), vc)
    assert_attn_close(to_f64(out2), ref, "fused decode step")


def test_fused_decode_step_slot_rules():
    """A negative slot leaves the row unwritten and reads the cache's row (as
    a separate scatter that skips it would); a slot that is not the last
    position's slot is flagged."""
    b = _decode([40, 70], nq=8, nkv=2, d=64, seed=3)
    b.slot_mapping = b.slot_mapping.copy()
    b.slot_mapping[1] = -1
    d1, out1 = run_gpu_step(b)
    d2 = W.to_device(b)
    out2 = ops.decode_step(d2.q, d2.k_new, d2.v_new, d2.k_cache, d2.v_cache, d2.block_tables,
                           d2.seq_lens, d2.query_start_loc, d2.slot_mapping, b.scale,
                           max_seq_len=b.max_seq_len)
    ops.check_device_errors()
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(d1.k_cache.view(torch.int16), d2.k_cache.view(torch.int16))
    bad = b.slot_mapping.copy()
    bad[0] = bad[0] - 1 if bad[0] > 0 else bad[0] + 1
    d3 = W.to_device(b)
    ops.decode_step(d3.q, d3.k_new, d3.v_new, d3.k_cache, d3.v_cache, d3.block_tables,
                    d3.seq_lens, d3.query_start_loc, W.int32_tensor(bad, "cuda"), b.scale,
                    max_seq_len=b.max_seq_len)
    with pytest.raises(ops.PagedAttnError) as ei:
        ops.check_device_errors()
    assert ei.value.code == 4
