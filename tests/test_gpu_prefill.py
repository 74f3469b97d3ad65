"""Chunked-prefill attention (q_len >= 2) on the tcgen05 path against the
fp64 oracle: the mixed chunked-prefill step and edge cases."""
import numpy as np
import pytest
import torch

from paged_kv_cache_174_gb300 import ops
from paged_kv_cache_174_gb300 import workloads as W

from gpu_util import assert_attn_close, run_gpu_step, run_oracle_step, to_f64

pytestmark = pytest.mark.gpu


def test_mixed_step_workload():
    b = W.mixed_step()
    d, out = run_gpu_step(b)
    kc, vc, ref = run_oracle_step(b)
    assert np.array_equal(W.bits_of(d.k_cache), kc), "scatter not bit-exact"
    assert np.array_equal(W.bits_of(d.v_cache), vc), "scatter not bit-exact"
    got = to_f64(out)
    assert_attn_close(got, ref, "mixed step (all rows)")
    chunk = slice(b.query_start_loc[-2], b.query_start_loc[-1])
    assert_attn_close(got[chunk], ref[chunk], "mixed step (prefill chunk rows)")


def _batch(lens, q_lens, nq=32, nkv=8, d=128, seed=0, extra_blocks=9):
    nb = sum(-(-L // 16) for L in lens) + extra_blocks
    return W.make_batch("prefill-edge", lens, q_lens, num_q_heads=nq, num_kv_heads=nkv,
                        head_dim=d, block_size=16, num_blocks=nb, seed=seed)


@pytest.mark.parametrize("lens,q_lens,nq,nkv,d", [
    ([2], [2], 32, 8, 128),                       # smallest prefill
    ([37], [37], 32, 8, 128),                     # fresh prompt, one ragged tile
    ([300], [77], 32, 8, 128),                    # chunk at an offset, ragged tiles
    ([128, 129, 255, 256, 257], [128, 2, 100, 33, 257], 32, 8, 128),  # tile edges
    ([1000, 50, 700], [512, 1, 40], 32, 8, 128),  # prefill + decode mixed
    ([513], [513], 8, 8, 128),                    # group 1: 128 tokens per tile
    ([400, 90], [131, 90], 16, 8, 128),           # group 2
    ([600], [200], 64, 8, 128),                   # group 8: 16 tokens per tile
    ([333, 41], [150, 41], 8, 2, 64),             # head_dim 64
    ([250], [250], 4, 1, 64),                     # multi-query, head_dim 64
    ([4096], [64], 32, 8, 128),                   # two query tiles: keys in 4 pieces + merge
    ([4096, 100], [64, 100], 32, 8, 128),         # short request: pieces with no key tile
    ([1100], [1024], 8, 8, 128),                  # rows that see no key of a piece
    ([3000], [40], 8, 2, 64),                     # head_dim 64, keys in pieces
    ([96], [32], 32, 8, 128),                     # one full tile, the second tile empty
    ([600], [65], 32, 8, 128),                    # two row blocks, the last of 1 row
    ([777], [230], 16, 2, 64),                    # group 8, head_dim 64
    ([2000, 1500], [300, 700], 16, 8, 128),       # group 2: 128-token row blocks
])
def test_prefill_edge_shapes(lens, q_lens, nq, nkv, d):
    b = _batch(lens, q_lens, nq, nkv, d, seed=sum(lens) % 97)
    _, out = run_gpu_step(b)
    _, _, ref = run_oracle_step(b)
    assert_attn_close(to_f64(out), ref, f"lens={lens} q_lens={q_lens} nq={nq} nkv={nkv} d={d}")


def test_many_prefill_requests():
    rng = np.random.default_rng(5)
    lens = list(rng.integers(2, 600, size=40))
    q_lens = [int(rng.integers(2, L + 1)) for L in lens]
    b = _batch(lens, q_lens, seed=11)
    _, out = run_gpu_step(b)
    _, _, ref = run_oracle_step(b)
    assert_attn_close(to_f64(out), ref, "40 prefill requests")


def test_more_prefill_requests_than_the_listed_maximum():
    """Over 1024 requests with prefill rows: the kernel walks the sequences
    instead of its per-CTA request list; decode rows interleaved."""
    rng = np.random.default_rng(9)
    lens, q_lens = [], []
    for i in range(1100):
        L = int(rng.integers(48, 97))
        lens.append(L)
        q_lens.append(1 if i % 7 == 3 else int(rng.integers(2, 7)))
    b = _batch(lens, q_lens, nq=4, nkv=2, d=64, seed=12)
    _, out = run_gpu_step(b)
    _, _, ref = run_oracle_step(b)
    assert_attn_close(to_f64(out), ref, "1100 requests")


def test_prefill_physical_permutation_gives_identical_bits():
    b = _batch([700, 260], [300, 260], seed=6, extra_blocks=40)
    _, out1 = run_gpu_step(b)
    pi = np.random.default_rng(3).permutation(b.num_blocks).astype(np.int32)
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


def test_prefill_chunk_equals_rows_of_full_prompt():
    """Chunked prefill: the last 64 rows computed as a chunk at offset 256
    equal those rows of the whole 320-token prompt computed at once."""
    full = _batch([320], [320], seed=8)
    _, out_full = run_gpu_step(full)
    chunk = W.PagedBatch(**{**full.__dict__})
    chunk.q = full.q[256:]
    chunk.k_new = full.k_new[256:]
    chunk.v_new = full.v_new[256:]
    chunk.slot_mapping = full.slot_mapping[256:]
    chunk.query_start_loc = np.array([0, 64], np.int32)
    # the cache already holds positions 0..255 (written by the full step's scatter)
    kc, vc, _ = run_oracle_step(full, attention=False)
    chunk.k_cache, chunk.v_cache = kc, vc
    _, out_chunk = run_gpu_step(chunk)
    a = to_f64(out_full)[256:]
    c = to_f64(out_chunk)
    assert_attn_close(c, a, "chunk vs full prompt")


@pytest.mark.parametrize("lens,q_lens,nq,nkv,d,pieces", [
    ([4096], [64], 32, 8, 128, 4),
    ([4096, 100], [64, 100], 32, 8, 128, 3),
    ([1100], [1024], 8, 8, 128, 2),
    ([3000], [40], 8, 2, 64, 4),
    ([300], [77], 32, 8, 128, 1),
    ([4096], [512], 32, 8, 128, 1),               # the mixed step's chunk alone
])
def test_prefill_key_split_plan(lens, q_lens, nq, nkv, d, pieces):
    """The cases above that are meant to split the keys really do (on a
    152-SM GB300; other SM counts may choose differently)."""
    if torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("plan thresholds depend on the SM count")
    assert ops.prefill_splits(sum(q_lens), nq, nkv, d, max(q_lens), max(lens)) == pieces


def test_one_workspace_for_a_large_step_serves_a_short_one():
    """pa_workspace_size bounds every call with smaller sizes: a buffer sized
    for a 2048-token step serves a 64-token chunk whose keys split into
    pieces (fewer tokens, more pieces); a buffer with only the decode scratch
    runs the same call without pieces.  Both agree with the oracle."""
    b = _batch([4096], [64], seed=13)
    _, _, ref = run_oracle_step(b)
    big = ops.alloc_workspace(8, 2048, 32, 8, 128, 512, 4096, "cuda")
    small = ops.alloc_workspace(1, 64, 32, 8, 128, 1, 4096, "cuda")  # decode scratch only
    assert ops.prefill_splits(64, 32, 8, 128, 64, 4096) > 1
    for ws in (big, small):
        d = W.to_device(b, "cuda")
        ops.reshape_and_cache(d.k_new, d.v_new, d.k_cache, d.v_cache, d.slot_mapping)
        out = torch.full_like(d.q, float("nan"))
        ops.paged_attention(d.q, d.k_cache, d.v_cache, d.block_tables, d.seq_lens,
                            d.query_start_loc, b.scale, max_q_len=64, max_seq_len=4096, out=out,
                            workspace=ws)
        ops.check_device_errors()
        assert_attn_close(to_f64(out), ref, f"workspace of {ws.numel()} bytes")


def test_min_q_len_bound_skips_the_decode_launch_with_identical_bits():
    """pa_paged_attention_qrange with min_q_len >= 2 (no decode rows) gives
    the same bits as the plain call; a request with one row under that
    promise is flagged."""
    b = _batch([700, 300, 90], [64, 300, 2], seed=14)
    _, out1 = run_gpu_step(b)
    d = W.to_device(b, "cuda")
    ops.reshape_and_cache(d.k_new, d.v_new, d.k_cache, d.v_cache, d.slot_mapping)
    out2 = torch.full_like(d.q, float("nan"))
    ops.paged_attention(d.q, d.k_cache, d.v_cache, d.block_tables, d.seq_lens,
                        d.query_start_loc, b.scale, max_q_len=b.max_q_len,
                        max_seq_len=b.max_seq_len, out=out2, min_q_len=2)
    ops.check_device_errors()
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    bad = _batch([50, 40], [4, 1], seed=15)
    d = W.to_device(bad, "cuda")
    with pytest.raises(ops.PagedAttnError) as ei:
        ops.paged_attention(d.q, d.k_cache, d.v_cache, d.block_tables, d.seq_lens,
                            d.query_start_loc, bad.scale, max_q_len=4, max_seq_len=50,
                            min_q_len=2)
        ops.check_device_errors()
    assert ei.value.code == 4
