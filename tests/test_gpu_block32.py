"""Attention over a pool of 32-token blocks ("PagedAttention 显存分页与连续批处理
(Continuous Batching)实战", configuration table: block size 16 or 32) against
the fp64 oracle, and against the same cache viewed as 16-token blocks."""
import numpy as np
import pytest
import torch

from paged_kv_cache_174_gb300 import workloads as W

from gpu_util import assert_attn_close, run_gpu_step, run_oracle_step, to_f64

pytestmark = pytest.mark.gpu


def _batch(lens, q_lens, nq=32, nkv=8, d=128, seed=0, extra_blocks=5):
    nb = sum(-(-L // 32) for L in lens) + extra_blocks
    return W.make_batch("block32", lens, q_lens, num_q_heads=nq, num_kv_heads=nkv, head_dim=d,
                        block_size=32, num_blocks=nb, seed=seed)


def as_16_token_blocks(b: W.PagedBatch) -> W.PagedBatch:
    """The same bytes as a pool of 16-token blocks: block x of 32 tokens is
    blocks 2x and 2x + 1; slots keep their numbers."""
    nb = b.k_cache.shape[0]
    t = b.block_tables
    t16 = np.full((t.shape[0], 2 * t.shape[1]), -1, np.int32)
    t16[:, 0::2] = np.where(t >= 0, 2 * t, -1)
    t16[:, 1::2] = np.where(t >= 0, 2 * t + 1, -1)
    b16 = W.PagedBatch(**{**b.__dict__})
    b16.k_cache = b.k_cache.reshape(2 * nb, 16, *b.k_cache.shape[2:])
    b16.v_cache = b.v_cache.reshape(2 * nb, 16, *b.v_cache.shape[2:])
    b16.block_tables = t16
    b16.block_size = 16
    return b16


@pytest.mark.parametrize("lens,q_lens,nq,nkv,d", [
    ([1, 2, 16, 17, 31, 32, 33, 63, 64, 65], [1] * 10, 32, 8, 128),  # block and page edges
    ([5000, 3, 900], [1, 1, 1], 16, 8, 128),
    ([257, 1000], [1, 1], 8, 2, 64),
    ([300], [77], 32, 8, 128),                    # prefill chunk at an offset
    ([1000, 50, 700], [512, 1, 40], 32, 8, 128),  # prefill + decode
    ([333, 41], [150, 41], 8, 2, 64),
    ([4096], [64], 32, 8, 128),                   # prefill keys in pieces
])
def test_block32_against_oracle(lens, q_lens, nq, nkv, d):
    b = _batch(lens, q_lens, nq, nkv, d, seed=sum(lens) % 89)
    dev, out = run_gpu_step(b)
    kc, vc, ref = run_oracle_step(b)
    assert np.array_equal(W.bits_of(dev.k_cache), kc), "scatter not bit-exact"
    assert_attn_close(to_f64(out), ref, f"block 32 lens={lens[:4]} q_lens={q_lens[:4]}")


@pytest.mark.parametrize("lens,q_lens", [
    (list(range(1, 600, 9)), None),
    ([2000, 700, 129], [300, 1, 129]),
])
def test_block32_equals_the_16_token_view_bit_for_bit(lens, q_lens):
    """The kernels walk 16-token pages either way, so the two layouts of the
    same bytes give identical output bits."""
    q_lens = [1] * len(lens) if q_lens is None else q_lens
    b = _batch(lens, q_lens, seed=4)
    _, out32 = run_gpu_step(b)
    _, out16 = run_gpu_step(as_16_token_blocks(b))
    assert torch.equal(out32.view(torch.int16), out16.view(torch.int16))


def test_mixed_step_block32():
    b = W.mixed_step(block_size=32)
    _, out = run_gpu_step(b)
    _, _, ref = run_oracle_step(b)
    assert_attn_close(to_f64(out), ref, "mixed step, 32-token blocks")
