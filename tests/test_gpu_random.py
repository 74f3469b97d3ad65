"""Seeded random sweep over every supported shape: head_dim {64, 128}, GQA
group {1, 2, 4, 8}, kv heads {1, 2, 4, 8}, block size {16, 32}, with a random
mix of decode rows, prefill chunks and fresh prompts per batch.  Each step
(scatter + attention) is compared with the oracle: the cache bit for bit,
attention within the tolerance.  Decode-only draws also run the fused decode
step and must give the same bits as scatter followed by attention."""
import numpy as np
import pytest
import torch

from paged_kv_cache_174_gb300 import ops
from paged_kv_cache_174_gb300 import workloads as W

from gpu_util import assert_attn_close, run_gpu_step, run_oracle_step, to_f64

pytestmark = pytest.mark.gpu

N_CASES = 32


def _draw(seed: int):
    rng = np.random.default_rng(1000 + seed)
    d = int(rng.choice([64, 128]))
    g = int(rng.choice([1, 2, 4, 8]))
    nkv = int(rng.choice([1, 2, 4, 8]))
    bs = int(rng.choice([16, 32]))
    S = int(rng.integers(1, 13))
    decode_only = seed % 4 == 0
    lens, q_lens = [], []
    for _ in range(S):
        L = int(rng.integers(1, 900))
        kind = rng.random()
        if decode_only or kind < 0.5:
            ql = 1
        elif kind < 0.8:
            ql = int(rng.integers(2, min(L, 160) + 1)) if L >= 2 else 1  # chunk at an offset
        else:
            L = min(L, 300)
            ql = L  # fresh prompt
        lens.append(L)
        q_lens.append(ql)
    nb = sum(-(-L // bs) for L in lens) + int(rng.integers(1, 20))
    b = W.make_batch("random", lens, q_lens, num_q_heads=g * nkv, num_kv_heads=nkv,
                     head_dim=d, block_size=bs, num_blocks=nb, seed=2000 + seed)
    return b, decode_only, (d, g, nkv, bs, lens, q_lens)


@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_step_against_oracle(seed):
    b, decode_only, desc = _draw(seed)
    d1, out = run_gpu_step(b)
    kc, vc, ref = run_oracle_step(b)
    assert np.array_equal(W.bits_of(d1.k_cache), kc), f"scatter not bit-exact: {desc}"
    assert np.array_equal(W.bits_of(d1.v_cache), vc), f"scatter not bit-exact: {desc}"
    assert_attn_close(to_f64(out), ref, f"random step {desc}")
    if decode_only:
        d2 = W.to_device(b)
        out2 = torch.full_like(d2.q, float("nan"))
        ops.decode_step(d2.q, d2.k_new, d2.v_new, d2.k_cache, d2.v_cache, d2.block_tables,
                        d2.seq_lens, d2.query_start_loc, d2.slot_mapping, b.scale,
                        max_seq_len=b.max_seq_len, out=out2)
        ops.check_device_errors()
        assert torch.equal(out.view(torch.int16), out2.view(torch.int16)), desc
        assert torch.equal(d1.k_cache.view(torch.int16), d2.k_cache.view(torch.int16)), desc


@pytest.mark.parametrize("seed", range(16))
def test_random_fp8_against_oracle(seed):
    """The same sweep over the 8-bit cache (the oracle's attention runs on
    code x scale): even seeds decode rows only, odd seeds a mix of decode
    rows, chunks at an offset and fresh prompts; the pool's unwritten slots
    hold NaN codes and scales."""
    from test_gpu_fp8 import fp8_step
    rng = np.random.default_rng(3000 + seed)
    d = int(rng.choice([64, 128]))
    g = int(rng.choice([1, 2, 4, 8]))
    nkv = int(rng.choice([1, 2, 4, 8]))
    bs = int(rng.choice([16, 32]))
    lens = [int(x) for x in rng.integers(1, 1500, size=int(rng.integers(1, 10)))]
    q_lens = [1] * len(lens)
    if seed % 2:
        for i, L in enumerate(lens):
            kind = rng.random()
            if kind < 0.3 or L < 2:
                continue
            q_lens[i] = int(rng.integers(2, min(L, 300) + 1)) if kind < 0.8 else L
    nb = sum(-(-L // bs) for L in lens) + 3
    b = W.make_batch("random-fp8", lens, q_lens, num_q_heads=g * nkv,
                     num_kv_heads=nkv, head_dim=d, block_size=bs, num_blocks=nb,
                     seed=4000 + seed)
    got, ref = fp8_step(b, poison=True)
    assert_attn_close(got, ref, f"random fp8 d={d} g={g} nkv={nkv} bs={bs} lens={lens} "
                                f"q_lens={q_lens}")
