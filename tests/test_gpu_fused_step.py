"""pa_paged_attention_step: one serving step's slot scatter and attention with
no scatter kernel, for any mix of decode and chunked-prefill rows.  Outputs
and the cache afterwards must be bit-identical to the separate calls
(pa_reshape_and_cache, then pa_paged_attention) and agree with the fp64
oracle; unused slots are NaN-poisoned, so reading a new position from the
cache before its row is stored would show."""
import numpy as np
import pytest
import torch

from paged_kv_cache_174_gb300 import ops
from paged_kv_cache_174_gb300 import workloads as W

from gpu_util import assert_attn_close, run_gpu_step, run_oracle_step, to_f64

pytestmark = pytest.mark.gpu


def _fused(b):
    d = W.to_device(b, "cuda")
    out = torch.full_like(d.q, float("nan"))
    ops.attention_step(d.q, d.k_new, d.v_new, d.k_cache, d.v_cache, d.block_tables, d.seq_lens,
                       d.query_start_loc, d.slot_mapping, b.scale, max_q_len=b.max_q_len,
                       max_seq_len=b.max_seq_len, out=out)
    ops.check_device_errors()
    return d, out


def _batch(lens, q_lens, nq=32, nkv=8, d=128, bs=16, seed=0):
    nb = sum(-(-L // bs) for L in lens) + 7
    return W.make_batch("fused", lens, q_lens, num_q_heads=nq, num_kv_heads=nkv, head_dim=d,
                        block_size=bs, num_blocks=nb, seed=seed)


CASES = [
    ([1000, 50, 700], [300, 1, 40], 32, 8, 128, 16),    # chunk starting mid-page (700 % 16 = 12)
    ([20, 333], [3, 1], 32, 8, 128, 16),                # a chunk inside one page
    ([300, 97], [300, 1], 32, 8, 128, 16),              # fresh prompt (no cached rows)
    ([4096], [64], 32, 8, 128, 16),                     # keys in pieces: only piece 0 stores
    ([513, 77, 1800], [513, 1, 129], 8, 8, 128, 16),    # group 1
    ([600, 2000], [200, 1], 64, 8, 128, 16),            # group 8
    ([333, 41, 900], [150, 41, 37], 8, 2, 64, 16),      # head_dim 64
    ([1000, 700, 64], [300, 1, 1], 32, 8, 128, 32),     # 32-token blocks
    ([2300, 1500, 400, 90], [512, 257, 1, 1], 16, 8, 128, 16),  # group 2, two chunks
]


@pytest.mark.parametrize("lens,q_lens,nq,nkv,d,bs", CASES)
def test_fused_step_equals_separate_calls_bit_for_bit(lens, q_lens, nq, nkv, d, bs):
    b = _batch(lens, q_lens, nq, nkv, d, bs, seed=sum(lens) % 89)
    dsep, out_sep = run_gpu_step(b)
    dfus, out_fus = _fused(b)
    assert torch.equal(out_fus.view(torch.int16), out_sep.view(torch.int16))
    assert torch.equal(dfus.k_cache.view(torch.int16), dsep.k_cache.view(torch.int16))
    assert torch.equal(dfus.v_cache.view(torch.int16), dsep.v_cache.view(torch.int16))
    kc, vc, ref = run_oracle_step(b)
    assert np.array_equal(W.bits_of(dfus.k_cache), kc), "fused scatter not bit-exact"
    assert np.array_equal(W.bits_of(dfus.v_cache), vc), "fused scatter not bit-exact"
    assert_attn_close(to_f64(out_fus), ref, f"fused step lens={lens} q_lens={q_lens}")


def test_fused_mixed_step_workload():
    b = W.mixed_step()
    dsep, out_sep = run_gpu_step(b)
    dfus, out_fus = _fused(b)
    assert torch.equal(out_fus.view(torch.int16), out_sep.view(torch.int16))
    assert torch.equal(dfus.k_cache.view(torch.int16), dsep.k_cache.view(torch.int16))
    assert torch.equal(dfus.v_cache.view(torch.int16), dsep.v_cache.view(torch.int16))
    _, _, ref = run_oracle_step(b)
    assert_attn_close(to_f64(out_fus), ref, "fused mixed step")


def test_fused_step_flags_a_prefill_slot_off_its_position():
    """A chunk token whose slot is not its position's slot is not stored and
    flags a bounds error; the other rows are stored."""
    b = _batch([700, 60], [100, 1], seed=3)
    bad = int(b.query_start_loc[0]) + 5
    good_slot = int(b.slot_mapping[bad])
    b.slot_mapping = b.slot_mapping.copy()
    b.slot_mapping[bad] = int(b.slot_mapping[bad + 1])  # another row's slot
    d = W.to_device(b, "cuda")
    ops.attention_step(d.q, d.k_new, d.v_new, d.k_cache, d.v_cache, d.block_tables, d.seq_lens,
                       d.query_start_loc, d.slot_mapping, b.scale, max_q_len=b.max_q_len,
                       max_seq_len=b.max_seq_len)
    with pytest.raises(ops.PagedAttnError) as ei:
        ops.check_device_errors()
    assert ei.value.code == 4
    kflat = W.bits_of(d.k_cache).reshape(-1, b.num_kv_heads, b.head_dim)
    assert np.all(kflat[good_slot] == W.BF16_NAN), "a flagged row was stored"
    nxt = int(b.slot_mapping[bad + 1])
    assert np.array_equal(kflat[nxt], b.k_new[bad + 1]), "the row's own token was not stored"
