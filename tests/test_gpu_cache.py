"""Slot scatter and copy-on-write block copy on the GPU, bit-exact against
the oracle (whole-cache comparison)."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_174_gb300 import ops
from paged_kv_cache_174_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _random_cache(rng, nb, nkv, d):
    return W.randn_bf16(rng, (nb, 16, nkv, d)), W.randn_bf16(rng, (nb, 16, nkv, d))


@pytest.mark.parametrize("T,nkv,d,nb", [(1, 2, 64, 4), (37, 8, 128, 64), (640, 8, 128, 2000),
                                        (2048, 8, 128, 4096), (300, 1, 64, 40)])
def test_scatter_bit_exact(T, nkv, d, nb):
    rng = np.random.default_rng(T + nkv)
    kc, vc = _random_cache(rng, nb, nkv, d)
    k = W.randn_bf16(rng, (T, nkv, d))
    v = W.randn_bf16(rng, (T, nkv, d))
    slots = rng.permutation(nb * 16)[:T].astype(np.int32)
    slots[::7] = -1  # padding tokens are skipped
    dk, dv = W.bf16_tensor(kc, "cuda"), W.bf16_tensor(vc, "cuda")
    ops.reshape_and_cache(W.bf16_tensor(k, "cuda"), W.bf16_tensor(v, "cuda"), dk, dv,
                          W.int32_tensor(slots, "cuda"))
    ops.check_device_errors()
    oracle.reshape_and_cache(k, v, kc, vc, slots)
    assert np.array_equal(W.bits_of(dk), kc)
    assert np.array_equal(W.bits_of(dv), vc)


def test_scatter_empty_is_noop():
    kc = torch.zeros(4, 16, 2, 64, dtype=torch.bfloat16, device="cuda")
    e = torch.zeros(0, 2, 64, dtype=torch.bfloat16, device="cuda")
    ops.reshape_and_cache(e, e, kc, kc.clone(), torch.zeros(0, dtype=torch.int32, device="cuda"))
    ops.check_device_errors()
    assert not kc.any()


def test_scatter_out_of_range_slot_is_flagged_and_skipped():
    kc = torch.zeros(4, 16, 2, 64, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    k = torch.ones(2, 2, 64, dtype=torch.bfloat16, device="cuda")
    slots = torch.tensor([3, 64], dtype=torch.int32, device="cuda")  # 64 == 4 * 16: out of range
    ops.reshape_and_cache(k, k, kc, vc, slots)
    with pytest.raises(ops.PagedAttnError) as ei:
        ops.check_device_errors()
    assert ei.value.code == 4
    assert kc.view(-1, 2, 64)[3].eq(1).all() and kc.sum().item() == 128
    ops.check_device_errors()  # the word was cleared


@pytest.mark.parametrize("nkv,d,nb,npairs", [(2, 64, 32, 1), (8, 128, 512, 100),
                                             (8, 128, 4096, 1000)])
def test_copy_blocks_bit_exact(nkv, d, nb, npairs):
    rng = np.random.default_rng(nb + npairs)
    kc, vc = _random_cache(rng, nb, nkv, d)
    perm = rng.permutation(nb)
    src = perm[:npairs]
    dst = perm[npairs:2 * npairs]
    src = np.where(np.arange(npairs) % 3 == 0, src[0], src)  # one source shared by many
    pairs = np.stack([src, dst], 1).astype(np.int32)
    dk, dv = W.bf16_tensor(kc, "cuda"), W.bf16_tensor(vc, "cuda")
    ops.copy_blocks(dk, dv, W.int32_tensor(pairs, "cuda"))
    ops.check_device_errors()
    k0 = kc.copy()
    oracle.copy_blocks(kc, vc, pairs)
    assert np.array_equal(W.bits_of(dk), kc)
    assert np.array_equal(W.bits_of(dv), vc)
    # sources unchanged, destinations equal their source
    for s_, d_ in pairs[:20]:
        assert np.array_equal(kc[d_], k0[s_]) and np.array_equal(kc[s_], k0[s_])


def test_copy_blocks_bad_id_flagged():
    kc = torch.zeros(4, 16, 2, 64, dtype=torch.bfloat16, device="cuda")
    pairs = torch.tensor([[0, 4]], dtype=torch.int32, device="cuda")
    ops.copy_blocks(kc, kc.clone(), pairs)
    with pytest.raises(ops.PagedAttnError) as ei:
        ops.check_device_errors()
    assert ei.value.code == 4
