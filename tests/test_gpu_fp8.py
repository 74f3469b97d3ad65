"""The 8-bit (FP8 E4M3) KV cache on the GPU against the oracle: the
quantising scatter bit for bit (codes and scales), decode and chunked-prefill
attention over the 8-bit cache against the oracle's attention over
code * scale, and the block copy of codes and scales."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_174_gb300 import ops
from paged_kv_cache_174_gb300 import workloads as W

from gpu_util import assert_attn_close, to_f64

pytestmark = pytest.mark.gpu


def _context_slots(b):
    """Slots of every cached (context) position of every request, and the
    bf16 rows that live there."""
    slots = []
    for s in range(b.num_seqs):
        ctx = int(b.seq_lens[s]) - int(b.query_start_loc[s + 1] - b.query_start_loc[s])
        for p in range(ctx):
            slots.append(oracle.slot_of(b.block_tables[s], p, b.block_size))
    slots = np.array(slots, np.int32)
    nkv, d = b.k_cache.shape[2:]
    rows_k = b.k_cache.reshape(-1, nkv, d)[slots]
    rows_v = b.v_cache.reshape(-1, nkv, d)[slots]
    return slots, rows_k, rows_v


def fp8_slot_arrays(cache, nkv, d):
    """(codes [slots, n_kv, d], scales [slots, n_kv]) of a device 8-bit cache,
    in slot order, on the host."""
    codes, scales = ops.fp8_cache_views(cache, nkv, d)
    return (codes.cpu().numpy().reshape(-1, nkv, d), scales.cpu().numpy().reshape(-1, nkv))


def fp8_step(b, poison=False):
    """Quantise the batch's context and its new tokens into an 8-bit cache on
    both sides (GPU scatter and oracle scatter, compared bit for bit), then
    run attention (decode and prefill rows) on both.  With poison, every GPU
    slot that is not written holds NaN codes and NaN scales, which no output
    may see.  Returns (gpu out, oracle out)."""
    nb, bs, nkv, d = b.k_cache.shape
    slots, rk, rv = _context_slots(b)
    dk8, dv8 = ops.empty_fp8_cache(nb, bs, nkv, d)
    if poison:
        for t in (dk8, dv8):
            codes, scales = ops.fp8_cache_views(t, nkv, d)
            codes.fill_(0x7F)  # E4M3 NaN
            scales.fill_(float("nan"))
    ok8, ov8, oks, ovs = oracle.fp8_cache(nb, bs, nkv, d, fill_code=0)
    oks[:] = 0
    ovs[:] = 0
    for ks_, vs_, sl in ((rk, rv, slots), (b.k_new, b.v_new, b.slot_mapping)):
        if len(sl) == 0:
            continue
        ops.reshape_and_cache_fp8(W.bf16_tensor(ks_, "cuda"), W.bf16_tensor(vs_, "cuda"), dk8,
                                  dv8, W.int32_tensor(sl, "cuda"))
        oracle.reshape_and_cache_fp8(ks_, vs_, ok8, ov8, oks, ovs, sl)
    ops.check_device_errors()
    written = np.zeros(nb * bs, bool)
    written[slots] = True
    written[b.slot_mapping[b.slot_mapping >= 0]] = True
    dks_, dvs_ = fp8_slot_arrays(dk8, nkv, d), fp8_slot_arrays(dv8, nkv, d)
    for got, ref, what in ((dks_[0], ok8, "K codes"), (dvs_[0], ov8, "V codes"),
                           (dks_[1], oks, "K scales"), (dvs_[1], ovs, "V scales")):
        if got.dtype == np.float32:
            got, ref = got.view(np.uint32), ref.view(np.uint32)
        got = got.reshape(nb * bs, -1)[written]
        assert np.array_equal(got, ref.reshape(nb * bs, -1)[written]), f"{what} differ"
    out = torch.full((b.num_tokens, b.num_q_heads, d), float("nan"), dtype=torch.bfloat16,
                     device="cuda")
    ops.paged_attention_fp8(W.bf16_tensor(b.q, "cuda"), dk8, dv8,
                            W.int32_tensor(b.block_tables, "cuda"),
                            W.int32_tensor(b.seq_lens, "cuda"),
                            W.int32_tensor(b.query_start_loc, "cuda"), b.scale,
                            max_q_len=b.max_q_len, max_seq_len=b.max_seq_len, out=out)
    ops.check_device_errors()
    ref = oracle.paged_attention_fp8(b.q, ok8, ov8, oks, ovs, b.block_tables, b.seq_lens,
                                     b.query_start_loc, b.scale)
    return to_f64(out), ref


def _decode(lens, nq=32, nkv=8, d=128, seed=0, bs=16):
    nb = sum(-(-L // bs) for L in lens) + 5
    return W.make_batch("fp8", lens, [1] * len(lens), num_q_heads=nq, num_kv_heads=nkv,
                        head_dim=d, block_size=bs, num_blocks=nb, seed=seed)


@pytest.mark.parametrize("lens,nq,nkv,d,bs", [
    ([1, 2, 15, 16, 17, 31, 33], 32, 8, 128, 16),  # ragged page tails
    ([5000, 3, 900], 16, 8, 128, 16),              # group 2, split across CTAs
    ([4096, 4095, 1], 64, 8, 128, 16),             # group 8
    ([257, 1000], 8, 2, 64, 16),                   # 2 kv heads, d 64
    ([130, 7, 64], 4, 1, 128, 16),                 # multi-query
    ([300, 47], 32, 8, 128, 32),                   # 32-token blocks
    ([20] * 300, 32, 8, 128, 16),                  # many short requests
])
def test_fp8_decode_edge_shapes(lens, nq, nkv, d, bs):
    got, ref = fp8_step(_decode(lens, nq, nkv, d, seed=len(lens), bs=bs))
    assert_attn_close(got, ref, f"fp8 lens={lens[:4]} nq={nq} nkv={nkv} d={d} bs={bs}")


def test_fp8_decode_batch_workload():
    """The 64-request decode batch (lens U[128, 4096], 32/8 heads, d 128)."""
    got, ref = fp8_step(W.decode_batch())
    assert_attn_close(got, ref, "fp8 decode batch")


@pytest.mark.parametrize("mag", [1e-2, 3e3])
def test_fp8_decode_small_and_large_values(mag):
    """Values far from unit size: the decode kernel multiplies p by each
    token's value scale in f16 (times a power of two), which must neither
    lose small products nor overflow.  Compared after dividing by mag."""
    b = _decode([700, 130, 2000, 1], seed=21)
    for name in ("v_cache", "v_new"):
        a = W.f32_from_bf16(getattr(b, name)) * np.float32(mag)
        setattr(b, name, W.bf16_from_f32(a.astype(np.float32)))
    got, ref = fp8_step(b)
    assert_attn_close(got / mag, ref / mag, f"fp8 values x {mag}")


def test_fp8_quantises_zero_and_large_rows():
    """All-zero rows (scale 1, zero codes) and rows of large bf16 magnitudes
    quantise bit for bit like the oracle."""
    rng = np.random.default_rng(4)
    k = W.randn_bf16(rng, (24, 8, 128))
    v = W.randn_bf16(rng, (24, 8, 128))
    k[3] = 0
    v[5, 2] = 0
    big = (W.f32_from_bf16(k[7]) * np.float32(3e37)).astype(np.float32)
    k[7] = W.bf16_from_f32(big)
    slots = rng.permutation(64)[:24].astype(np.int32)
    dk8, dv8 = ops.empty_fp8_cache(4, 16, 8, 128)
    ok8, ov8, oks, ovs = oracle.fp8_cache(4, 16, 8, 128, fill_code=0)
    oks[:] = 0
    ovs[:] = 0
    ops.reshape_and_cache_fp8(W.bf16_tensor(k, "cuda"), W.bf16_tensor(v, "cuda"), dk8, dv8,
                              W.int32_tensor(slots, "cuda"))
    ops.check_device_errors()
    oracle.reshape_and_cache_fp8(k, v, ok8, ov8, oks, ovs, slots)
    (kc, ks), (vc, vs) = fp8_slot_arrays(dk8, 8, 128), fp8_slot_arrays(dv8, 8, 128)
    assert np.array_equal(kc, ok8.reshape(64, 8, 128))
    assert np.array_equal(vc, ov8.reshape(64, 8, 128))
    assert np.array_equal(ks.view(np.uint32), oks.reshape(64, 8).view(np.uint32))
    assert np.array_equal(vs.view(np.uint32), ovs.reshape(64, 8).view(np.uint32))


def test_fp8_page_format():
    """The page format: a 16-token page holds its codes, then its scales, and
    the slot of row r of page p of block b is b * block_size + 16 p + r."""
    nkv, d, bs = 2, 64, 32
    assert ops.fp8_page_bytes(nkv, d) == 16 * nkv * (d + 4)
    assert int(ops._load().pa_fp8_page_bytes(nkv, d)) == ops.fp8_page_bytes(nkv, d)
    rng = np.random.default_rng(5)
    k = W.randn_bf16(rng, (3, nkv, d))
    slots = np.array([0, 17, 2 * bs + 31], np.int32)  # block 0 page 0 row 0; page 1 row 1; ...
    dk8, dv8 = ops.empty_fp8_cache(3, bs, nkv, d)
    ops.reshape_and_cache_fp8(W.bf16_tensor(k, "cuda"), W.bf16_tensor(k, "cuda"), dk8, dv8,
                              W.int32_tensor(slots, "cuda"))
    ops.check_device_errors()
    ok8, _, oks, _ = oracle.fp8_cache(3, bs, nkv, d, fill_code=0)
    oks[:] = 0
    oracle.reshape_and_cache_fp8(k, k, ok8, ok8.copy(), oks, oks.copy(), slots)
    raw = dk8.cpu().numpy()  # [blocks, pages, bytes]
    cb = 16 * nkv * d
    for t, slot in enumerate(slots):
        blk, p, r = slot // bs, (slot % bs) // 16, slot % 16
        page = raw[blk, p]
        codes = page[(r * nkv) * d:(r * nkv + nkv) * d].reshape(nkv, d)
        scales = page[cb + r * nkv * 4:cb + (r + 1) * nkv * 4].view(np.float32)
        assert np.array_equal(codes, ok8.reshape(-1, nkv, d)[slot])
        assert np.array_equal(scales.view(np.uint32), oks.reshape(-1, nkv)[slot].view(np.uint32))
    # nothing else was written
    mask = np.ones(raw.shape, bool)
    for slot in slots:
        blk, p, r = slot // bs, (slot % bs) // 16, slot % 16
        mask[blk, p, (r * nkv) * d:(r * nkv + nkv) * d] = False
        mask[blk, p, cb + r * nkv * 4:cb + (r + 1) * nkv * 4] = False
    assert not raw[mask].any()


@pytest.mark.parametrize("bs", [16, 32])
def test_fp8_copy_blocks_moves_codes_and_scales(bs):
    rng = np.random.default_rng(8)
    dk8, dv8 = ops.empty_fp8_cache(10, bs, 8, 128)
    for t in (dk8, dv8):
        t.copy_(torch.from_numpy(rng.integers(0, 256, tuple(t.shape), dtype=np.uint8)))
    before = [t.cpu().numpy().copy() for t in (dk8, dv8)]
    pairs = np.array([[1, 4], [-1, -1], [6, 2]], np.int32)
    ops.copy_blocks_fp8(dk8, dv8, W.int32_tensor(pairs, "cuda"), num_kv_heads=8, head_dim=128)
    ops.check_device_errors()
    for dev_t, host in zip((dk8, dv8), before):
        host[4] = host[1]
        host[2] = host[6]
        assert np.array_equal(dev_t.cpu().numpy(), host)


def _mixed(lens, q_lens, nq=32, nkv=8, d=128, seed=0, bs=16):
    nb = sum(-(-L // bs) for L in lens) + 5
    return W.make_batch("fp8", lens, q_lens, num_q_heads=nq, num_kv_heads=nkv, head_dim=d,
                        block_size=bs, num_blocks=nb, seed=seed)


@pytest.mark.parametrize("lens,q_lens,nq,nkv,d,bs", [
    ([2], [2], 32, 8, 128, 16),                    # smallest prefill
    ([37], [37], 32, 8, 128, 16),                  # fresh prompt, one ragged tile
    ([300], [77], 32, 8, 128, 16),                 # chunk at an offset, ragged tiles
    ([1000, 50, 700], [512, 1, 40], 32, 8, 128, 16),  # prefill + decode rows
    ([513], [513], 8, 8, 128, 16),                 # group 1
    ([600], [200], 64, 8, 128, 16),                # group 8
    ([333, 41], [150, 41], 8, 2, 64, 16),          # head_dim 64
    ([250], [250], 4, 1, 64, 16),                  # multi-query, head_dim 64
    ([4096], [64], 32, 8, 128, 16),                # keys in 4 pieces + merge
    ([3000], [40], 8, 2, 64, 16),                  # head_dim 64, keys in pieces
    ([600], [65], 32, 8, 128, 16),                 # two row blocks, the last of 1 row
    ([777, 90], [230, 1], 16, 2, 64, 16),          # group 8, head_dim 64, + a decode row
    ([700, 47], [300, 1], 32, 8, 128, 32),         # 32-token blocks
])
def test_fp8_prefill_edge_shapes(lens, q_lens, nq, nkv, d, bs):
    """Chunked-prefill rows over the 8-bit cache (the tcgen05 kernel on
    f16(code * scale)) against the oracle, with every unwritten slot of the
    pool holding NaN codes and scales."""
    b = _mixed(lens, q_lens, nq, nkv, d, seed=sum(lens) % 89, bs=bs)
    got, ref = fp8_step(b, poison=True)
    assert_attn_close(got, ref, f"fp8 prefill lens={lens} q_lens={q_lens} nq={nq} nkv={nkv} "
                                f"d={d} bs={bs}")


def test_fp8_mixed_step_workload():
    """The mixed chunked-prefill step (a 512-token chunk over 3,584 cached
    tokens plus 128 decode rows, 32/8 heads, d 128) over the 8-bit cache."""
    got, ref = fp8_step(W.mixed_step(poison=False), poison=True)
    assert_attn_close(got, ref, "fp8 mixed step")


@pytest.mark.parametrize("mag", [1e-2, 3e3])
def test_fp8_prefill_small_and_large_values(mag):
    """Keys and values far from unit size through the prefill kernel's f16
    operands: f16(code * scale) must neither flush small rows nor overflow
    large ones.  Compared after dividing by mag.  Every row sees at least 130
    keys, so the outputs stay near unit size: a row of one or two keys can
    reach |out| ~ 5, where the bf16 output's own rounding (2^-9 relative) is
    already 1e-2."""
    b = _mixed([700, 230], [300, 100], seed=23)
    for name in ("k_cache", "k_new", "v_cache", "v_new"):
        a = W.f32_from_bf16(getattr(b, name)) * np.float32(mag)
        setattr(b, name, W.bf16_from_f32(a.astype(np.float32)))
    # the scores keep unit size: the keys are scaled by mag, the queries by 1 / mag
    b.q = W.bf16_from_f32((W.f32_from_bf16(b.q) / np.float32(mag)).astype(np.float32))
    got, ref = fp8_step(b)
    assert_attn_close(got / mag, ref / mag, f"fp8 prefill values x {mag}")
