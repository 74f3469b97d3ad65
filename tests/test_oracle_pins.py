"""Pins for the fp64 CPU oracle: each test ties it to something other than
itself (a value the pages print, a closed form, a library routine on dense
memory, or an invariant that must hold exactly), so that a dropped term, a
wrong sign or index, or a transposed operand in the oracle fails here.

CPU only.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_174_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------------------
# helpers: dense, contiguous inputs turned into a paged cache by whole-block
# assignment (logical block b of a request is physical block table[b])
# ---------------------------------------------------------------------------

def _paged_from_dense(rng, lens, q_lens, nq, nkv, d, bs, num_blocks, scale=None, poison=True):
    """Returns (dense pieces, paged inputs for the oracle)."""
    S = len(lens)
    nblk = [-(-L // bs) for L in lens]
    perm = rng.permutation(num_blocks)
    tables, off = [], 0
    for n in nblk:
        tables.append(perm[off:off + n])
        off += n
    maxb = max(nblk)
    bt = np.full((S, maxb), -1, np.int32)
    fill = W.BF16_NAN if poison else np.uint16(0)
    kc = np.full((num_blocks, bs, nkv, d), fill, np.uint16)
    vc = np.full((num_blocks, bs, nkv, d), fill, np.uint16)
    Ks, Vs, Qs = [], [], []
    for s, L in enumerate(lens):
        K = W.randn_bf16(rng, (L, nkv, d))
        V = W.randn_bf16(rng, (L, nkv, d))
        Q = W.randn_bf16(rng, (L, nq, d))  # a query for every position
        Ks.append(K), Vs.append(V), Qs.append(Q)
        bt[s, :nblk[s]] = tables[s]
        for b in range(nblk[s]):
            rows = K[b * bs:(b + 1) * bs]
            kc[tables[s][b], :rows.shape[0]] = rows
            vc[tables[s][b], :rows.shape[0]] = V[b * bs:(b + 1) * bs]
    qsl = np.zeros(S + 1, np.int32)
    qsl[1:] = np.cumsum(q_lens)
    q = np.concatenate([Qs[s][lens[s] - q_lens[s]:] for s in range(S)], axis=0)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    paged = dict(q=q, k_cache=kc, v_cache=vc, block_tables=bt,
                 seq_lens=np.asarray(lens, np.int32), query_start_loc=qsl, scale=scale)
    return (Qs, Ks, Vs), paged


def _sdpa_reference(Qs, Ks, Vs, lens, q_lens, scale):
    """torch's scaled_dot_product_attention in float64 on dense memory:
    full square causal attention over all positions (is_causal=True), GQA via
    enable_gqa, keeping the last q_len query rows of each request."""
    outs = []
    for s, L in enumerate(lens):
        q = torch.from_numpy(W.f32_from_bf16(Qs[s]).astype(np.float64)).permute(1, 0, 2)
        k = torch.from_numpy(W.f32_from_bf16(Ks[s]).astype(np.float64)).permute(1, 0, 2)
        v = torch.from_numpy(W.f32_from_bf16(Vs[s]).astype(np.float64)).permute(1, 0, 2)
        o = torch.nn.functional.scaled_dot_product_attention(
            q[None], k[None], v[None], is_causal=True, scale=scale, enable_gqa=True)[0]
        outs.append(o.permute(1, 0, 2)[L - q_lens[s]:].numpy())
    return np.concatenate(outs, axis=0)


CASES = [
    # (lens, q_lens, nq, nkv, d, bs)
    ([5, 17, 33, 48], [1, 1, 1, 1], 4, 2, 64, 16),           # the tiny decode shape
    ([1, 2, 16, 31, 40], [1, 2, 16, 7, 40], 8, 2, 16, 16),   # mixed prefill / decode
    ([23, 9, 64], [5, 9, 3], 6, 3, 8, 4),                    # group 2, block 4
    ([37, 50], [37, 11], 4, 4, 32, 5),                       # no GQA, odd block
    ([70], [70], 8, 1, 16, 16),                              # multi-query
]


@pytest.mark.parametrize("lens,q_lens,nq,nkv,d,bs", CASES)
def test_pin_dense_library_attention(lens, q_lens, nq, nkv, d, bs):
    """P1: the paged oracle equals torch's dense fp64 SDPA on the contiguous
    K/V (causal, GQA), up to fp64 rounding."""
    rng = np.random.default_rng(7 + sum(lens))
    nb = sum(-(-L // bs) for L in lens) + 5
    (Qs, Ks, Vs), P = _paged_from_dense(rng, lens, q_lens, nq, nkv, d, bs, nb)
    got = oracle.paged_attention(**P)
    ref = _sdpa_reference(Qs, Ks, Vs, lens, q_lens, P["scale"])
    assert got.shape == ref.shape
    np.testing.assert_allclose(got, ref, rtol=1e-10, atol=1e-12)


def test_pin_rows_equal_full():
    rng = np.random.default_rng(3)
    lens, q_lens = [40, 18], [40, 3]
    (Qs, Ks, Vs), P = _paged_from_dense(rng, lens, q_lens, 4, 2, 16, 16, 12)
    full = oracle.paged_attention(**P)
    samples = np.array([[0, 0, 0], [0, 39, 3], [1, 2, 1], [1, 0, 2]], np.int32)
    rows = oracle.paged_attention_rows(**P, samples=samples)
    qsl = P["query_start_loc"]
    for n, (s, i, h) in enumerate(samples):
        assert np.array_equal(rows[n], full[qsl[s] + i, h])


def test_pin_closed_form_two_keys():
    """Two keys with scores ln 3 and 0 give weights 3/4 and 1/4."""
    bs, d = 16, 2
    one = W.bf16_from_f32(np.array([1.0], np.float32))[0]
    zero = np.uint16(0)
    q = np.array([[[one, zero]]], np.uint16)  # [T=1, nq=1, d=2]
    kc = np.full((2, bs, 1, d), W.BF16_NAN, np.uint16)
    vc = np.full((2, bs, 1, d), W.BF16_NAN, np.uint16)
    kc[1, 0, 0] = [one, zero]       # key 0 = (1, 0)
    kc[1, 1, 0] = [zero, zero]      # key 1 = (0, 0)
    vc[1, 0, 0] = [one, zero]       # value 0 = (1, 0)
    vc[1, 1, 0] = [zero, one]       # value 1 = (0, 1)
    out = oracle.paged_attention(q, kc, vc, np.array([[1]], np.int32), np.array([2], np.int32),
                                 np.array([0, 1], np.int32), scale=math.log(3.0))
    np.testing.assert_allclose(out[0, 0], [0.75, 0.25], rtol=0, atol=1e-15)


def test_pin_length_one_returns_v():
    """P3: a request with one token attends only to itself: out == v exactly."""
    rng = np.random.default_rng(11)
    b = W.make_batch("t", [1, 1, 1], [1, 1, 1], num_q_heads=8, num_kv_heads=2, head_dim=32,
                     block_size=16, num_blocks=9, seed=5)
    kc, vc = b.k_cache.copy(), b.v_cache.copy()
    oracle.reshape_and_cache(b.k_new, b.v_new, kc, vc, b.slot_mapping)
    out = oracle.paged_attention(b.q, kc, vc, b.block_tables, b.seq_lens, b.query_start_loc,
                                 b.scale)
    v = W.f32_from_bf16(b.v_new).astype(np.float64)  # [T, nkv, d]
    for h in range(8):
        assert np.array_equal(out[:, h], v[:, h // 4])
    del rng


def test_pin_identical_keys_mean_of_v():
    """P4: if every key is the same vector, all weights are equal and the
    output is the plain mean of the visible values."""
    rng = np.random.default_rng(12)
    lens, q_lens, nq, nkv, d, bs = [29, 16], [4, 1], 4, 2, 16, 8
    (Qs, Ks, Vs), P = _paged_from_dense(rng, lens, q_lens, nq, nkv, d, bs, 10)
    kc = P["k_cache"]
    key = W.randn_bf16(rng, (nkv, d))
    bt = P["block_tables"]
    for s, L in enumerate(lens):
        for b in range(-(-L // bs)):
            n = min(bs, L - b * bs)
            kc[bt[s, b], :n] = key
    out = oracle.paged_attention(**P)
    qsl = P["query_start_loc"]
    for s, L in enumerate(lens):
        V = W.f32_from_bf16(Vs[s]).astype(np.float64)
        for i in range(q_lens[s]):
            p = L - q_lens[s] + i
            for h in range(nq):
                np.testing.assert_allclose(out[qsl[s] + i, h], V[:p + 1, h // 2].mean(axis=0),
                                           rtol=1e-12, atol=1e-14)


def test_pin_physical_permutation_invariance():
    """P2: relabelling physical blocks (moving their contents and remapping the
    tables) leaves the output bit-identical."""
    rng = np.random.default_rng(13)
    lens, q_lens = [45, 3, 70], [1, 3, 12]
    nb = 20
    _, P = _paged_from_dense(rng, lens, q_lens, 8, 4, 16, 16, nb)
    a = oracle.paged_attention(**P)
    pi = rng.permutation(nb).astype(np.int32)
    kc2 = np.empty_like(P["k_cache"])
    vc2 = np.empty_like(P["v_cache"])
    kc2[pi] = P["k_cache"]
    vc2[pi] = P["v_cache"]
    bt2 = np.where(P["block_tables"] >= 0, pi[np.maximum(P["block_tables"], 0)], -1)
    b = oracle.paged_attention(**{**P, "k_cache": kc2, "v_cache": vc2,
                                  "block_tables": bt2.astype(np.int32)})
    assert np.array_equal(a, b)


def test_pin_poison_does_not_leak():
    """P9: NaN in every unused slot, unused block and padding table entry
    leaves the output finite and identical to a zero-filled pool."""
    rng1 = np.random.default_rng(14)
    rng2 = np.random.default_rng(14)
    lens, q_lens = [17, 33, 2], [1, 5, 2]
    _, P1 = _paged_from_dense(rng1, lens, q_lens, 4, 2, 16, 16, 12, poison=True)
    _, P2 = _paged_from_dense(rng2, lens, q_lens, 4, 2, 16, 16, 12, poison=False)
    a = oracle.paged_attention(**P1)
    b = oracle.paged_attention(**P2)
    assert np.isfinite(a).all()
    assert np.array_equal(a, b)


def test_pin_causal_future_keys_ignored():
    """P10: changing keys/values after a query row's position leaves that row
    unchanged (bottom-right aligned causal mask of a chunk)."""
    rng = np.random.default_rng(15)
    lens, q_lens, bs = [40], [10], 16
    _, P = _paged_from_dense(rng, lens, q_lens, 4, 2, 16, bs, 4)
    a = oracle.paged_attention(**P)
    kc, vc, bt = P["k_cache"].copy(), P["v_cache"].copy(), P["block_tables"]
    cut = 35  # rows 0..4 of the chunk sit at positions 30..34
    for pos in range(cut, 40):
        kc[bt[0, pos // bs], pos % bs] = W.randn_bf16(rng, (2, 16))
        vc[bt[0, pos // bs], pos % bs] = W.randn_bf16(rng, (2, 16))
    b = oracle.paged_attention(**{**P, "k_cache": kc, "v_cache": vc})
    assert np.array_equal(a[:5], b[:5])
    assert not np.array_equal(a[5:], b[5:])


def test_pin_block_table_example_from_pages():
    """P6: the printed Block Table (0->7, 1->12, 2->3, 3->19, 16 tokens per
    block) and the 48-token = 3 logical blocks example."""
    g = _golden("block_table_example.json")
    table = np.array(g["block_table"], np.int32)
    for pos, slot in g["expected_slots"].items():
        assert oracle.slot_of(table, int(pos), g["block_size"]) == slot
    for lb, (lo, hi) in g["logical_block_of_tokens_48"].items():
        for pos in range(lo, hi + 1):
            assert oracle.slot_of(table, pos, 16) // 16 == table[int(lb)]
    # the scatter puts a 48-token request's rows into physical blocks 7, 12, 3
    nkv, d = 1, 8
    k = (np.arange(48 * nkv * d, dtype=np.uint16) + 1).reshape(48, nkv, d)
    kc = np.zeros((20, 16, nkv, d), np.uint16)
    vc = np.zeros_like(kc)
    slots = np.array([oracle.slot_of(table, p, 16) for p in range(48)], np.int32)
    oracle.reshape_and_cache(k, k, kc, vc, slots)
    for lb in range(3):
        assert np.array_equal(kc[table[lb]], k[16 * lb:16 * (lb + 1)])
    assert not kc[table[3]].any()


def test_generator_slots_agree_with_oracle_addressing():
    """The seeded generator's slot mapping is the oracle's addressing rule."""
    b = W.make_batch("t", [5, 17, 33, 48], [1, 3, 16, 20], num_q_heads=4, num_kv_heads=2,
                     head_dim=8, block_size=16, num_blocks=16, seed=2)
    t = 0
    for s in range(b.num_seqs):
        L, ql = int(b.seq_lens[s]), int(b.q_lens[s])
        for pos in range(L - ql, L):
            assert b.slot_mapping[t] == oracle.slot_of(b.block_tables[s], pos, 16)
            t += 1


def test_pin_reshape_and_cache_skips_negative_and_is_bit_copy():
    rng = np.random.default_rng(16)
    k = W.randn_bf16(rng, (6, 2, 8))
    v = W.randn_bf16(rng, (6, 2, 8))
    kc = np.full((4, 4, 2, 8), W.BF16_NAN, np.uint16)
    vc = kc.copy()
    slots = np.array([0, -1, 5, 15, -7, 9], np.int32)
    oracle.reshape_and_cache(k, v, kc, vc, slots)
    kf, vf = kc.reshape(16, 2, 8), vc.reshape(16, 2, 8)
    for t, s in enumerate(slots):
        if s >= 0:
            assert np.array_equal(kf[s], k[t]) and np.array_equal(vf[s], v[t])
    untouched = [i for i in range(16) if i not in set(slots.tolist())]
    assert (kf[untouched] == W.BF16_NAN).all()
    with pytest.raises(oracle.OracleError):
        oracle.reshape_and_cache(k[:1], v[:1], kc, vc, np.array([16], np.int32))


def test_pin_copy_blocks_cow():
    """P5: after a copy, dst equals src bit for bit, src and every other block
    are unchanged (whole-cache hash)."""
    rng = np.random.default_rng(17)
    kc = W.randn_bf16(rng, (10, 16, 2, 8))
    vc = W.randn_bf16(rng, (10, 16, 2, 8))
    k0, v0 = kc.copy(), vc.copy()
    pairs = np.array([[3, 7], [3, 1], [9, 0]], np.int32)
    oracle.copy_blocks(kc, vc, pairs)
    for src, dst in pairs:
        assert np.array_equal(kc[dst], k0[src]) and np.array_equal(vc[dst], v0[src])
    others = [i for i in range(10) if i not in (7, 1, 0)]
    assert np.array_equal(kc[others], k0[others]) and np.array_equal(vc[others], v0[others])
    with pytest.raises(oracle.OracleError):
        oracle.copy_blocks(kc, vc, np.array([[0, 10]], np.int32))


def test_pin_split_merge_identity():
    """The log-sum-exp merge a split-KV kernel uses is exact: attention over
    keys 0..p equals the merge of attention over two disjoint key ranges,
    each computed by the oracle as a request whose keys are that range
    (the query placed last so that every key is visible)."""
    rng = np.random.default_rng(18)
    d, bs, L, cut = 16, 16, 50, 21
    K = W.randn_bf16(rng, (L, 1, d))
    V = W.randn_bf16(rng, (L, 1, d))
    q = W.randn_bf16(rng, (1, 1, d))

    def run(lo, hi):
        n = hi - lo
        nb = -(-n // bs)
        kc = np.zeros((nb, bs, 1, d), np.uint16)
        vc = np.zeros_like(kc)
        kc.reshape(nb * bs, 1, d)[:n] = K[lo:hi]
        vc.reshape(nb * bs, 1, d)[:n] = V[lo:hi]
        o = oracle.paged_attention(q, kc, vc, np.arange(nb, dtype=np.int32)[None],
                                   np.array([n], np.int32), np.array([0, 1], np.int32), 0.25)
        qf = W.f32_from_bf16(q).astype(np.float64)[0, 0]
        x = 0.25 * (W.f32_from_bf16(K[lo:hi]).astype(np.float64)[:, 0] @ qf)
        m = x.max()
        return o[0, 0], m, np.exp(x - m).sum()

    full, _, _ = run(0, L)
    o1, m1, l1 = run(0, cut)
    o2, m2, l2 = run(cut, L)
    m = max(m1, m2)
    w1, w2 = l1 * math.exp(m1 - m), l2 * math.exp(m2 - m)
    np.testing.assert_allclose((o1 * w1 + o2 * w2) / (w1 + w2), full, rtol=1e-12, atol=1e-14)


def test_oracle_rejects_bad_lengths():
    b = W.tiny_decode()
    with pytest.raises(oracle.OracleError):
        oracle.paged_attention(b.q, b.k_cache, b.v_cache, b.block_tables,
                               np.array([5, 17, 33, 49], np.int32), b.query_start_loc, b.scale)
    with pytest.raises(oracle.OracleError):
        oracle.paged_attention(b.q, b.k_cache, b.v_cache, b.block_tables,
                               np.array([0, 17, 33, 48], np.int32), b.query_start_loc, b.scale)


def test_pin_swap_round_trip_and_library_gather():
    """Swap is a block-grained bit copy ("vLLM中的PagedAttention机制与显存优化实践",
    section 2.1): swap-out equals numpy's take along the block axis; swapping
    the blocks back in at other ids moves them there bit for bit and leaves
    every other block alone."""
    rng = np.random.default_rng(21)
    nb, bs, nkv, d = 12, 16, 2, 64
    kc = rng.integers(0, 65536, size=(nb, bs, nkv, d), dtype=np.uint16)
    vc = rng.integers(0, 65536, size=(nb, bs, nkv, d), dtype=np.uint16)
    ids = np.array([7, 2, 9, 2], np.int32)  # repeats allowed on swap-out
    hk, hv = oracle.swap_out(kc, vc, ids)
    assert np.array_equal(hk, np.take(kc, ids, axis=0))
    assert np.array_equal(hv, np.take(vc, ids, axis=0))
    k2, v2 = kc.copy(), vc.copy()
    dst = np.array([0, 11, 4, 5], np.int32)
    oracle.swap_in(k2, v2, dst, hk, hv)
    for i, b in enumerate(dst):
        assert np.array_equal(k2[b], kc[ids[i]]) and np.array_equal(v2[b], vc[ids[i]])
    others = np.setdiff1d(np.arange(nb), dst)
    assert np.array_equal(k2[others], kc[others]) and np.array_equal(v2[others], vc[others])
    with pytest.raises(oracle.OracleError):
        oracle.swap_out(kc, vc, np.array([nb], np.int32))
    with pytest.raises(oracle.OracleError):
        oracle.swap_in(k2, v2, np.array([-1], np.int32), hk[:1], hv[:1])


# ---------------------------------------------------------------------------
# The 8-bit (FP8 E4M3) cache variant
# ---------------------------------------------------------------------------

def test_pin_e4m3_codec_against_torch():
    """The oracle's E4M3 decode equals torch.float8_e4m3fn on all 256 codes;
    its encode equals torch's conversion on every finite value, every midpoint
    between neighbours (ties to even) and random values; beyond 448 it
    saturates."""
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.e4m3_to_double(codes)
    assert np.array_equal(got, ref, equal_nan=True)
    fin = np.unique(np.abs(got[np.isfinite(got)]))
    mids = (fin[1:] + fin[:-1]) / 2
    rng = np.random.default_rng(3)
    vals = np.concatenate([fin, mids, -fin, -mids, rng.uniform(-448, 448, 4000),
                           rng.normal(0, 1e-2, 4000)]).astype(np.float32)
    t = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_from_float(vals), t)
    assert oracle.e4m3_from_float(np.array([460, 1000, 3e38, -1000], np.float32)).tolist() == \
        [0x7E, 0x7E, 0x7E, 0xFE]
    assert oracle.e4m3_from_float(np.array([np.nan], np.float32)).tolist() == [0x7F]
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9 and got[0x08] == 2.0 ** -6


def _torch_quantise(x_bf16_bits):
    """Independent quantiser: per row (last axis) amax / 448 in fp32, x / scale
    in fp32, torch's float8_e4m3fn conversion."""
    x = torch.from_numpy(W.f32_from_bf16(x_bf16_bits))
    amax = x.abs().amax(dim=-1, keepdim=True)
    sc = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    codes = (x / sc).to(torch.float8_e4m3fn)
    return codes.view(torch.uint8).numpy(), sc[..., 0].numpy()


@pytest.mark.parametrize("lens,q_lens,nq,nkv,d,bs", CASES[:3])
def test_pin_fp8_cache_attention_equals_dense_sdpa_on_dequantised(lens, q_lens, nq, nkv, d, bs):
    """Scatter into the 8-bit cache gives, through the block tables, exactly
    the codes and scales of an independent torch quantiser of the dense rows;
    attention over the 8-bit cache equals torch's fp64 SDPA on the dequantised
    dense K/V."""
    rng = np.random.default_rng(11 + sum(lens))
    nb = sum(-(-L // bs) for L in lens) + 3
    (Qs, Ks, Vs), P = _paged_from_dense(rng, lens, q_lens, nq, nkv, d, bs, nb)
    kc8, vc8, ks, vs = oracle.fp8_cache(nb, bs, nkv, d)
    for s, L in enumerate(lens):
        slots = np.array([oracle.slot_of(P["block_tables"][s], p, bs) for p in range(L)],
                         np.int32)
        oracle.reshape_and_cache_fp8(Ks[s], Vs[s], kc8, vc8, ks, vs, slots)
    Kd, Vd = [], []
    for s, L in enumerate(lens):
        kq, kscale = _torch_quantise(Ks[s])
        vq, vscale = _torch_quantise(Vs[s])
        t = P["block_tables"][s]
        pos = np.arange(L)
        blk, row = t[pos // bs], pos % bs
        assert np.array_equal(kc8[blk, row], kq) and np.array_equal(vc8[blk, row], vq)
        assert np.array_equal(ks[blk, row], kscale) and np.array_equal(vs[blk, row], vscale)
        deq = lambda c, sc: torch.from_numpy(c.copy()).view(torch.float8_e4m3fn).to(
            torch.float64).numpy() * sc[..., None].astype(np.float64)
        Kd.append(deq(kq, kscale))
        Vd.append(deq(vq, vscale))
    got = oracle.paged_attention_fp8(P["q"], kc8, vc8, ks, vs, P["block_tables"], P["seq_lens"],
                                     P["query_start_loc"], P["scale"])
    outs = []
    for s, L in enumerate(lens):
        q = torch.from_numpy(W.f32_from_bf16(Qs[s]).astype(np.float64)).permute(1, 0, 2)
        k = torch.from_numpy(Kd[s]).permute(1, 0, 2)
        v = torch.from_numpy(Vd[s]).permute(1, 0, 2)
        o = torch.nn.functional.scaled_dot_product_attention(
            q[None], k[None], v[None], is_causal=True, scale=P["scale"], enable_gqa=True)[0]
        outs.append(o.permute(1, 0, 2)[L - q_lens[s]:].numpy())
    np.testing.assert_allclose(got, np.concatenate(outs, axis=0), rtol=1e-10, atol=1e-12)


def test_pin_fp8_quantisation_error_bound_and_edges():
    """Each dequantised value is within half a code spacing (times the row
    scale) of the input; the row's largest magnitude maps to +-448 exactly; an
    all-zero row has scale 1 and zero codes."""
    rng = np.random.default_rng(5)
    k = W.randn_bf16(rng, (40, 2, 64))
    k[3, 1] = 0  # an all-zero row
    kc8, vc8, ks, vs = oracle.fp8_cache(4, 16, 2, 64)
    oracle.reshape_and_cache_fp8(k, k, kc8, vc8, ks, vs, np.arange(40, dtype=np.int32))
    x = W.f32_from_bf16(k).astype(np.float64)
    codes = kc8.reshape(-1, 2, 64)[:40]
    sc = ks.reshape(-1, 2)[:40].astype(np.float64)
    deq = oracle.e4m3_to_double(codes) * sc[..., None]
    y = np.abs(x) / np.where(sc > 0, sc, 1)[..., None]
    e = np.floor(np.log2(np.maximum(y, 2.0 ** -6)))
    half = 2.0 ** (e - 3) / 2 * sc[..., None]
    assert (np.abs(deq - x) <= half * (1 + 1e-6) + 1e-30).all()
    assert sc[3, 1] == 1.0 and (codes[3, 1] == 0).all()
    am = np.abs(x).argmax(axis=-1)
    top = np.take_along_axis(codes, am[..., None], axis=-1)[..., 0]
    nz = np.abs(x).max(axis=-1) > 0
    assert set((top[nz] & 0x7F).tolist()) == {0x7E}
