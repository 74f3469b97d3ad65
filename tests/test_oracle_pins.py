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
