"""Host-side block allocator and continuous-batching step driver.  CPU only."""
import dataclasses
import json
import os

import numpy as np
import pytest

import oracle
from paged_kv_cache_174_gb300.host import (BlockAllocator, ContinuousBatchingTrace, OutOfBlocks,
                                           TraceConfig)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def test_allocation_example_from_pages():
    g = _golden("allocation_example.json")
    a = BlockAllocator(g["pool_blocks"], 16)
    tables = {}
    for req, n in g["requests"].items():
        tables[req] = [a.allocate() for _ in range(n)]
    assert tables == g["expected_tables_in_order_of_allocation"]
    assert a.free_count == g["free_after_all"]
    a.free_all(tables[g["finish"]])
    assert a.free_count == g["free_after_finish"]
    reused = {a.allocate() for _ in range(len(g["reused_blocks_after_finish"]))}
    assert reused == set(g["reused_blocks_after_finish"])  # immediate reuse
    a.check()


def test_prefix_sharing_example_from_pages():
    g = _golden("prefix_sharing_example.json")
    bs, n, P = g["block_size"], g["num_requests"], g["prefix_tokens"]
    a = BlockAllocator(1000, bs)
    nblk = -(-P // bs)
    assert nblk == g["expected_prefix_blocks"]
    assert P // bs == g["expected_full_prefix_blocks"]
    assert P - (P // bs) * bs == g["expected_tokens_in_last_prefix_block"]
    first = [a.allocate() for _ in range(nblk)]
    others = [[a.share(b) for b in first] for _ in range(n - 1)]
    assert all(t == first for t in others)
    assert a.used_count == nblk * g["expected_physical_prefix_copies"]
    assert all(a.refcount(b) == 1 + g["expected_references_beyond_owner"] for b in first)
    assert n * nblk - a.used_count == g["expected_blocks_saved"]
    a.check()


def test_copy_on_write_and_refcounts():
    a = BlockAllocator(10, 16)
    t1 = [a.allocate(), a.allocate()]
    t2 = [a.share(b) for b in t1]
    copies = []
    assert a.make_private(t1, 0, copies) != t2[0]      # shared: copied
    assert copies == [(t2[0], t1[0])]
    assert a.refcount(t2[0]) == 1 and a.refcount(t1[0]) == 1
    assert a.make_private(t1, 0, copies) == t1[0]      # now private: no copy
    assert len(copies) == 1
    a.free_all(t2)
    assert a.refcount(t1[1]) == 1                      # still held by t1
    a.free_all(t1)
    assert a.free_count == 10
    a.check()


def test_exhaustion_is_an_error_not_ub():
    a = BlockAllocator(3, 16)
    [a.allocate() for _ in range(3)]
    with pytest.raises(OutOfBlocks):
        a.allocate()
    with pytest.raises(ValueError):
        BlockAllocator(0, 16)


def test_random_operations_keep_invariants():
    rng = np.random.default_rng(0)
    a = BlockAllocator(64, 16)
    tables = []
    for _ in range(3000):
        op = rng.integers(4)
        if op == 0 and a.free_count:
            tables.append([a.allocate()])
        elif op == 1 and tables:
            t = tables[rng.integers(len(tables))]
            tables.append([a.share(b) for b in t])
        elif op == 2 and tables:
            a.free_all(tables.pop(rng.integers(len(tables))))
        elif op == 3 and tables and a.free_count:
            t = tables[rng.integers(len(tables))]
            copies = []
            a.make_private(t, 0, copies)
            for s, d in copies:
                assert s != d and a.refcount(d) == 1
        a.check()
        held = {}
        for t in tables:
            for b in t:
                held[b] = held.get(b, 0) + 1
        assert held == a.refcounts()


def _small(**kw):
    base = dict(steps=60, arrival_rate=3.0, prompt_median=300.0, num_blocks=3000, seed=77,
                max_num_seqs=64)
    base.update(kw)
    return TraceConfig(**base)


def test_trace_is_deterministic():
    a = ContinuousBatchingTrace(_small())
    b = ContinuousBatchingTrace(_small())
    for _ in range(40):
        pa, pb = a.step(), b.step()
        for f in ("copy_pairs", "slot_mapping", "block_tables", "seq_lens", "query_start_loc"):
            assert np.array_equal(getattr(pa, f), getattr(pb, f)), f


@pytest.mark.parametrize("cfg", [_small(), _small(num_blocks=400, seed=5),
                                 _small(prompt_median=40.0, prompt_min=4, prefix=20, seed=9)])
def test_trace_step_invariants(cfg):
    tr = ContinuousBatchingTrace(cfg)
    bs = cfg.block_size
    saw_copy = saw_prefill = saw_decode = False
    for _ in range(cfg.steps):
        p = tr.step()
        tr.check()
        ql = np.diff(p.query_start_loc)
        assert p.num_tokens <= cfg.budget
        assert (ql >= 1).all() and (ql <= cfg.chunk).all()
        # decodes (q_len 1 of a request past its prompt) come first
        assert p.num_decode + p.num_prefill_tokens == p.num_tokens
        assert len(set(p.rids)) == len(p.rids), "a request twice in one step"
        # copies: distinct destinations, none of them a source
        dst = p.copy_pairs[:, 1].tolist()
        assert len(set(dst)) == len(dst)
        assert not set(dst) & set(p.copy_pairs[:, 0].tolist())
        # each new token's slot is the oracle's addressing of its position
        t = 0
        for s in range(len(p.rids)):
            for pos in range(p.seq_lens[s] - ql[s], p.seq_lens[s]):
                assert p.slot_mapping[t] == oracle.slot_of(p.block_tables[s], pos, bs)
                t += 1
        # slots written in one step are distinct
        assert len(set(p.slot_mapping.tolist())) == p.num_tokens
        # waste confined to the last block of each request
        for s in range(len(p.rids)):
            used = int((p.block_tables[s] >= 0).sum())
            assert used * bs - p.seq_lens[s] < bs
        saw_copy |= len(p.copy_pairs) > 0
        saw_prefill |= p.num_prefill_tokens > 0
        saw_decode |= p.num_decode > 0
    assert saw_copy and saw_prefill and saw_decode


def test_trace_preempts_under_memory_pressure():
    tr = ContinuousBatchingTrace(_small(num_blocks=120, arrival_rate=6.0, prompt_median=200.0,
                                        prompt_max=400, output_mean=400.0, seed=3))
    for _ in range(60):
        tr.step()
        tr.check()
    assert any(r.preemptions for r in list(tr.waiting) + tr.running + tr.finished)


def test_first_write_after_prefix_copies_the_shared_block():
    cfg = _small(arrival_rate=0.0)
    tr = ContinuousBatchingTrace(cfg)
    from paged_kv_cache_174_gb300.host.trace import Request
    tr.waiting.append(Request(0, 530, 3, 0))
    p = tr.step()
    # positions 500..529: block 31 (tokens 496..511) is shared, so it is copied
    assert p.copy_pairs.tolist() == [[tr.prefix_blocks[31], p.block_tables[0, 31]]]
    assert p.block_tables[0, :31].tolist() == tr.prefix_blocks[:31]
    assert p.seq_lens.tolist() == [530] and p.query_start_loc.tolist() == [0, 30]


def _token_id_replay(cfg, steps):
    """Replay every plan on a model of the pool in which each slot holds the
    identity of the token whose K/V it caches (prefix position i -> i + 1,
    position p of request r -> (r + 1) * 10**6 + p, never written -> 0),
    executing the step in its stated order: swap-in, swap-out, block copies,
    scatter.  Then every scheduled request's block table must read its own
    tokens at positions 0 .. seq_len - 1: a wrong swap order, a swapped
    block left out or a copy into a live block shows up here."""
    tr = ContinuousBatchingTrace(cfg)
    bs = cfg.block_size
    pool = np.zeros((cfg.num_blocks, bs), np.int64)
    for i in range(cfg.prefix):
        pool[tr.prefix_blocks[i // bs], i % bs] = i + 1
    host = np.zeros((max(cfg.swap_blocks, 1), bs), np.int64)
    prompt = {}
    for _ in range(steps):
        p = tr.step()
        tr.check()
        for r in list(tr.waiting) + list(tr.swapped) + tr.running + tr.finished:
            prompt[r.rid] = r.prompt_len
        if len(p.swap_in):
            pool[p.swap_in[:, 1]] = host[p.swap_in[:, 0]]
        if len(p.swap_out):
            host[p.swap_out[:, 1]] = pool[p.swap_out[:, 0]]
        for src, dst in p.copy_pairs:
            pool[dst] = pool[src]

        def ident(rid, pos):
            return pos + 1 if pos < min(prompt[rid], cfg.prefix) else (rid + 1) * 10**6 + pos

        pool.reshape(-1)[p.slot_mapping] = [ident(int(r), int(q))
                                            for r, q in zip(p.token_rid, p.positions)]
        for s, rid in enumerate(p.rids):
            L = int(p.seq_lens[s])
            pos = np.arange(L)
            got = pool[p.block_tables[s, pos // bs], pos % bs]
            want = np.array([ident(rid, int(q)) for q in pos])
            assert np.array_equal(got, want), f"step {p.index}: request {rid} reads wrong tokens"
    return tr


@pytest.mark.parametrize("preempt", ["recompute", "swap", "auto"])
def test_preemption_keeps_every_request_reading_its_own_tokens(preempt):
    cfg = _small(num_blocks=160, arrival_rate=1.0, prompt_median=200.0, prompt_max=700,
                 output_mean=60.0, prefix=40, chunk=128, budget=512, seed=13, preempt=preempt,
                 swap_blocks=2000, swap_min_tokens=250)
    tr = _token_id_replay(cfg, 150)
    s = tr.summary()
    assert s["finished"] > 10
    if preempt == "recompute":
        assert s["preempt_recompute"] > 0 and s["preempt_swap"] == 0
    elif preempt == "swap":
        assert s["preempt_swap"] > 0 and s["preempt_recompute"] == 0
        assert s["swap_in_blocks"] > 0 and s["swap_out_blocks"] >= s["swap_in_blocks"]
    else:
        assert s["preempt_swap"] > 0 and s["preempt_recompute"] > 0


def test_swap_falls_back_to_recompute_when_the_host_space_is_full():
    cfg = _small(num_blocks=160, arrival_rate=1.0, prompt_median=200.0, prompt_max=700,
                 output_mean=60.0, prefix=40, chunk=128, budget=512, seed=13, preempt="swap",
                 swap_blocks=12)
    tr = _token_id_replay(cfg, 150)
    s = tr.summary()
    assert s["preempt_swap"] > 0 and s["preempt_recompute"] > 0


def test_swapped_request_resumes_with_its_prefix_shared_again():
    """A victim holding prefix blocks copies out only its private blocks; on
    resumption it shares the same prefix blocks and gets its own blocks back
    through swap-in (host slot -> fresh device block)."""
    cfg = _small(arrival_rate=0.0, num_blocks=36, prefix=100, chunk=512, budget=2048,
                 preempt="swap", swap_blocks=64)
    from paged_kv_cache_174_gb300.host.trace import Request
    tr = ContinuousBatchingTrace(cfg)   # 7 prefix blocks
    tr.waiting.append(Request(0, 300, 100, 0))   # 19 blocks
    tr.waiting.append(Request(1, 300, 100, 0))
    tr.step()
    tr.step()
    assert [r.rid for r in tr.running] == [0, 1]
    # both decode; the pool runs dry when a request crosses into a new block
    seen_out = None
    for _ in range(40):
        p = tr.step()
        tr.check()
        if len(p.swap_out):
            seen_out = p
            break
    assert seen_out is not None
    victim = tr.swapped[0]
    assert victim.host_table[:6] == [-1] * 6
    # prefix block 6 (tokens 96..99 of 112) was copied on write: private, swapped out
    assert all(h >= 0 for h in victim.host_table[6:])
    assert len(seen_out.swap_out) == len(victim.host_table) - 6
    assert sorted(seen_out.swap_out[:, 1].tolist()) == sorted(victim.host_table[6:])
    # once the other request finishes, the victim comes back
    for _ in range(200):
        p = tr.step()
        tr.check()
        if len(p.swap_in):
            break
    assert sorted(p.swap_in[:, 0].tolist()) == sorted(seen_out.swap_out[:, 1].tolist())
    assert victim in tr.running and victim.table[:6] == tr.prefix_blocks[:6]
    assert victim.table[6:6 + len(p.swap_in)] == p.swap_in[:, 1].tolist()
