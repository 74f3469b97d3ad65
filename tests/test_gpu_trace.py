"""The continuous-batching trace on the GPU: every step's block swap-in and
swap-out, copy-on-write block copies, slot scatter and mixed decode /
chunked-prefill attention, replayed on the fp64 oracle from the same step
plans."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_174_gb300 import ops
from paged_kv_cache_174_gb300 import workloads as W
from paged_kv_cache_174_gb300.host import CONTINUOUS_BATCHING_TRACE, ContinuousBatchingTrace, \
    TraceConfig

from gpu_util import MAX_ABS, REL_L2, attn_errors, to_f64

pytestmark = pytest.mark.gpu


def _swaps(plan, dk, dv, kc, vc, host_g, host_o):
    """The step's swap-in, then its swap-out, through the library and the
    oracle; each side keeps its own host swap space."""
    if len(plan.swap_in):
        hs, db = plan.swap_in[:, 0], plan.swap_in[:, 1]
        ops.swap_in(dk, dv, W.int32_tensor(db, "cuda"), host_g[0][hs].contiguous(),
                    host_g[1][hs].contiguous())
        oracle.swap_in(kc, vc, db, host_o[0][hs], host_o[1][hs])
    if len(plan.swap_out):
        db, hs = plan.swap_out[:, 0], plan.swap_out[:, 1]
        shape = (len(db),) + tuple(host_g[0].shape[1:])
        tk = torch.empty(shape, dtype=torch.bfloat16).pin_memory()
        tv = torch.empty(shape, dtype=torch.bfloat16).pin_memory()
        ops.swap_out(dk, dv, W.int32_tensor(db, "cuda"), tk, tv)
        ops.check_device_errors()
        ok, ov = oracle.swap_out(kc, vc, db)
        assert np.array_equal(W.bits_of(tk), ok) and np.array_equal(W.bits_of(tv), ov), \
            f"step {plan.index}: swapped-out blocks differ from the oracle"
        host_g[0][hs], host_g[1][hs] = tk, tv
        host_o[0][hs], host_o[1][hs] = ok, ov


def _replay(cfg, steps, full_rows, sample_rows=24, seed=0):
    tr = ContinuousBatchingTrace(cfg)
    kc, vc = W.trace_initial_cache(cfg, tr.prefix_blocks)
    dk, dv = W.bf16_tensor(kc, "cuda"), W.bf16_tensor(vc, "cuda")
    scale = 1.0 / np.sqrt(cfg.head_dim)
    rng = np.random.default_rng(seed)
    worst = (0.0, 0.0)
    checked = 0
    hshape = (max(cfg.swap_blocks, 1), cfg.block_size, cfg.num_kv_heads, cfg.head_dim)
    host_o = (np.zeros(hshape, np.uint16), np.zeros(hshape, np.uint16))  # oracle's swap space
    host_g = (torch.zeros(hshape, dtype=torch.bfloat16), torch.zeros(hshape, dtype=torch.bfloat16))
    for _ in range(steps):
        plan = tr.step()
        _swaps(plan, dk, dv, kc, vc, host_g, host_o)
        if plan.num_tokens == 0:
            continue
        q, k, v = W.trace_step_inputs(cfg, plan.index, plan.num_tokens)
        if len(plan.copy_pairs):
            ops.copy_blocks(dk, dv, W.int32_tensor(plan.copy_pairs, "cuda"))
            oracle.copy_blocks(kc, vc, plan.copy_pairs)
        ops.reshape_and_cache(W.bf16_tensor(k, "cuda"), W.bf16_tensor(v, "cuda"), dk, dv,
                              W.int32_tensor(plan.slot_mapping, "cuda"))
        oracle.reshape_and_cache(k, v, kc, vc, plan.slot_mapping)
        dq = W.bf16_tensor(q, "cuda")
        out = ops.paged_attention(dq, dk, dv, W.int32_tensor(plan.block_tables, "cuda"),
                                  W.int32_tensor(plan.seq_lens, "cuda"),
                                  W.int32_tensor(plan.query_start_loc, "cuda"), scale,
                                  max_q_len=plan.max_q_len, max_seq_len=plan.max_seq_len)
        ops.check_device_errors()
        got = to_f64(out)
        if full_rows:
            ref = oracle.paged_attention(q, kc, vc, plan.block_tables, plan.seq_lens,
                                         plan.query_start_loc, scale)
            g, r = got, ref
        else:
            # sampled rows: always one decode row and one prefill row when present
            ql = np.diff(plan.query_start_loc)
            cand = list(rng.integers(0, len(plan.rids), size=sample_rows))
            if plan.num_decode:
                cand[0] = 0
            if (ql > 1).any():
                cand[1 % len(cand)] = int(np.flatnonzero(ql > 1)[0])
            samples = []
            for s in cand:
                i = int(rng.integers(0, ql[s]))
                samples.append((s, i, int(rng.integers(0, cfg.num_q_heads))))
            samples = np.array(samples, np.int32)
            r = oracle.paged_attention_rows(q, kc, vc, plan.block_tables, plan.seq_lens,
                                            plan.query_start_loc, scale, samples)
            tok = plan.query_start_loc[samples[:, 0]] + samples[:, 1]
            g = got[tok, samples[:, 2]]
        mx, rel = attn_errors(g, r)
        assert np.isfinite(g).all(), f"step {plan.index}: non-finite output"
        assert mx <= MAX_ABS and rel <= REL_L2, f"step {plan.index}: max {mx:.3e} rel {rel:.3e}"
        worst = (max(worst[0], mx), max(worst[1], rel))
        checked += 1
    assert checked > 0
    # the whole pool, bit for bit, after all the copies and scatters
    assert np.array_equal(W.bits_of(dk), kc), "K cache differs from the oracle"
    assert np.array_equal(W.bits_of(dv), vc), "V cache differs from the oracle"
    return tr, worst


def _sample_sequences(plan, rng, n=8):
    """n random sequences of the step, always one decode request and one
    chunked-prefill request when the step has them."""
    ql = np.diff(plan.query_start_loc)
    live = np.flatnonzero(ql > 0)
    pick = list(rng.choice(live, size=min(n, len(live)), replace=False))
    dec, pre = np.flatnonzero(ql == 1), np.flatnonzero(ql > 1)
    if len(dec) and not any(ql[s] == 1 for s in pick):
        pick[0] = int(rng.choice(dec))
    if len(pre) and not any(ql[s] > 1 for s in pick):
        pick[-1 if len(pick) > 1 else 0] = int(rng.choice(pre))
    return sorted(set(int(s) for s in pick))


def _rows_of(plan, seqs, rng, nq, rows_per_seq=4):
    """(sequence, row, q head) samples: for each sequence up to rows_per_seq
    rows (always its last one, the row that sees every key), every q head."""
    ql = np.diff(plan.query_start_loc)
    out = []
    for s in seqs:
        n = int(ql[s])
        rows = {n - 1} | set(int(i) for i in rng.integers(0, n, size=rows_per_seq - 1))
        for i in sorted(rows):
            out.extend((s, i, h) for h in range(nq))
    return np.array(out, np.int32)


def test_trace_full_configuration_every_step_three_paths():
    """The whole continuous-batching trace at its full configuration (200
    steps, 40000-block pool, 32/8 heads, d 128, 512-token chunks under a
    2048-token budget, up to 256 running requests, copy-on-write of the
    shared 500-token prefix), run three ways in lockstep on the same inputs:
    separate library calls; the step graph at the benchmark's maxima (2048
    tokens, 256 sequences, q_len 512) on device buffers; and the same graph
    with host I/O (inputs from and output to pinned host memory).  Every step,
    8 random requests (always one decode and one chunk when the step has
    them) are compared with the oracle, all q heads of up to 4 rows each; at
    the end every pool is compared with the oracle's bit for bit."""
    cfg = CONTINUOUS_BATCHING_TRACE
    driver = ContinuousBatchingTrace(cfg)
    plans = [driver.step() for _ in range(cfg.steps)]
    tr = ContinuousBatchingTrace(cfg)  # a fresh driver, for the prefix blocks
    kc, vc = W.trace_initial_cache(cfg, tr.prefix_blocks)
    scale = 1.0 / np.sqrt(cfg.head_dim)
    caches = [(W.bf16_tensor(kc, "cuda"), W.bf16_tensor(vc, "cuda")) for _ in range(3)]
    max_seq_len = max(p.max_seq_len for p in plans)
    max_blocks = max(p.block_tables.shape[1] for p in plans)
    max_pairs = max(len(p.copy_pairs) for p in plans)
    graphs = [ops.StepGraph(caches[i][0], caches[i][1], num_q_heads=cfg.num_q_heads,
                            max_tokens=cfg.budget, max_seqs=cfg.max_num_seqs,
                            max_blocks=max_blocks, max_pairs=max_pairs, max_q_len=cfg.chunk,
                            max_seq_len=max_seq_len, scale=scale, host_io=(i == 2))
              for i in (1, 2)]
    rng = np.random.default_rng(5)
    checked, kinds = 0, set()
    worst = [(0.0, 0.0)] * 3
    for p in plans:
        assert len(p.swap_in) == 0 and len(p.swap_out) == 0  # recompute preemption
        if p.num_tokens == 0:
            continue
        T = p.num_tokens
        q, k, v = W.trace_step_inputs(cfg, p.index, T)
        dq, dk_new, dv_new = (W.bf16_tensor(x, "cuda") for x in (q, k, v))
        # (1) separate calls
        ek, ev = caches[0]
        if len(p.copy_pairs):
            ops.copy_blocks(ek, ev, W.int32_tensor(p.copy_pairs, "cuda"))
        ops.reshape_and_cache(dk_new, dv_new, ek, ev, W.int32_tensor(p.slot_mapping, "cuda"))
        eout = ops.paged_attention(dq, ek, ev, W.int32_tensor(p.block_tables, "cuda"),
                                   W.int32_tensor(p.seq_lens, "cuda"),
                                   W.int32_tensor(p.query_start_loc, "cuda"), scale,
                                   max_q_len=p.max_q_len, max_seq_len=p.max_seq_len)
        # (2) the step graph on device buffers
        g = graphs[0]
        g.q[:T].copy_(dq)
        g.k_new[:T].copy_(dk_new)
        g.v_new[:T].copy_(dv_new)
        g.launch(p.slot_mapping, p.block_tables, p.seq_lens, p.query_start_loc, p.copy_pairs)
        gout = g.output()[:T].clone()
        # (3) the step graph with host I/O
        h = graphs[1]
        qh, kh, vh = h.inputs_host()
        qh[:T] = W.bf16_tensor(q, "cpu")
        kh[:T] = W.bf16_tensor(k, "cpu")
        vh[:T] = W.bf16_tensor(v, "cpu")
        h.launch(p.slot_mapping, p.block_tables, p.seq_lens, p.query_start_loc, p.copy_pairs)
        h.wait_output()
        hout = h.output_host()[:T].clone()
        ops.check_device_errors()
        # the oracle: copies, scatter, the sampled rows
        if len(p.copy_pairs):
            oracle.copy_blocks(kc, vc, p.copy_pairs)
        oracle.reshape_and_cache(k, v, kc, vc, p.slot_mapping)
        seqs = _sample_sequences(p, rng)
        ql = np.diff(p.query_start_loc)
        kinds |= {"decode" if ql[s] == 1 else "chunk" for s in seqs}
        smp = _rows_of(p, seqs, rng, cfg.num_q_heads)
        ref = oracle.paged_attention_rows(q, kc, vc, p.block_tables, p.seq_lens,
                                          p.query_start_loc, scale, smp)
        tok = p.query_start_loc[smp[:, 0]] + smp[:, 1]
        for i, out in enumerate((eout, gout, hout)):
            got = to_f64(out)[tok, smp[:, 2]]
            assert np.isfinite(got).all(), f"path {i} step {p.index}: non-finite output"
            mx, rel = attn_errors(got, ref)
            assert mx <= MAX_ABS and rel <= REL_L2, \
                f"path {i} step {p.index}: max {mx:.3e} rel {rel:.3e}"
            worst[i] = (max(worst[i][0], mx), max(worst[i][1], rel))
        checked += 1
    for g in graphs:
        g.close()
    assert checked == sum(1 for p in plans if p.num_tokens) and checked >= 190
    assert kinds == {"decode", "chunk"}
    for i, (dk, dv) in enumerate(caches):
        assert np.array_equal(W.bits_of(dk), kc), f"path {i}: K cache differs from the oracle"
        assert np.array_equal(W.bits_of(dv), vc), f"path {i}: V cache differs from the oracle"


@pytest.mark.parametrize("block_size", [16, 32])
def test_trace_small_heads_all_rows(block_size):
    cfg = TraceConfig(steps=40, arrival_rate=4.0, prompt_median=150.0, prompt_min=8,
                      prompt_max=700, output_mean=20.0, prefix=60, chunk=64, budget=256,
                      max_num_seqs=32, num_blocks=1200 * 16 // block_size, num_q_heads=8,
                      num_kv_heads=2, head_dim=64, seed=21, block_size=block_size)
    tr, worst = _replay(cfg, steps=40, full_rows=True)
    assert tr.total_copies > 0 and len(tr.finished) > 0


@pytest.mark.parametrize("preempt", ["swap", "auto"])
def test_trace_preempting_by_swap_all_rows(preempt):
    """A pool too small for the load: running requests are swapped out to host
    memory block by block and later swapped back into other physical blocks
    (every slot the trace never wrote holds NaN, so a block left behind or
    restored to the wrong place shows in the output)."""
    cfg = TraceConfig(steps=80, arrival_rate=1.0, prompt_median=200.0, prompt_min=8,
                      prompt_max=700, output_mean=60.0, prefix=40, chunk=128, budget=512,
                      max_num_seqs=64, num_blocks=160, num_q_heads=8, num_kv_heads=2,
                      head_dim=64, seed=13, preempt=preempt, swap_blocks=2000,
                      swap_min_tokens=250)
    tr, worst = _replay(cfg, steps=80, full_rows=True)
    s = tr.summary()
    assert s["preempt_swap"] > 0 and s["swap_in_blocks"] > 0
