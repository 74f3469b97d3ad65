"""The serving step captured as a CUDA graph (pa_step_graph_*): the
continuous-batching trace replayed through one graph launch per step, with
every step padded to fixed maxima, against the fp64 oracle; and padded block
copy lists."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_174_gb300 import ops
from paged_kv_cache_174_gb300 import workloads as W
from paged_kv_cache_174_gb300.host import ContinuousBatchingTrace, TraceConfig

from gpu_util import MAX_ABS, REL_L2, assert_attn_close, attn_errors, run_oracle_step, to_f64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("block_size", [16, 32])
def test_trace_through_the_step_graph(block_size):
    cfg = TraceConfig(steps=40, arrival_rate=4.0, prompt_median=150.0, prompt_min=8,
                      prompt_max=700, output_mean=20.0, prefix=60, chunk=64, budget=256,
                      max_num_seqs=32, num_blocks=1200 * 16 // block_size, num_q_heads=8,
                      num_kv_heads=2, head_dim=64, seed=21, block_size=block_size)
    plans = [p for p in (ContinuousBatchingTrace(cfg).step() for _ in range(cfg.steps))]
    tr = ContinuousBatchingTrace(cfg)  # a second driver for the prefix blocks
    kc, vc = W.trace_initial_cache(cfg, tr.prefix_blocks)
    dk, dv = W.bf16_tensor(kc, "cuda"), W.bf16_tensor(vc, "cuda")
    max_seq_len = max(p.max_seq_len for p in plans)
    g = ops.StepGraph(dk, dv, num_q_heads=cfg.num_q_heads, max_tokens=cfg.budget,
                      max_seqs=cfg.max_num_seqs, max_blocks=-(-max_seq_len // block_size),
                      max_pairs=max(len(p.copy_pairs) for p in plans) + 2,
                      max_q_len=cfg.chunk, max_seq_len=max_seq_len,
                      scale=1.0 / np.sqrt(cfg.head_dim))
    checked = 0
    for p in plans:
        if p.num_tokens == 0:
            continue
        q, k, v = W.trace_step_inputs(cfg, p.index, p.num_tokens)
        T = p.num_tokens
        g.q[:T].copy_(W.bf16_tensor(q, "cuda"))
        g.k_new[:T].copy_(W.bf16_tensor(k, "cuda"))
        g.v_new[:T].copy_(W.bf16_tensor(v, "cuda"))
        g.launch(p.slot_mapping, p.block_tables, p.seq_lens, p.query_start_loc, p.copy_pairs)
        if len(p.copy_pairs):
            oracle.copy_blocks(kc, vc, p.copy_pairs)
        oracle.reshape_and_cache(k, v, kc, vc, p.slot_mapping)
        ref = oracle.paged_attention(q, kc, vc, p.block_tables, p.seq_lens, p.query_start_loc,
                                     1.0 / np.sqrt(cfg.head_dim))
        got = to_f64(g.out[:T])
        mx, rel = attn_errors(got, ref)
        assert mx <= MAX_ABS and rel <= REL_L2, f"step {p.index}: max {mx:.3e} rel {rel:.3e}"
        checked += 1
    ops.check_device_errors()
    assert checked > 20
    assert np.array_equal(W.bits_of(dk), kc), "K cache differs from the oracle"
    assert np.array_equal(W.bits_of(dv), vc), "V cache differs from the oracle"
    g.close()


def test_graph_matches_eager_calls_bit_for_bit_on_a_decode_step():
    """A decode-only step padded into a graph built for larger steps gives the
    same bits as the eager calls with the step's exact sizes."""
    b = W.decode_batch(num_seqs=24, seed=7)
    d = W.to_device(b)
    kc0, vc0 = d.k_cache.clone(), d.v_cache.clone()
    ops.reshape_and_cache(d.k_new, d.v_new, d.k_cache, d.v_cache, d.slot_mapping)
    eager = ops.paged_attention(d.q, d.k_cache, d.v_cache, d.block_tables, d.seq_lens,
                                d.query_start_loc, b.scale, max_q_len=1,
                                max_seq_len=b.max_seq_len)
    g = ops.StepGraph(kc0, vc0, num_q_heads=b.num_q_heads, max_tokens=64, max_seqs=40,
                      max_blocks=b.block_tables.shape[1] + 3, max_pairs=4, max_q_len=1,
                      max_seq_len=b.max_seq_len, scale=b.scale)
    T = b.num_tokens
    g.q[:T].copy_(d.q)
    g.k_new[:T].copy_(d.k_new)
    g.v_new[:T].copy_(d.v_new)
    g.launch(b.slot_mapping, b.block_tables, b.seq_lens, b.query_start_loc)
    ops.check_device_errors()
    assert torch.equal(g.out[:T].view(torch.int16), eager.view(torch.int16))
    assert torch.equal(kc0.view(torch.int16), d.k_cache.view(torch.int16))
    g.close()


def test_padded_copy_pairs_are_skipped():
    rng = np.random.default_rng(2)
    kc = rng.integers(0, 65536, size=(12, 16, 2, 64), dtype=np.uint16)
    vc = rng.integers(0, 65536, size=(12, 16, 2, 64), dtype=np.uint16)
    dk, dv = W.bf16_tensor(kc, "cuda"), W.bf16_tensor(vc, "cuda")
    pairs = np.array([[3, 7], [-1, -1], [5, 9], [-1, -1]], np.int32)
    ops.copy_blocks(dk, dv, W.int32_tensor(pairs, "cuda"))
    ops.check_device_errors()  # padding flags nothing
    oracle.copy_blocks(kc, vc, pairs[pairs[:, 0] >= 0])
    assert np.array_equal(W.bits_of(dk), kc) and np.array_equal(W.bits_of(dv), vc)


def test_host_io_graph_round_trip():
    """host_io: the step's q / k_new / v_new go in with the integer inputs in
    one pinned region, out comes back into pinned memory; the bits equal the
    eager calls'."""
    b = W.decode_batch(num_seqs=20, seed=9)
    d = W.to_device(b)
    kc0, vc0 = d.k_cache.clone(), d.v_cache.clone()
    ops.reshape_and_cache(d.k_new, d.v_new, d.k_cache, d.v_cache, d.slot_mapping)
    eager = ops.paged_attention(d.q, d.k_cache, d.v_cache, d.block_tables, d.seq_lens,
                                d.query_start_loc, b.scale, max_q_len=1,
                                max_seq_len=b.max_seq_len)
    g = ops.StepGraph(kc0, vc0, num_q_heads=b.num_q_heads, max_tokens=32, max_seqs=24,
                      max_blocks=b.block_tables.shape[1], max_pairs=0, max_q_len=1,
                      max_seq_len=b.max_seq_len, scale=b.scale, host_io=True)
    T = b.num_tokens
    for _ in range(3):  # both pinned buffers, then the first again
        qh, kh, vh = g.inputs_host()
        qh[:T] = W.bf16_tensor(b.q, "cpu")
        kh[:T] = W.bf16_tensor(b.k_new, "cpu")
        vh[:T] = W.bf16_tensor(b.v_new, "cpu")
        g.launch(b.slot_mapping, b.block_tables, b.seq_lens, b.query_start_loc)
        g.wait_output()
        got = g.output_host()[:T]
        assert torch.equal(got.view(torch.int16), eager.cpu().view(torch.int16))
    ops.check_device_errors()
    assert torch.equal(kc0.view(torch.int16), d.k_cache.view(torch.int16))
    g.close()


def test_host_io_overlapped_launches_keep_every_output():
    """Back-to-back host_io launches (inputs copied in on one side stream,
    outputs out on another, two buffers in turn): each launch's output, read
    after wait_output, is its own step's, and relaunch repeats a step."""
    steps = []
    for seed in range(4):
        steps.append(W.make_batch("io", [200 + 37 * seed, 90], [1, 1], num_q_heads=8,
                                  num_kv_heads=2, head_dim=64, block_size=16, num_blocks=40,
                                  seed=seed, poison=False))
    kc = torch.zeros(40, 16, 2, 64, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    g = ops.StepGraph(kc, vc, num_q_heads=8, max_tokens=4, max_seqs=4, max_blocks=20,
                      max_pairs=0, max_q_len=1, max_seq_len=320, scale=0.125, host_io=True)
    outs = []
    for b in steps:
        # each step brings its own cache contents: copy them in first
        kc.copy_(W.bf16_tensor(b.k_cache, "cuda"))
        vc.copy_(W.bf16_tensor(b.v_cache, "cuda"))
        qh, kh, vh = g.inputs_host()
        qh[:2] = W.bf16_tensor(b.q, "cpu")
        kh[:2] = W.bf16_tensor(b.k_new, "cpu")
        vh[:2] = W.bf16_tensor(b.v_new, "cpu")
        g.launch(b.slot_mapping, b.block_tables, b.seq_lens, b.query_start_loc)
        g.wait_output()
        outs.append(g.output_host()[:2].clone())
        _, _, ref = run_oracle_step(b)
        assert_attn_close(to_f64(outs[-1]), ref, "host_io step")
    g.relaunch()  # buffer 0 again: the third step's inputs, over the last step's cache
    g.wait_output()
    assert g.output_host().shape[0] == 4
    ops.check_device_errors()
    g.close()
