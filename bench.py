"""Benchmark: attention over a paged KV cache on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload decode_batch|long_decode|mixed_step|tiny_decode]

One step is one pass of the whole hot path over one batch of the workload:
the slot scatter of the step's new K/V, then paged attention over every
request (split-KV decode kernel + merge, and the tensor-core prefill kernel
for chunked-prefill rows), through the C ABI.  Inputs are synthetic and
seeded; the KV cache (hundreds of MB to GB) is far larger than the 129 MB L2,
so no explicit L2 flush is done between steps.  The kernel durations behind
the roofline figures come from CUDA graphs of back-to-back calls (no idle
time from the host's per-call work); where a call's inputs fit in L2 (the
prefill chunk alone, the tiny decode), a 256 MB write evicts L2 before each
call and the time of those writes alone is subtracted.

Prints one JSON line (rank 0).  With N > 1 (torchrun, one process per GPU)
every rank runs its own replica of the batch and `value` is the bytes all
ranks processed divided by the slowest rank's time (weak scaling).

--impl reference times the fp64 CPU oracle on a bounded sample of the same
workload (there is no other implementation of this method to run).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged-attn decode HBM GB/s (% of peak); mixed-batch tokens/s per step"


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            j = json.load(f)
        return {"hbm_gbs": float(j["hbm_gbs"]), "bf16_tflops": float(j["bf16_tflops"]),
                "bf16_tflops_sustained": float(j.get("bf16_tflops_sustained", j["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self._t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self._t:
            self._t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def _profiled_traffic(profile: str, sources, workload: str, want_workload: str):
    """DRAM bytes per launch recorded by an ncu capture under profiles/, or
    None when the workload differs or the kernel sources changed since."""
    import hashlib
    if workload != want_workload:
        return None
    path = os.path.join(ROOT, "profiles", profile)
    if not os.path.exists(path):
        return None
    h = hashlib.sha256()
    for src in sources:
        with open(os.path.join(ROOT, "paged_kv_cache_174_gb300", "csrc", src), "rb") as f:
            h.update(f.read())
    fields = {}
    with open(path) as f:
        for line in f:
            if ":" in line and line.strip().split(":")[0] in (
                    "kernel_source_sha256_16", "traffic_bytes_per_launch"):
                k, v = line.strip().split(":", 1)
                fields[k] = v.strip()
    if fields.get("kernel_source_sha256_16") != h.hexdigest()[:16]:
        return None
    try:
        return int(fields["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(values, dist, device):
    """Element-wise max of a list of floats over all ranks (identity for one
    process): the slowest rank's time is the job's time."""
    import torch
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return list(values)
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def _config(b, world):
    """The workload as the JSON line names it (both arms use the same)."""
    from paged_kv_cache_174_gb300 import workloads as W
    return {"workload": b.name, "description": W.WORKLOADS[b.name].description,
            "num_seqs": b.num_seqs, "num_tokens": b.num_tokens,
            "kv_tokens": int(b.seq_lens.sum()), "block_size": b.block_size,
            "algorithmic_bytes_per_step": W.algorithmic_bytes(b)["total"],
            "l2": "inputs larger than L2 (KV read per step >> 129 MB); no flush",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


def _make(workload: str, rank: int):
    from paged_kv_cache_174_gb300 import workloads as W
    b = W.by_name(workload, poison=False)
    return b


def ops_splits(b) -> int:
    from paged_kv_cache_174_gb300 import ops
    return ops.prefill_splits(b.num_tokens, b.num_q_heads, b.num_kv_heads, b.head_dim,
                              b.max_q_len, b.max_seq_len)


def _launch_count(b) -> int:
    n = 1 if b.num_tokens else 0        # scatter
    n += 2                              # split-KV decode + merge
    if b.max_q_len >= 2:
        n += 1                          # prefill
        if ops_splits(b) > 1:
            n += 1                      # merge of the prefill key pieces
    if b.copy_pairs.size:
        n += 1
    return n


def _graph_launch_count(b) -> int:
    """Kernels one ops.StepGraph launch runs: a decode-only step does its
    slot scatter inside the decode kernel (pa_decode_step), a step with
    prefill rows launches the scatter kernel first."""
    return _launch_count(b) - (1 if b.num_tokens and b.max_q_len <= 1 else 0)


L2_FLUSH_BYTES = 256 << 20  # a write of this many bytes evicts the 129 MB L2
_FLUSH = {}


def _flush_buffer(dev):
    import torch
    if dev not in _FLUSH:
        _FLUSH[dev] = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    return _FLUSH[dev]


def _flush_if_small(b, dev):
    """The flush buffer when batch b's attention inputs would stay in L2
    between calls (the tiny decode), else None (they are larger than L2)."""
    from paged_kv_cache_174_gb300 import workloads as W
    if W.algorithmic_bytes(b)["attention"] < L2_FLUSH_BYTES:
        return _flush_buffer(dev)
    return None


def _device_ms(call, steps, warmup, stream, flush_buf=None, reps=5):
    """Device milliseconds per call of `call`: CUDA events on `stream` around
    the replay of a CUDA graph holding `steps` back-to-back calls (median of
    `reps` replays), so the host's per-call work (Python, argument checks)
    leaves no idle GPU time inside the measurement.  With flush_buf (larger
    than L2), every call in the graph follows a write of the whole buffer and
    the replay time of a graph of those writes alone is subtracted: each call
    then starts with its inputs out of L2."""
    import torch

    for _ in range(warmup):
        call()
    torch.cuda.synchronize()

    def replay_ms(body):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(steps):
                body()
        times = []
        with torch.cuda.stream(stream):
            g.replay()
            for _ in range(reps):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                g.replay()
                e1.record(stream)
                torch.cuda.synchronize()
                times.append(e0.elapsed_time(e1))
        del g
        return statistics.median(times)

    if flush_buf is None:
        return replay_ms(call) / steps

    def flush():
        flush_buf.fill_(1)

    def flush_then_call():
        flush()
        call()

    return (replay_ms(flush_then_call) - replay_ms(flush)) / steps


def _time_steps(b, d, ws, out, steps, warmup, stream, ops, flush_buf=None):
    """Device-resident steps (scatter + attention) launched one call at a time
    from Python; returns per-step milliseconds, the mean of CUDA events around
    each attention call in that loop (host gaps included), and the attention
    call's device time from back-to-back launches (`_device_ms`, the roofline
    figure)."""
    import torch

    def attention():
        ops.paged_attention(d.q, d.k_cache, d.v_cache, d.block_tables, d.seq_lens,
                            d.query_start_loc, b.scale, max_q_len=b.max_q_len,
                            max_seq_len=b.max_seq_len, out=out, workspace=ws)

    def step(ev=None):
        if d.copy_pairs.numel():
            ops.copy_blocks(d.k_cache, d.v_cache, d.copy_pairs)
        ops.reshape_and_cache(d.k_new, d.v_new, d.k_cache, d.v_cache, d.slot_mapping)
        if ev is not None:
            ev[0].record(stream)
        attention()
        if ev is not None:
            ev[1].record(stream)

    for _ in range(warmup):
        step()
    ops.check_device_errors()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(steps):
        step(evs[i])
    t1.record(stream)
    torch.cuda.synchronize()
    ops.check_device_errors()
    dev_ms = _device_ms(attention, steps, warmup, stream, flush_buf)
    ops.check_device_errors()
    return (t0.elapsed_time(t1) / steps,
            statistics.mean(e0.elapsed_time(e1) for e0, e1 in evs), dev_ms)


def _time_graph_steps(b, d, steps, warmup, stream, ops):
    """The same step (scatter + attention) as one launch of the step captured
    as a CUDA graph (ops.StepGraph): the step's inputs are copied to the
    device once, before the timed region, and every timed launch uses them
    where they are (nothing is copied).  Returns (ms per step, device out)."""
    import torch
    from paged_kv_cache_174_gb300 import workloads as W
    g = ops.StepGraph(d.k_cache, d.v_cache, num_q_heads=b.num_q_heads,
                      max_tokens=b.num_tokens, max_seqs=b.num_seqs,
                      max_blocks=b.block_tables.shape[1], max_pairs=len(b.copy_pairs),
                      max_q_len=b.max_q_len, max_seq_len=b.max_seq_len, scale=b.scale,
                      host_io=True)
    host_qkv = [W.bf16_tensor(x, "cpu") for x in (b.q, b.k_new, b.v_new)]
    for _ in range(2):  # both buffers' inputs onto the device
        qh, kh, vh = g.inputs_host()
        qh.copy_(host_qkv[0])
        kh.copy_(host_qkv[1])
        vh.copy_(host_qkv[2])
        g.launch(b.slot_mapping, b.block_tables, b.seq_lens, b.query_start_loc, b.copy_pairs,
                 stream=stream, copy_out=False)
    for _ in range(warmup):
        g.relaunch(stream=stream, copy_in=False, copy_out=False)
    torch.cuda.synchronize()
    ops.check_device_errors()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(steps):
        g.relaunch(stream=stream, copy_in=False, copy_out=False)
    t1.record(stream)
    torch.cuda.synchronize()
    ops.check_device_errors()
    out = g.output().clone()
    g.close()
    return t0.elapsed_time(t1) / steps, out


def _prefill_only(b, d):
    """The requests of b with q_len >= 2, as their own batch (same device
    K/V cache and q rows)."""
    import torch
    from paged_kv_cache_174_gb300 import workloads as W
    idx = [s for s in range(b.num_seqs) if b.q_lens[s] >= 2]
    if not idx:
        return None
    rows = np.concatenate([np.arange(b.query_start_loc[s], b.query_start_loc[s + 1])
                           for s in idx])
    ql = b.q_lens[idx]
    qsl = np.zeros(len(idx) + 1, np.int32)
    qsl[1:] = np.cumsum(ql)
    sub = W.PagedBatch(name=b.name + "/prefill", q=b.q[rows], k_new=b.k_new[rows],
                       v_new=b.v_new[rows], k_cache=b.k_cache[:1], v_cache=b.v_cache[:1],
                       block_tables=b.block_tables[idx], seq_lens=b.seq_lens[idx],
                       query_start_loc=qsl, slot_mapping=b.slot_mapping[rows], scale=b.scale,
                       block_size=b.block_size, seed=b.seed)
    dev = d.q.device
    rows_t = torch.from_numpy(rows).to(dev)
    return sub, dict(q=d.q.index_select(0, rows_t).contiguous(),
                     block_tables=W.int32_tensor(sub.block_tables, dev),
                     seq_lens=W.int32_tensor(sub.seq_lens, dev),
                     query_start_loc=W.int32_tensor(qsl, dev))


def _time_prefill(b, d, steps, warmup, stream, ops, flush_buf):
    """The batch's prefill rows alone (one prefill launch, plus the key-split
    merge when the plan splits): device time per call with L2 flushed before
    every call (`_device_ms`)."""
    import torch
    from paged_kv_cache_174_gb300 import workloads as W
    po = _prefill_only(b, d)
    if po is None:
        return None
    sub, t = po
    out = torch.empty_like(t["q"])
    ws = ops.alloc_workspace(sub.num_seqs, sub.num_tokens, sub.num_q_heads, sub.num_kv_heads,
                             sub.head_dim, sub.max_q_len, sub.max_seq_len, d.q.device)

    def call():
        # prefill rows only: min_q_len >= 2 lets the call skip the decode launch
        ops.paged_attention(t["q"], d.k_cache, d.v_cache, t["block_tables"], t["seq_lens"],
                            t["query_start_loc"], sub.scale, max_q_len=sub.max_q_len,
                            max_seq_len=sub.max_seq_len, out=out, workspace=ws,
                            min_q_len=int(sub.q_lens.min()))

    ms = _device_ms(call, steps, warmup, stream, flush_buf)
    ops.check_device_errors()
    flops = W.causal_flops(sub)
    return {"ms": round(ms, 5), "flops": flops, "tflops": round(flops / (ms * 1e-3) / 1e12, 2),
            "tokens": sub.num_tokens}


def _mixed_bounds(b, peaks):
    """Per-kernel roofline times (ms) of one step of batch b: the scatter and
    the decode rows against the HBM peak, the chunk's causal FLOPs against
    the bf16 tensor peak (burst: the step is short)."""
    from paged_kv_cache_174_gb300 import workloads as W
    kv_row = b.num_kv_heads * b.head_dim * 2
    dec = b.q_lens == 1
    dec_bytes = int(b.seq_lens[dec].astype(np.int64).sum()) * 2 * kv_row
    dec_bytes += 2 * int(dec.sum()) * b.num_q_heads * b.head_dim * 2
    dec_bytes += sum(-(-int(L) // b.block_size) for L in b.seq_lens[dec]) * 4
    flops = W.causal_flops(b)
    scatter = W.algorithmic_bytes(b)["scatter"]
    t_dec = dec_bytes / (peaks["hbm_gbs"] * 1e9) * 1e3
    t_pre = flops / (peaks["bf16_tflops"] * 1e12) * 1e3
    t_sc = scatter / (peaks["hbm_gbs"] * 1e9) * 1e3
    return {"decode_bytes": dec_bytes, "chunk_flops": flops, "scatter_bytes": scatter,
            "decode_bound_ms": round(t_dec, 5), "chunk_bound_ms": round(t_pre, 5),
            "scatter_bound_ms": round(t_sc, 5), "sum_bound_ms": round(t_dec + t_pre + t_sc, 5)}


def _run_trace(dev, stream, ops, warmup):
    """The continuous-batching trace: every step's CoW copies, scatter and
    attention timed with CUDA events (schedule precomputed on the host,
    inputs generated on the device before each step's events)."""
    import torch
    from paged_kv_cache_174_gb300 import workloads as W
    from paged_kv_cache_174_gb300.host import CONTINUOUS_BATCHING_TRACE, ContinuousBatchingTrace

    cfg = CONTINUOUS_BATCHING_TRACE
    tr = ContinuousBatchingTrace(cfg)
    plans = [tr.step() for _ in range(cfg.steps)]
    shape = (cfg.num_blocks, cfg.block_size, cfg.num_kv_heads, cfg.head_dim)
    gen = torch.Generator(device=dev)

    def fresh_cache():
        kc = torch.zeros(shape, dtype=torch.bfloat16, device=dev)
        vc = torch.zeros(shape, dtype=torch.bfloat16, device=dev)
        pos = torch.arange(cfg.prefix, device=dev)
        blocks = torch.tensor(tr.prefix_blocks, device=dev)
        slots = blocks[pos // cfg.block_size] * cfg.block_size + pos % cfg.block_size
        gen.manual_seed(cfg.seed)
        kc.view(-1, cfg.num_kv_heads, cfg.head_dim)[slots] = torch.randn(
            cfg.prefix, cfg.num_kv_heads, cfg.head_dim, generator=gen, device=dev).bfloat16()
        vc.view(-1, cfg.num_kv_heads, cfg.head_dim)[slots] = torch.randn(
            cfg.prefix, cfg.num_kv_heads, cfg.head_dim, generator=gen, device=dev).bfloat16()
        return kc, vc

    S = max(len(pl.rids) for pl in plans)
    T = max(pl.num_tokens for pl in plans)
    ws = ops.alloc_workspace(S, T, cfg.num_q_heads, cfg.num_kv_heads, cfg.head_dim,
                             max(pl.max_q_len for pl in plans),
                             max(pl.max_seq_len for pl in plans), dev)
    scale = 1.0 / (cfg.head_dim ** 0.5)

    def run(kc, vc, plan_list, record):
        times = []
        for pl in plan_list:
            if pl.num_tokens == 0:
                continue
            meta = {k: W.int32_tensor(getattr(pl, k), dev) for k in
                    ("copy_pairs", "slot_mapping", "block_tables", "seq_lens", "query_start_loc")}
            q = torch.randn(pl.num_tokens, cfg.num_q_heads, cfg.head_dim, generator=gen,
                            device=dev).bfloat16()
            k = torch.randn(pl.num_tokens, cfg.num_kv_heads, cfg.head_dim, generator=gen,
                            device=dev).bfloat16()
            v = torch.randn(pl.num_tokens, cfg.num_kv_heads, cfg.head_dim, generator=gen,
                            device=dev).bfloat16()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            if len(pl.copy_pairs):
                ops.copy_blocks(kc, vc, meta["copy_pairs"])
            ops.reshape_and_cache(k, v, kc, vc, meta["slot_mapping"])
            ops.paged_attention(q, kc, vc, meta["block_tables"], meta["seq_lens"],
                                meta["query_start_loc"], scale, max_q_len=pl.max_q_len,
                                max_seq_len=pl.max_seq_len, workspace=ws)
            e1.record(stream)
            if record:
                times.append((pl, e0, e1))
        torch.cuda.synchronize()
        ops.check_device_errors()
        return [(pl, a.elapsed_time(b)) for pl, a, b in times]

    kc, vc = fresh_cache()
    run(kc, vc, plans[:warmup], False)
    kc, vc = fresh_cache()
    res = run(kc, vc, plans, True)
    ms = np.array([t for _, t in res])
    toks = sum(pl.num_tokens for pl, _ in res)
    launches = sum(3 + (pl.max_q_len >= 2) + (len(pl.copy_pairs) > 0) for pl, _ in res)
    del kc, vc

    # the same steps, each one launch of the step captured as a CUDA graph at
    # fixed maxima (metadata copied from pinned host memory inside the graph)
    def run_graph(g, plan_list, record):
        times = []
        for pl in plan_list:
            if pl.num_tokens == 0:
                continue
            T = pl.num_tokens
            g.q[:T] = torch.randn(T, cfg.num_q_heads, cfg.head_dim, generator=gen,
                                  device=dev).bfloat16()
            g.k_new[:T] = torch.randn(T, cfg.num_kv_heads, cfg.head_dim, generator=gen,
                                      device=dev).bfloat16()
            g.v_new[:T] = torch.randn(T, cfg.num_kv_heads, cfg.head_dim, generator=gen,
                                      device=dev).bfloat16()
            g.stage(pl.slot_mapping, pl.block_tables, pl.seq_lens, pl.query_start_loc,
                    pl.copy_pairs)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.launch(stream=stream)
            e1.record(stream)
            if record:
                times.append((pl, e0, e1))
        torch.cuda.synchronize()
        ops.check_device_errors()
        return [(pl, a.elapsed_time(b)) for pl, a, b in times]

    def make_graph(kc, vc):
        return ops.StepGraph(kc, vc, num_q_heads=cfg.num_q_heads, max_tokens=cfg.budget,
                             max_seqs=cfg.max_num_seqs,
                             max_blocks=max(pl.block_tables.shape[1] for pl in plans),
                             max_pairs=max(len(pl.copy_pairs) for pl in plans),
                             max_q_len=cfg.chunk,
                             max_seq_len=max(pl.max_seq_len for pl in plans), scale=scale)

    kc, vc = fresh_cache()
    g = make_graph(kc, vc)
    run_graph(g, plans[:warmup], False)
    g.close()
    kc, vc = fresh_cache()
    g = make_graph(kc, vc)
    gres = run_graph(g, plans, True)
    g.close()
    gms = np.array([t for _, t in gres])
    graph = {"tokens_per_s": round(toks / (gms.sum() * 1e-3), 1),
             "gpu_ms_total": round(float(gms.sum()), 3),
             "step_ms_p50": round(float(np.percentile(gms, 50)), 5),
             "step_ms_p99": round(float(np.percentile(gms, 99)), 5),
             "graph_launches": len(gres),
             # every replay runs the kernels captured at the maxima: the CoW
             # copy, the scatter, the prefill (+ its key-piece merge), decode
             # + merge
             "gpu_launches": len(gres) * (5 + (ops.prefill_splits(
                 cfg.budget, cfg.num_q_heads, cfg.num_kv_heads, cfg.head_dim, cfg.chunk,
                 max(pl.max_seq_len for pl in plans)) > 1)),
             "maxima": {"tokens": cfg.budget, "seqs": cfg.max_num_seqs, "q_len": cfg.chunk}}
    return {"workload": "continuous-batching trace", "steps": len(res),
            "description": "200 steps, Poisson 8 arrivals/step, lognormal prompts (median 600, "
                           "sigma 1, clamp 64-8192), geometric outputs (mean 200), 500-token "
                           "shared prefix with copy-on-write, 512-token chunks, 2048-token "
                           "budget, max 256 running, 40000-block pool, 32/8 heads, d 128",
            "tokens": int(toks), "tokens_per_s": round(toks / (ms.sum() * 1e-3), 1),
            "gpu_ms_total": round(float(ms.sum()), 3),
            "step_ms_p50": round(float(np.percentile(ms, 50)), 5),
            "step_ms_p99": round(float(np.percentile(ms, 99)), 5),
            "cow_copies": int(tr.total_copies), "finished_requests": len(tr.finished),
            "mean_block_utilisation": round(tr.summary()["mean_block_utilisation"], 4),
            "mean_waste_fraction": round(tr.summary()["mean_waste_fraction"], 4),
            "gpu_launches": int(launches), "step_graph": graph}


def _fp8(args, dev, stream, ops, peaks, bf16_attn_ms):
    """The decode batch over the 8-bit cache (E4M3 codes + one fp32 scale per
    cached row): the context is quantised once on the device, then each step
    quantises the new tokens and runs decode attention, timed like the main
    line.  Then the mixed chunked-prefill step over the 8-bit cache, and its
    chunk alone."""
    import torch
    from paged_kv_cache_174_gb300 import workloads as W

    b = W.decode_batch(poison=False)
    nb, bs, nkv, d = b.k_cache.shape
    k8, v8 = ops.empty_fp8_cache(nb, bs, nkv, d, dev)
    slots = W.context_slots(b)
    rows = b.k_cache.reshape(-1, nkv, d)
    ops.reshape_and_cache_fp8(W.bf16_tensor(rows[slots], dev),
                              W.bf16_tensor(b.v_cache.reshape(-1, nkv, d)[slots], dev),
                              k8, v8, W.int32_tensor(slots, dev))
    q = W.bf16_tensor(b.q, dev)
    kn, vn = W.bf16_tensor(b.k_new, dev), W.bf16_tensor(b.v_new, dev)
    meta = {k: W.int32_tensor(getattr(b, k), dev)
            for k in ("slot_mapping", "block_tables", "seq_lens", "query_start_loc")}
    ws = ops.alloc_workspace(b.num_seqs, b.num_tokens, b.num_q_heads, nkv, d, 1,
                             b.max_seq_len, dev)
    out = torch.empty_like(q)

    def attention():
        ops.paged_attention_fp8(q, k8, v8, meta["block_tables"], meta["seq_lens"],
                                meta["query_start_loc"], b.scale, max_q_len=1,
                                max_seq_len=b.max_seq_len, out=out, workspace=ws)

    def step(ev=None):
        ops.reshape_and_cache_fp8(kn, vn, k8, v8, meta["slot_mapping"])
        if ev is not None:
            ev[0].record(stream)
        attention()
        if ev is not None:
            ev[1].record(stream)

    for _ in range(args.warmup):
        step()
    ops.check_device_errors()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(args.steps):
        step(evs[i])
    t1.record(stream)
    torch.cuda.synchronize()
    ops.check_device_errors()
    ms = t0.elapsed_time(t1) / args.steps
    loop_attn_ms = statistics.mean(a.elapsed_time(c) for a, c in evs)
    # the roofline's duration: back-to-back launches (inputs larger than L2)
    attn_ms = _device_ms(attention, args.steps, args.warmup, stream)
    ops.check_device_errors()
    alg = W.algorithmic_bytes_fp8(b)
    gbs = alg["attention"] / (attn_ms * 1e-3) / 1e9
    mixed = None if args.no_mixed else _fp8_mixed(args, dev, stream, ops, peaks)
    return {"workload": "decode_batch, 8-bit cache (E4M3 codes + fp32 scale per row)",
            "ms_per_step": round(ms, 5), "attention_ms": round(attn_ms, 5),
            "attention_ms_host_loop": round(loop_attn_ms, 5),
            "tokens_per_s": round(b.num_tokens / (ms * 1e-3), 1),
            "kv_tokens_per_s": round(int(b.seq_lens.sum()) / (attn_ms * 1e-3), 1),
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4),
                         "algorithmic_bytes_per_launch": alg["attention"],
                         "traffic": _profiled_traffic(
                             "decode_kernel_fp8_decode_batch.md",
                             ["pa_decode_kernel.cuh", "pa_decode_fp8.cu", "pa_common.cuh"],
                             "decode_batch", "decode_batch")},
            "attention_speedup_vs_bf16": round(bf16_attn_ms / attn_ms, 3),
            "mixed_step": mixed}


def _fp8_mixed(args, dev, stream, ops, peaks):
    """The mixed step (128 decode rows + a 512-token chunk at offset 3584)
    over the 8-bit cache: each step quantises the 640 new rows and runs
    attention over codes and scales; then the chunk's rows alone (its call
    also launches the empty decode grid: the 8-bit entry point takes no
    min_q_len)."""
    import types
    import torch
    from paged_kv_cache_174_gb300 import workloads as W

    b = W.mixed_step(poison=False)
    nb, bs, nkv, d = b.k_cache.shape
    k8, v8 = ops.empty_fp8_cache(nb, bs, nkv, d, dev)
    slots = W.context_slots(b)
    rows = b.k_cache.reshape(-1, nkv, d)
    ops.reshape_and_cache_fp8(W.bf16_tensor(rows[slots], dev),
                              W.bf16_tensor(b.v_cache.reshape(-1, nkv, d)[slots], dev),
                              k8, v8, W.int32_tensor(slots, dev))
    q = W.bf16_tensor(b.q, dev)
    kn, vn = W.bf16_tensor(b.k_new, dev), W.bf16_tensor(b.v_new, dev)
    meta = {k: W.int32_tensor(getattr(b, k), dev)
            for k in ("slot_mapping", "block_tables", "seq_lens", "query_start_loc")}
    ws = ops.alloc_workspace(b.num_seqs, b.num_tokens, b.num_q_heads, nkv, d, b.max_q_len,
                             b.max_seq_len, dev)
    out = torch.empty_like(q)
    sub, t = _prefill_only(b, types.SimpleNamespace(q=q))
    sout = torch.empty_like(t["q"])

    def step():
        ops.reshape_and_cache_fp8(kn, vn, k8, v8, meta["slot_mapping"])
        ops.paged_attention_fp8(q, k8, v8, meta["block_tables"], meta["seq_lens"],
                                meta["query_start_loc"], b.scale, max_q_len=b.max_q_len,
                                max_seq_len=b.max_seq_len, out=out, workspace=ws)

    def chunk():
        ops.paged_attention_fp8(t["q"], k8, v8, t["block_tables"], t["seq_lens"],
                                t["query_start_loc"], sub.scale, max_q_len=sub.max_q_len,
                                max_seq_len=sub.max_seq_len, out=sout, workspace=ws)

    # device time per call (`_device_ms`): the step's inputs are larger than
    # L2; the chunk's K/V are not, so L2 is flushed before each chunk call
    res = {"step": _device_ms(step, args.steps, args.warmup, stream),
           "chunk": _device_ms(chunk, args.steps, args.warmup, stream, _flush_buffer(dev))}
    ops.check_device_errors()
    flops = W.causal_flops(sub)
    tflops = flops / (res["chunk"] * 1e-3) / 1e12
    return {"workload": "mixed_step over the 8-bit cache",
            "ms_per_step": round(res["step"], 5),
            "tokens_per_s": round(b.num_tokens / (res["step"] * 1e-3), 1),
            "chunk_ms": round(res["chunk"], 5),
            "chunk_tflops": round(tflops, 2),
            "chunk_frac_of_bf16_peak": round(tflops / peaks["bf16_tflops"], 4)}


def _other_decodes(args, dev, stream, ops, peaks, host_batches=None):
    """The tiny decode (latency only), the long-context decode (8 x 32768
    tokens, HBM-bound) and the decode batch at group 8 (64 q / 8 kv heads,
    the same cache), timed like the main line."""
    import torch
    from paged_kv_cache_174_gb300 import workloads as W
    res = {}
    for name in ("tiny_decode", "long_decode", "group8_decode"):
        if name == "group8_decode":
            b = W.decode_batch(poison=False, num_q_heads=64)
        else:
            b = W.by_name(name, poison=False)
            if host_batches is not None:
                host_batches[name] = b
        d = W.to_device(b, dev)
        ws = ops.alloc_workspace(b.num_seqs, b.num_tokens, b.num_q_heads, b.num_kv_heads,
                                 b.head_dim, b.max_q_len, b.max_seq_len, dev)
        out = torch.empty_like(d.q)
        ms, loop_ms, attn_ms = _time_steps(b, d, ws, out, args.steps, args.warmup, stream, ops,
                                           _flush_if_small(b, dev))
        # the same step as one graph launch (decode-only: the decode kernel
        # does the scatter), which shows the device latency of a small step
        # without the host's per-call overhead
        graph_ms, _ = _time_graph_steps(b, d, args.steps, args.warmup, stream, ops)
        alg = W.algorithmic_bytes(b)
        gbs = alg["attention"] / (attn_ms * 1e-3) / 1e9
        desc = (W.WORKLOADS[name].description if name in W.WORKLOADS else
                "decode batch of 64 requests (lens U[128, 4096]) at 64 q / 8 kv heads, d 128")
        res[name] = {"description": desc,
                     "ms_per_step": round(ms, 5), "attention_ms": round(attn_ms, 5),
                     "attention_ms_host_loop": round(loop_ms, 5),
                     "graph_ms_per_step": round(graph_ms, 5),
                     "attention_GB_per_s": round(gbs, 1),
                     "attention_frac_of_hbm": round(gbs / peaks["hbm_gbs"], 4)}
        del d, ws, out
    return res


def _block32(args, dev, stream, ops, peaks):
    """32-token blocks against 16: the decode batch and the mixed step with the
    same token slots in half as many blocks, timed like the main line, and
    the trace's fragmentation at both block sizes (host-side counters)."""
    import dataclasses

    import torch
    from paged_kv_cache_174_gb300 import workloads as W
    from paged_kv_cache_174_gb300.host import CONTINUOUS_BATCHING_TRACE, ContinuousBatchingTrace

    res = {}
    for name, make in (("decode_batch", W.decode_batch), ("mixed_step", W.mixed_step)):
        b = make(poison=False, block_size=32)
        d = W.to_device(b, dev)
        ws = ops.alloc_workspace(b.num_seqs, b.num_tokens, b.num_q_heads, b.num_kv_heads,
                                 b.head_dim, b.max_q_len, b.max_seq_len, dev)
        out = torch.empty_like(d.q)
        ms, _, attn_ms = _time_steps(b, d, ws, out, args.steps, args.warmup, stream, ops)
        alg = W.algorithmic_bytes(b)
        res[name] = {"ms_per_step": round(ms, 5), "attention_ms": round(attn_ms, 5),
                     "GB_per_s": round(alg["total"] / (ms * 1e-3) / 1e9, 1),
                     "attention_frac_of_hbm": round(
                         alg["attention"] / (attn_ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                     "tokens_per_s": round(b.num_tokens / (ms * 1e-3), 1)}
        del d, ws, out
    frag = {}
    for bs in (16, 32):
        cfg = dataclasses.replace(CONTINUOUS_BATCHING_TRACE, block_size=bs,
                                  num_blocks=CONTINUOUS_BATCHING_TRACE.num_blocks * 16 // bs)
        tr = ContinuousBatchingTrace(cfg)
        for _ in range(cfg.steps):
            tr.step()
        sm = tr.summary()
        frag[str(bs)] = {"mean_block_utilisation": round(sm["mean_block_utilisation"], 4),
                         "mean_waste_fraction": round(sm["mean_waste_fraction"], 4),
                         "cow_copies": sm["copies"]}
    res["trace_fragmentation"] = frag
    return res


def _summary(line):
    """The headline numbers again, compact, last in the line."""
    out = {"decode_batch_GBps": line.get("value"),
           "decode_attention_frac_hbm": _dig(line, ("roofline", "frac")),
           "e2e_GBps": _dig(line, ("e2e", "value")),
           "mixed_graph_tokens_per_s": _dig(line, ("mixed_batch", "graph_tokens_per_s")),
           "mixed_roofline_frac": _dig(line, ("mixed_batch", "roofline", "frac")),
           "prefill_frac_bf16": _dig(line, ("roofline_prefill", "frac")),
           "prefill_TFLOPs": _dig(line, ("roofline_prefill", "achieved")),
           "trace_graph_tokens_per_s": _dig(line, ("trace", "step_graph", "tokens_per_s")),
           "fp8_decode_frac_hbm": _dig(line, ("fp8_cache", "roofline", "frac")),
           "fp8_mixed_tokens_per_s": _dig(line, ("fp8_cache", "mixed_step", "tokens_per_s")),
           "fp8_chunk_frac_bf16": _dig(line, ("fp8_cache", "mixed_step",
                                              "chunk_frac_of_bf16_peak")),
           "long_decode_frac_hbm": _dig(line, ("other_decodes", "long_decode",
                                               "attention_frac_of_hbm")),
           "group8_decode_frac_hbm": _dig(line, ("other_decodes", "group8_decode",
                                                 "attention_frac_of_hbm"))}
    cb = line.get("cpu_baselines")
    if cb:
        out["oracle_all_cores"] = {k: [v["value"], v["unit"]] for k, v in cb.items()}
        out["oracle_one_core"] = {k: v["one_core_value"] for k, v in cb.items()}
        out["oracle_cores"] = next(iter(cb.values()))["cores"]
    return out


def _dig(d, keys):
    for k in keys:
        if not isinstance(d, dict) or k not in d:
            return None
        d = d[k]
    return d


def run_ours(args):
    import torch
    import torch.distributed as dist

    from paged_kv_cache_174_gb300 import ops
    from paged_kv_cache_174_gb300 import workloads as W

    world, rank, local = _dist()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peaks = _peaks()
    stream = torch.cuda.current_stream(dev)

    b = _make(args.workload, rank)
    host_batches = {b.name: b}  # the CPU baseline times the oracle on these
    d = W.to_device(b, dev)
    alg = W.algorithmic_bytes(b)
    step_bytes = alg["total"]
    ws = ops.alloc_workspace(b.num_seqs, b.num_tokens, b.num_q_heads, b.num_kv_heads,
                             b.head_dim, b.max_q_len, b.max_seq_len, dev)
    out = torch.empty_like(d.q)

    # ---- device-resident timed region (clocks sampled meanwhile)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    # separate launches per step; the attention call's device time (roofline)
    ms_sep, loop_attn_ms, attn_ms = _time_steps(b, d, ws, out, args.steps, args.warmup, stream,
                                                ops, _flush_if_small(b, dev))
    if world > 1:
        dist.barrier()
    # the step as one graph launch (the value)
    ms, gout = _time_graph_steps(b, d, args.steps, args.warmup, stream, ops)
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    if not torch.equal(gout[:b.num_tokens].view(torch.int16), out.view(torch.int16)):
        raise RuntimeError("the graph step's output differs from the separate launches'")
    ms, ms_sep, attn_ms, loop_attn_ms = reduce_max([ms, ms_sep, attn_ms, loop_attn_ms],
                                                   dist if world > 1 else None, dev)

    # ---- end to end through the public API from pinned host memory: the
    # step captured as a graph (ops.StepGraph, host_io) whose launch copies
    # the step's inputs (integer arrays and q / k_new / v_new, one pinned
    # region) to the device, runs scatter + attention and copies out back
    g = ops.StepGraph(d.k_cache, d.v_cache, num_q_heads=b.num_q_heads,
                      max_tokens=b.num_tokens, max_seqs=b.num_seqs,
                      max_blocks=b.block_tables.shape[1], max_pairs=len(b.copy_pairs),
                      max_q_len=b.max_q_len, max_seq_len=b.max_seq_len, scale=b.scale,
                      host_io=True)

    host_qkv = [W.bf16_tensor(x, "cpu") for x in (b.q, b.k_new, b.v_new)]
    for _ in range(2):  # the step's inputs into both pinned regions
        qh, kh, vh = g.inputs_host()
        qh.copy_(host_qkv[0])
        kh.copy_(host_qkv[1])
        vh.copy_(host_qkv[2])
        g.launch(b.slot_mapping, b.block_tables, b.seq_lens, b.query_start_loc, b.copy_pairs,
                 stream=stream)
    h2d, d2h = g.input_bytes, g.output_bytes
    for _ in range(args.warmup):
        g.relaunch(stream=stream)
    torch.cuda.synchronize()
    g.wait_output()
    ops.check_device_errors()
    got = g.output_host()[:b.num_tokens]
    if not torch.equal(got.view(torch.int16), out.cpu().view(torch.int16)):
        raise RuntimeError("the graph's host output differs from the device-resident step")
    if world > 1:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    g.fork(stream)
    for _ in range(args.steps):
        g.relaunch(stream=stream)
    g.join(stream)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / args.steps
    (e2e_ms,) = reduce_max([e2e_ms], dist if world > 1 else None, dev)
    g.close()
    if world > 1:
        dist.barrier()

    gbs = step_bytes * world / (ms * 1e-3) / 1e9
    attn_gbs = alg["attention"] / (attn_ms * 1e-3) / 1e9
    line = {
        "metric": METRIC,
        "value": round(gbs, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 5),
        "step_path": "ops.StepGraph: one graph launch per step (slot scatter, attention) on "
                     "device-resident inputs",
        "ms_per_step_separate_launches": round(ms_sep, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16, shuffled physical blocks)",
        "config": _config(b, world),
        "tokens_per_s": round(b.num_tokens * world / (ms * 1e-3), 1),
        "pct_of_hbm_peak": round(100.0 * gbs / world / peaks["hbm_gbs"], 2),
        "roofline": {"bound": "hbm", "kernel": "pa_paged_attention (split-KV decode + merge)",
                     "achieved": round(attn_gbs, 1), "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": round(attn_gbs / peaks["hbm_gbs"], 4),
                     "peak_source": peaks["source"] + " (hbm_gbs)",
                     "traffic": _profiled_traffic("decode_kernel_decode_batch.md",
                                                  ["pa_decode_kernel.cuh", "pa_decode.cu",
                                                   "pa_common.cuh"], b.name, "decode_batch"),
                     "algorithmic_bytes_per_launch": alg["attention"],
                     "avg_launch_ms": round(attn_ms, 5),
                     "timing": "CUDA events around a CUDA graph of back-to-back attention "
                               "calls (median of 5 replays); inputs larger than L2",
                     "avg_launch_ms_host_loop": round(loop_attn_ms, 5)},
        "e2e": {"value": round(step_bytes * world / (e2e_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
                "ms_per_step": round(e2e_ms, 5), "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h),
                "path": "ops.StepGraph(host_io=True): per launch one copy of the step's "
                        "inputs from pinned host memory (side stream), scatter + attention, "
                        "one copy of out back to pinned memory (side stream); the copies "
                        "of one step overlap the kernels of its neighbours"},
        # the timed value path: a graph launch per step (a decode-only step
        # scatters inside the decode kernel)
        "gpu_launches": _graph_launch_count(b) * args.steps,
        "clocks": clk,
    }
    # ---- the mixed chunked-prefill step (second half of the metric)
    if not args.no_mixed and args.workload != "mixed_step":
        mb = _make("mixed_step", rank)
        md = W.to_device(mb, dev)
        mws = ops.alloc_workspace(mb.num_seqs, mb.num_tokens, mb.num_q_heads, mb.num_kv_heads,
                                  mb.head_dim, mb.max_q_len, mb.max_seq_len, dev)
        mout = torch.empty_like(md.q)
        mms, _, mattn = _time_steps(mb, md, mws, mout, args.steps, args.warmup, stream, ops)
        mgms, mgout = _time_graph_steps(mb, md, args.steps, args.warmup, stream, ops)
        if not torch.equal(mgout[:mb.num_tokens].view(torch.int16), mout.view(torch.int16)):
            raise RuntimeError("the mixed step's graph output differs from separate launches'")
        pre = _time_prefill(mb, md, args.steps, args.warmup, stream, ops, _flush_buffer(dev))
        bounds = _mixed_bounds(mb, peaks)
        line["mixed_batch"] = {
            "workload": mb.name, "description": W.WORKLOADS[mb.name].description,
            "tokens_per_s": round(mb.num_tokens * world / (mms * 1e-3), 1),
            "ms_per_step": round(mms, 5), "attention_ms": round(mattn, 5),
            "graph_tokens_per_s": round(mb.num_tokens * world / (mgms * 1e-3), 1),
            "graph_ms_per_step": round(mgms, 5),
            "gpu_launches": _graph_launch_count(mb) * args.steps,
            "gpu_launches_separate": _launch_count(mb) * args.steps,
            "roofline": {"bound": "mixed (hbm + tensor)",
                         "frac": round(bounds["sum_bound_ms"] / mgms, 4),
                         "frac_separate_launches": round(bounds["sum_bound_ms"] / mms, 4),
                         "definition": "sum over the step's kernels of their roofline time "
                                       "(decode and scatter bytes / HBM peak, chunk causal "
                                       "FLOPs / bf16 burst peak) / measured step time "
                                       "(one graph launch per step)",
                         **bounds}}
        host_batches["mixed_step"] = mb
        if pre:
            line["roofline_prefill"] = {
                "bound": "tensor", "kernel": "prefill chunk alone (tcgen05)",
                "achieved": pre["tflops"], "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": round(pre["tflops"] / peaks["bf16_tflops"], 4),
                "peak_source": peaks["source"] + " (bf16_tflops, burst)",
                "traffic": _profiled_traffic("prefill_kernel_mixed_step.md",
                                             ["pa_prefill_kernel.cuh", "pa_prefill.cu",
                                              "pa_common.cuh", "pa_tcgen05.cuh"],
                                             mb.name, "mixed_step"),
                "algorithmic_flops_per_launch": pre["flops"], "avg_launch_ms": pre["ms"],
                "timing": "CUDA events around a CUDA graph of back-to-back calls, each after "
                          "a 256 MB write that evicts L2, minus a graph of the writes alone "
                          "(median of 5 replays)"}
        del md, mws, mout
    if not args.no_trace:
        line["trace"] = _run_trace(dev, stream, ops, args.warmup)
    if not args.no_block32:
        line["block_size_32"] = _block32(args, dev, stream, ops, peaks)
    if not args.no_other_decodes:
        line["other_decodes"] = _other_decodes(args, dev, stream, ops, peaks, host_batches)
    if not args.no_fp8:
        line["fp8_cache"] = _fp8(args, dev, stream, ops, peaks, attn_ms)
    if rank == 0 and not args.no_cpu_baseline:
        cb = cpu_baselines(host_batches, trace_rows_full=args.cpu_full)
        main = cb.get(b.name)
        line["cpu_baseline"] = {"value": main["value"], "unit": main["unit"],
                                "cores": main["cores"], "kind": "oracle",
                                "single_thread_value": main["one_core_value"],
                                "sample": main["sample"]}
        line["cpu_baselines"] = cb
    line["summary"] = _summary(line)
    if world > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def _oracle_sample_step(b, n_seqs, rng, threads=0):
    """One oracle pass over a sample of n_seqs requests of batch b (scatter of
    their new tokens + attention); returns (seconds, algorithmic bytes)."""
    import oracle
    from paged_kv_cache_174_gb300 import workloads as W

    idx = np.sort(rng.choice(b.num_seqs, size=min(n_seqs, b.num_seqs), replace=False))
    ql = b.q_lens[idx]
    qsl = np.zeros(len(idx) + 1, np.int32)
    qsl[1:] = np.cumsum(ql)
    rows = np.concatenate([np.arange(b.query_start_loc[s], b.query_start_loc[s + 1])
                           for s in idx]).astype(np.int64)
    sub = W.PagedBatch(name=b.name, q=b.q[rows], k_new=b.k_new[rows], v_new=b.v_new[rows],
                       k_cache=b.k_cache, v_cache=b.v_cache, block_tables=b.block_tables[idx],
                       seq_lens=b.seq_lens[idx], query_start_loc=qsl,
                       slot_mapping=b.slot_mapping[rows], scale=b.scale,
                       block_size=b.block_size, seed=b.seed)
    t = time.perf_counter()
    oracle.reshape_and_cache(sub.k_new, sub.v_new, b.k_cache, b.v_cache, sub.slot_mapping)
    oracle.paged_attention(sub.q, b.k_cache, b.v_cache, sub.block_tables, sub.seq_lens,
                           sub.query_start_loc, sub.scale, threads=threads)
    dt = time.perf_counter() - t
    return dt, W.algorithmic_bytes(sub)["total"], len(idx)


def _oracle_full_step(b, threads=0):
    """One oracle pass over the whole batch b: scatter of the new tokens, then
    attention of every row.  Returns seconds."""
    import oracle
    kc, vc = b.k_cache, b.v_cache
    t = time.perf_counter()
    oracle.reshape_and_cache(b.k_new, b.v_new, kc, vc, b.slot_mapping)
    oracle.paged_attention(b.q, kc, vc, b.block_tables, b.seq_lens, b.query_start_loc,
                           b.scale, threads=threads)
    return time.perf_counter() - t


def _oracle_rows(b, samples, threads=0):
    """The oracle on the given (sequence, row, q head) samples of batch b
    (its cache already holds the step's new tokens).  Returns seconds."""
    import oracle
    t = time.perf_counter()
    oracle.paged_attention_rows(b.q, b.k_cache, b.v_cache, b.block_tables, b.seq_lens,
                                b.query_start_loc, b.scale, samples, threads=threads)
    return time.perf_counter() - t


def _all_rows(b, seqs, every=1, rng=None):
    """(sequence, row, q head) triples of the given sequences; with every > 1
    one row in `every` of each sequence (a random offset), all q heads."""
    out = []
    for s in seqs:
        n = int(b.q_lens[s])
        start = int(rng.integers(0, every)) if (rng is not None and every > 1) else 0
        for i in range(min(start, max(n - 1, 0)), n, every):
            out.extend((s, i, h) for h in range(b.num_q_heads))
    return np.array(out, np.int32).reshape(-1, 3)


def _cpu_decode(b, unit_bytes, one_core_frac=1.0):
    """A decode batch (C1-C3): the oracle over the whole batch on all cores;
    on one core the whole batch, or a random fraction of its requests (the
    unit is bytes per second, so a sample gives the rate directly)."""
    from paged_kv_cache_174_gb300 import workloads as W
    import oracle
    t_all = _oracle_full_step(b)
    reps = 1
    while t_all < 0.5 and reps < 1000:  # small batches: repeat for a stable time
        t_all += _oracle_full_step(b)
        reps += 1
    alg = W.algorithmic_bytes(b)["total"]
    rng = np.random.default_rng(3)
    if one_core_frac >= 1.0:
        t1 = _oracle_full_step(b, threads=1)
        b1, what1 = alg, "the whole batch"
    else:
        n = max(1, int(round(b.num_seqs * one_core_frac)))
        dt, b1, _ = _oracle_sample_step(b, n, rng, threads=1)
        t1, what1 = dt, f"{n} random requests of {b.num_seqs}"
    return {"unit": unit_bytes, "cores": oracle.num_threads(),
            "value": round(alg * reps / t_all / 1e9, 4),
            "seconds": round(t_all / reps, 4),
            "one_core_value": round(b1 / t1 / 1e9, 4),
            "sample": f"all cores: the whole batch (scatter + attention), {reps} pass(es); "
                      f"one core: {what1}"}


def _cpu_mixed(b):
    """The mixed step (C4): the whole step on all cores; on one core every
    decode row and one chunk row in 16 (all q heads), the chunk's time scaled
    by the rows it stands for."""
    import oracle
    t_all = _oracle_full_step(b)
    rng = np.random.default_rng(4)
    dec = [s for s in range(b.num_seqs) if b.q_lens[s] == 1]
    pre = [s for s in range(b.num_seqs) if b.q_lens[s] >= 2]
    t_dec = _oracle_rows(b, _all_rows(b, dec), threads=1)
    smp = _all_rows(b, pre, every=16, rng=rng)
    t_pre = _oracle_rows(b, smp, threads=1)
    n_pre = int(sum(b.q_lens[s] for s in pre)) * b.num_q_heads
    t1 = t_dec + t_pre * n_pre / max(len(smp), 1)
    return {"unit": "tokens/s", "cores": oracle.num_threads(),
            "value": round(b.num_tokens / t_all, 2), "seconds": round(t_all, 4),
            "one_core_value": round(b.num_tokens / t1, 3),
            "one_core_seconds_estimated": round(t1, 3),
            "sample": "all cores: the whole step (scatter + attention of all 640 rows); one "
                      "core: all decode rows, and 1 in 16 chunk rows (all q heads) with the "
                      "chunk's time scaled by 16"}


def _cpu_trace(every=10, full_rows=True):
    """The continuous-batching trace (C5): every step's copy-on-write copies
    and scatter replayed in the oracle, attention of every `every`-th step
    timed (all its rows on all cores, or 1 in 8 chunk rows when full_rows is
    False); on one core the attention of one timed step in 10, 1 in 16 chunk
    rows, scaled.  The q / k / v values are drawn with torch's CPU generator
    (the oracle's time does not depend on them)."""
    import oracle
    import torch
    from paged_kv_cache_174_gb300 import workloads as W
    from paged_kv_cache_174_gb300.host import CONTINUOUS_BATCHING_TRACE, ContinuousBatchingTrace

    cfg = CONTINUOUS_BATCHING_TRACE
    tr = ContinuousBatchingTrace(cfg)
    plans = [tr.step() for _ in range(cfg.steps)]
    kc, vc = W.trace_initial_cache(cfg, tr.prefix_blocks, poison=False)
    gen = torch.Generator().manual_seed(cfg.seed)

    def bits(*shape):
        return torch.randn(*shape, generator=gen).bfloat16().view(torch.int16).numpy().view(
            np.uint16)

    rng = np.random.default_rng(5)
    scale = 1.0 / np.sqrt(cfg.head_dim)
    t_all = t_one = 0.0
    toks = toks_one = timed = 0
    for p in plans:
        if p.num_tokens == 0:
            continue
        T = p.num_tokens
        k, v = bits(T, cfg.num_kv_heads, cfg.head_dim), bits(T, cfg.num_kv_heads, cfg.head_dim)
        take = p.index % every == 0
        t0 = time.perf_counter()
        if len(p.copy_pairs):
            oracle.copy_blocks(kc, vc, p.copy_pairs)
        oracle.reshape_and_cache(k, v, kc, vc, p.slot_mapping)
        t_io = time.perf_counter() - t0
        if not take:
            continue
        q = bits(T, cfg.num_q_heads, cfg.head_dim)
        b = W.PagedBatch(name="trace", q=q, k_new=k, v_new=v, k_cache=kc, v_cache=vc,
                         block_tables=p.block_tables, seq_lens=p.seq_lens,
                         query_start_loc=p.query_start_loc, slot_mapping=p.slot_mapping,
                         scale=scale, block_size=cfg.block_size, seed=cfg.seed)
        ql = b.q_lens
        if full_rows:
            t0 = time.perf_counter()
            oracle.paged_attention(q, kc, vc, p.block_tables, p.seq_lens, p.query_start_loc,
                                   scale)
            t_all += t_io + time.perf_counter() - t0
        else:
            dec = [s for s in range(b.num_seqs) if ql[s] == 1]
            pre = [s for s in range(b.num_seqs) if ql[s] >= 2]
            t_d = _oracle_rows(b, _all_rows(b, dec))
            smp = _all_rows(b, pre, every=8, rng=rng)
            t_p = _oracle_rows(b, smp) if len(smp) else 0.0
            n_pre = int(sum(ql[s] for s in pre)) * b.num_q_heads
            t_all += t_io + t_d + t_p * n_pre / max(len(smp), 1)
        toks += T
        if timed % 10 == 0:
            dec = [s for s in range(b.num_seqs) if ql[s] == 1]
            pre = [s for s in range(b.num_seqs) if ql[s] >= 2]
            t_d = _oracle_rows(b, _all_rows(b, dec), threads=1)
            smp = _all_rows(b, pre, every=16, rng=rng)
            t_p = _oracle_rows(b, smp, threads=1) if len(smp) else 0.0
            n_pre = int(sum(ql[s] for s in pre)) * b.num_q_heads
            t_one += t_io + t_d + t_p * n_pre / max(len(smp), 1)
            toks_one += T
        timed += 1
    rows = "all rows" if full_rows else "all decode rows and 1 in 8 chunk rows (scaled)"
    return {"unit": "tokens/s", "cores": oracle.num_threads(),
            "value": round(toks / t_all, 2), "seconds": round(t_all, 3),
            "one_core_value": round(toks_one / t_one, 3),
            "sample": f"all cores: {timed} steps (every {every}th of 200), {rows}, plus "
                      f"their copies and scatter (the other steps' copies and scatter "
                      f"replayed untimed); one core: one timed step in 10, all decode rows "
                      f"and 1 in 16 chunk rows with the chunk's time scaled by 16"}


def cpu_baselines(host_batches, trace_rows_full):
    """The oracle on every workload, on all host cores and on one core."""
    res = {}
    if "tiny_decode" in host_batches:
        res["tiny_decode"] = _cpu_decode(host_batches["tiny_decode"], "GB/s")
    if "decode_batch" in host_batches:
        res["decode_batch"] = _cpu_decode(host_batches["decode_batch"], "GB/s")
    if "long_decode" in host_batches:
        res["long_decode"] = _cpu_decode(host_batches["long_decode"], "GB/s",
                                         one_core_frac=0.25)
    if "mixed_step" in host_batches:
        res["mixed_step"] = _cpu_mixed(host_batches["mixed_step"])
    res["trace"] = _cpu_trace(full_rows=trace_rows_full)
    return res


def run_reference(args):
    world, rank, _ = _dist()
    if rank != 0:
        return
    import oracle
    from paged_kv_cache_174_gb300 import workloads as W

    b = _make(args.workload, rank)
    rng = np.random.default_rng(1)
    n_seqs = max(1, min(b.num_seqs, 8))
    for _ in range(args.warmup):
        _oracle_sample_step(b, n_seqs, rng)
    ts, bs = [], []
    for _ in range(args.steps):
        dt, nb, _ = _oracle_sample_step(b, n_seqs, rng)
        ts.append(dt)
        bs.append(nb)
    value = sum(bs) / sum(ts) / 1e9
    line = {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * sum(ts) / len(ts), 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) bf16, shuffled physical blocks)",
        "config": _config(b, world),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": oracle.num_threads(),
                         "kind": "oracle",
                         "sample": f"each step: {n_seqs} random requests of the batch "
                                   f"(scatter + attention)"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="decode_batch",
                    choices=["tiny_decode", "decode_batch", "long_decode", "mixed_step"])
    ap.add_argument("--cpu-full", action="store_true",
                    help="time the oracle on every row of the trace's sampled steps "
                         "(default: all decode rows and 1 in 8 chunk rows)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-mixed", action="store_true",
                    help="skip the mixed chunked-prefill step measurement")
    ap.add_argument("--no-trace", action="store_true",
                    help="skip the continuous-batching trace measurement")
    ap.add_argument("--no-other-decodes", action="store_true",
                    help="skip the tiny and long-context decode measurements")
    ap.add_argument("--no-fp8", action="store_true",
                    help="skip the 8-bit cache decode measurement")
    ap.add_argument("--no-block32", action="store_true",
                    help="skip the 32-token block comparison")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
