"""Seeded synthetic inputs for attention over a paged KV cache.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic.  Both the CUDA path's tests/benchmark and the CPU
oracle's tests take their inputs from here, so that the two sides see the same
bfloat16 bits.

Layout (the data structure the pages define): the KV cache is a pool of
``num_blocks`` physical blocks of ``block_size`` token slots, stored as
``[num_blocks, block_size, num_kv_heads, head_dim]`` bfloat16.  A request's
token at logical position ``pos`` lives in logical block ``pos // block_size``,
which its Block Table row maps to a physical block; inside that block it is row
``pos % block_size`` ("PagedAttention 显存分页与连续批处理实战", "PagedAttention
核心机理" part 1; "连续批处理：推理吞吐的范式革命", section 2.2, Block Table
figure).  Physical ids are drawn from a seeded random permutation of the pool,
so that neighbouring logical blocks are scattered in memory.

Conventions shared by every batch:
  * ``seq_lens[s]`` counts every token of request s, including the
    ``q_len[s]`` tokens of this step, whose K/V arrive in ``k_new``/``v_new``
    and are written by the slot scatter before attention runs;
  * the cache already holds positions ``0 .. seq_len - q_len - 1``;
  * slots that hold no token (the tail of a request's last block, blocks no
    request owns) are filled with a quiet-NaN pattern, so that any read of
    them shows up in the output;
  * block-table entries past a request's last block are -1.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, List, Optional, Sequence

import numpy as np

BF16_NAN = np.uint16(0x7FC0)


def bf16_from_f32(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round to nearest even); returns bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return rounded.astype(np.uint16)


def f32_from_bf16(b: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bits to float32 (exact)."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(
        np.float32)


def randn_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    return bf16_from_f32(rng.standard_normal(size=shape, dtype=np.float32))


@dataclass
class PagedBatch:
    """One step's inputs.  bfloat16 arrays hold raw bits (uint16)."""

    name: str
    q: np.ndarray  # [T, n_q, d]
    k_new: np.ndarray  # [T, n_kv, d]
    v_new: np.ndarray  # [T, n_kv, d]
    k_cache: np.ndarray  # [num_blocks, block_size, n_kv, d]
    v_cache: np.ndarray  # [num_blocks, block_size, n_kv, d]
    block_tables: np.ndarray  # [S, max_blocks] int32, -1 padded
    seq_lens: np.ndarray  # [S] int32
    query_start_loc: np.ndarray  # [S + 1] int32
    slot_mapping: np.ndarray  # [T] int32
    scale: float
    block_size: int
    seed: int
    copy_pairs: np.ndarray = field(default_factory=lambda: np.zeros((0, 2), np.int32))

    @property
    def num_tokens(self) -> int:
        return int(self.q.shape[0])

    @property
    def num_seqs(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def num_q_heads(self) -> int:
        return int(self.q.shape[1])

    @property
    def num_kv_heads(self) -> int:
        return int(self.k_cache.shape[2])

    @property
    def head_dim(self) -> int:
        return int(self.q.shape[2])

    @property
    def num_blocks(self) -> int:
        return int(self.k_cache.shape[0])

    @property
    def q_lens(self) -> np.ndarray:
        return np.diff(self.query_start_loc).astype(np.int32)

    @property
    def max_q_len(self) -> int:
        return int(self.q_lens.max()) if self.num_seqs else 0

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max()) if self.num_seqs else 0


def _blocks_needed(n_tokens: int, block_size: int) -> int:
    return -(-n_tokens // block_size)


def make_batch(name: str, seq_lens: Sequence[int], q_lens: Sequence[int], *, num_q_heads: int,
               num_kv_heads: int, head_dim: int, block_size: int, num_blocks: int, seed: int,
               scale: Optional[float] = None, poison: bool = True,
               max_blocks: Optional[int] = None, tables: Optional[List[List[int]]] = None,
               ) -> PagedBatch:
    """Random paged batch.

    ``tables`` may pin the physical ids of each request (else a seeded random
    permutation of the pool is dealt out).  Values are N(0, 1) rounded to
    bfloat16.
    """
    rng = np.random.default_rng(seed)
    S = len(seq_lens)
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    q_lens = np.asarray(q_lens, dtype=np.int64)
    assert seq_lens.shape == q_lens.shape
    assert np.all(q_lens >= 0) and np.all(q_lens <= seq_lens)
    nblk = [_blocks_needed(int(L), block_size) for L in seq_lens]
    if max_blocks is None:
        max_blocks = max(nblk) if nblk else 1
        max_blocks = max(max_blocks, 1)
    if tables is None:
        assert sum(nblk) <= num_blocks, "pool too small"
        perm = rng.permutation(num_blocks).astype(np.int32)
        tables = []
        off = 0
        for n in nblk:
            tables.append(list(perm[off:off + n]))
            off += n
    block_tables = np.full((S, max_blocks), -1, dtype=np.int32)
    for s, row in enumerate(tables):
        assert len(row) >= nblk[s]
        block_tables[s, :len(row)] = row

    nq, nkv, d = num_q_heads, num_kv_heads, head_dim
    fill = BF16_NAN if poison else np.uint16(0)
    k_cache = np.full((num_blocks, block_size, nkv, d), fill, dtype=np.uint16)
    v_cache = np.full((num_blocks, block_size, nkv, d), fill, dtype=np.uint16)
    kflat = k_cache.reshape(num_blocks * block_size, nkv, d)
    vflat = v_cache.reshape(num_blocks * block_size, nkv, d)

    T = int(q_lens.sum())
    qsl = np.zeros(S + 1, dtype=np.int32)
    qsl[1:] = np.cumsum(q_lens)
    slot_mapping = np.zeros(T, dtype=np.int32)

    def slots_of(s: int, lo: int, hi: int) -> np.ndarray:
        pos = np.arange(lo, hi, dtype=np.int64)
        return (block_tables[s, pos // block_size].astype(np.int64) * block_size
                + pos % block_size)

    for s in range(S):
        ctx = int(seq_lens[s] - q_lens[s])
        if ctx > 0:
            sl = slots_of(s, 0, ctx)
            kflat[sl] = randn_bf16(rng, (ctx, nkv, d))
            vflat[sl] = randn_bf16(rng, (ctx, nkv, d))
        if q_lens[s] > 0:
            slot_mapping[qsl[s]:qsl[s + 1]] = slots_of(s, ctx, int(seq_lens[s]))
    q = randn_bf16(rng, (T, nq, d))
    k_new = randn_bf16(rng, (T, nkv, d))
    v_new = randn_bf16(rng, (T, nkv, d))
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    return PagedBatch(name=name, q=q, k_new=k_new, v_new=v_new, k_cache=k_cache,
                      v_cache=v_cache, block_tables=block_tables,
                      seq_lens=seq_lens.astype(np.int32), query_start_loc=qsl,
                      slot_mapping=slot_mapping, scale=float(scale), block_size=block_size,
                      seed=seed)


# ---------------------------------------------------------------------------
# The named workloads.  Seeds are 1000 + the workload number.
# ---------------------------------------------------------------------------

@dataclass(frozen=True)
class Workload:
    key: str
    description: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    seed: int


WORKLOADS: Dict[str, Workload] = {
    "tiny_decode": Workload(
        "tiny_decode",
        "tiny decode: 4 seqs, lens {5,17,33,48}, 1 query token each, 4 q / 2 kv heads, "
        "head_dim 64, block_size 16, 32-block pool, scale 1/8", 4, 2, 64, 16, 32, 1001),
    "decode_batch": Workload(
        "decode_batch",
        "decode batch: 64 seqs, lens uniform in [128, 4096], 1 query token each, "
        "32 q / 8 kv heads, head_dim 128, block_size 16, 20000-block pool", 32, 8, 128, 16,
        20000, 1002),
    "long_decode": Workload(
        "long_decode",
        "long-context decode: 8 seqs x 32768 tokens, 1 query token each, 32 q / 8 kv heads, "
        "head_dim 128, block_size 16, 20480-block pool", 32, 8, 128, 16, 20480, 1003),
    "mixed_step": Workload(
        "mixed_step",
        "mixed chunked-prefill step: 128 decode seqs with lens uniform in [256, 2048] plus "
        "one 512-token causal prefill chunk at cached offset 3584 (640 tokens = "
        "max_num_batched_tokens), 32 q / 8 kv heads, head_dim 128, block_size 16, "
        "20000-block pool", 32, 8, 128, 16, 20000, 1004),
}


def tiny_decode(poison: bool = True) -> PagedBatch:
    w = WORKLOADS["tiny_decode"]
    return make_batch(w.key, [5, 17, 33, 48], [1, 1, 1, 1], num_q_heads=w.num_q_heads,
                      num_kv_heads=w.num_kv_heads, head_dim=w.head_dim,
                      block_size=w.block_size, num_blocks=w.num_blocks, seed=w.seed,
                      scale=1.0 / 8.0, poison=poison)


def decode_batch(poison: bool = True, num_seqs: int = 64, seed: Optional[int] = None,
                 block_size: int = 16, num_q_heads: Optional[int] = None) -> PagedBatch:
    """block_size 32 keeps the pool's token slots (half as many blocks);
    num_q_heads changes the GQA group over the same cache (64: group 8)."""
    w = WORKLOADS["decode_batch"]
    seed = w.seed if seed is None else seed
    rng = np.random.default_rng(seed + 7)
    lens = rng.integers(128, 4096, size=num_seqs, endpoint=True)
    nq = w.num_q_heads if num_q_heads is None else num_q_heads
    return make_batch(w.key, lens, [1] * num_seqs, num_q_heads=nq,
                      num_kv_heads=w.num_kv_heads, head_dim=w.head_dim,
                      block_size=block_size, num_blocks=w.num_blocks * w.block_size // block_size,
                      seed=seed, poison=poison)


def long_decode(poison: bool = True, seq_len: int = 32768, num_seqs: int = 8) -> PagedBatch:
    w = WORKLOADS["long_decode"]
    return make_batch(w.key, [seq_len] * num_seqs, [1] * num_seqs,
                      num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads,
                      head_dim=w.head_dim, block_size=w.block_size,
                      num_blocks=max(w.num_blocks, num_seqs * seq_len // w.block_size),
                      seed=w.seed, poison=poison)


def mixed_step(poison: bool = True, num_decode: int = 128, chunk: int = 512,
               cached: int = 3584, block_size: int = 16) -> PagedBatch:
    """Decodes first, then the prefill chunk (the order the step driver uses);
    block_size 32 keeps the pool's token slots (half as many blocks)."""
    w = WORKLOADS["mixed_step"]
    rng = np.random.default_rng(w.seed + 7)
    lens = list(rng.integers(256, 2048, size=num_decode, endpoint=True))
    seq_lens = lens + [cached + chunk]
    q_lens = [1] * num_decode + [chunk]
    return make_batch(w.key, seq_lens, q_lens, num_q_heads=w.num_q_heads,
                      num_kv_heads=w.num_kv_heads, head_dim=w.head_dim,
                      block_size=block_size, num_blocks=w.num_blocks * w.block_size // block_size,
                      seed=w.seed, poison=poison)


def by_name(name: str, **kw) -> PagedBatch:
    return {"tiny_decode": tiny_decode, "decode_batch": decode_batch,
            "long_decode": long_decode, "mixed_step": mixed_step}[name](**kw)


def algorithmic_bytes(b: PagedBatch) -> Dict[str, int]:
    """Bytes a perfect implementation must move for one step of batch b.

    attention: every cached key and value row of every request once, plus q,
    the output and the used block-table entries; scatter: read the new rows,
    write them to their slots.
    """
    e = 2  # bytes per bfloat16
    kv_row = b.num_kv_heads * b.head_dim * e
    ql = b.q_lens
    attn_kv = int(b.seq_lens.astype(np.int64).sum()) * 2 * kv_row
    q_out = 2 * int(ql.sum()) * b.num_q_heads * b.head_dim * e
    tables = int(sum(_blocks_needed(int(L), b.block_size) for L in b.seq_lens)) * 4
    meta = 4 * (2 * b.num_seqs + 1)
    scatter = 2 * 2 * int((b.slot_mapping >= 0).sum()) * kv_row
    return {"attention": attn_kv + q_out + tables + meta, "attention_kv": attn_kv,
            "scatter": scatter + 4 * b.num_tokens,
            "total": attn_kv + q_out + tables + meta + scatter + 4 * b.num_tokens}


def algorithmic_bytes_fp8(b: PagedBatch) -> Dict[str, int]:
    """algorithmic_bytes for the 8-bit cache: a cached row is head_dim one-byte
    codes plus one 4-byte scale per kv head; the scatter reads bf16 rows and
    writes codes and scales."""
    kv_row = b.num_kv_heads * (b.head_dim + 4)
    ql = b.q_lens
    attn_kv = int(b.seq_lens.astype(np.int64).sum()) * 2 * kv_row
    q_out = 2 * int(ql.sum()) * b.num_q_heads * b.head_dim * 2
    tables = int(sum(_blocks_needed(int(L), b.block_size) for L in b.seq_lens)) * 4
    meta = 4 * (2 * b.num_seqs + 1)
    n_new = int((b.slot_mapping >= 0).sum())
    scatter = n_new * 2 * (b.num_kv_heads * b.head_dim * 2 + kv_row)
    return {"attention": attn_kv + q_out + tables + meta, "attention_kv": attn_kv,
            "scatter": scatter + 4 * b.num_tokens,
            "total": attn_kv + q_out + tables + meta + scatter + 4 * b.num_tokens}


def context_slots(b: PagedBatch) -> np.ndarray:
    """Slots of every cached position before this step's tokens, request by
    request (the rows an 8-bit copy of the batch's cache must hold)."""
    out = []
    for s in range(b.num_seqs):
        ctx = int(b.seq_lens[s]) - int(b.q_lens[s])
        pos = np.arange(ctx, dtype=np.int64)
        out.append(b.block_tables[s, pos // b.block_size].astype(np.int64) * b.block_size
                   + pos % b.block_size)
    return np.concatenate(out).astype(np.int32) if out else np.zeros(0, np.int32)


def causal_flops(b: PagedBatch, min_q_len: int = 2) -> int:
    """QK^T and PV multiply-adds (2 flops each) over the causal (query, key)
    pairs of the requests with q_len >= min_q_len."""
    total = 0
    for s in range(b.num_seqs):
        ql = int(b.q_lens[s])
        if ql < min_q_len:
            continue
        L = int(b.seq_lens[s])
        # row i attends to L - ql + i + 1 keys
        pairs = ql * (L - ql) + ql * (ql + 1) // 2
        total += pairs * b.num_q_heads * b.head_dim * 4
    return total


@dataclass
class DeviceBatch:
    """torch tensors of a PagedBatch on one device (bf16 / int32)."""

    q: "object"
    k_new: "object"
    v_new: "object"
    k_cache: "object"
    v_cache: "object"
    block_tables: "object"
    seq_lens: "object"
    query_start_loc: "object"
    slot_mapping: "object"
    copy_pairs: "object"


def bf16_tensor(bits: np.ndarray, device):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.to(device)


def int32_tensor(a: np.ndarray, device):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


def to_device(b: PagedBatch, device="cuda") -> DeviceBatch:
    return DeviceBatch(q=bf16_tensor(b.q, device), k_new=bf16_tensor(b.k_new, device),
                       v_new=bf16_tensor(b.v_new, device), k_cache=bf16_tensor(b.k_cache, device),
                       v_cache=bf16_tensor(b.v_cache, device),
                       block_tables=int32_tensor(b.block_tables, device),
                       seq_lens=int32_tensor(b.seq_lens, device),
                       query_start_loc=int32_tensor(b.query_start_loc, device),
                       slot_mapping=int32_tensor(b.slot_mapping, device),
                       copy_pairs=int32_tensor(b.copy_pairs.reshape(-1, 2), device))


def bits_of(t) -> np.ndarray:
    """bf16 torch tensor (any device) -> uint16 numpy bits."""
    import torch
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


# ---------------------------------------------------------------------------
# Continuous-batching trace inputs (the schedule comes from host.trace)
# ---------------------------------------------------------------------------

def trace_initial_cache(cfg, prefix_blocks, poison: bool = True):
    """Pool for the trace: the shared prefix's K/V written into its blocks,
    every other slot poisoned (or zero)."""
    rng = np.random.default_rng(cfg.seed + 1)
    shape = (cfg.num_blocks, cfg.block_size, cfg.num_kv_heads, cfg.head_dim)
    if poison:
        kc = np.full(shape, BF16_NAN, dtype=np.uint16)
        vc = np.full(shape, BF16_NAN, dtype=np.uint16)
    else:  # zero pages are mapped lazily: only the slots a run writes cost memory
        kc = np.zeros(shape, dtype=np.uint16)
        vc = np.zeros(shape, dtype=np.uint16)
    kf = kc.reshape(-1, cfg.num_kv_heads, cfg.head_dim)
    vf = vc.reshape(-1, cfg.num_kv_heads, cfg.head_dim)
    pos = np.arange(cfg.prefix)
    slots = np.asarray(prefix_blocks, np.int64)[pos // cfg.block_size] * cfg.block_size + \
        pos % cfg.block_size
    kf[slots] = randn_bf16(rng, (cfg.prefix, cfg.num_kv_heads, cfg.head_dim))
    vf[slots] = randn_bf16(rng, (cfg.prefix, cfg.num_kv_heads, cfg.head_dim))
    return kc, vc


def trace_step_inputs(cfg, step_index: int, num_tokens: int):
    """q, k_new, v_new (bf16 bits) for one trace step, N(0, 1)."""
    rng = np.random.default_rng([cfg.seed, 7, step_index])
    q = randn_bf16(rng, (num_tokens, cfg.num_q_heads, cfg.head_dim))
    k = randn_bf16(rng, (num_tokens, cfg.num_kv_heads, cfg.head_dim))
    v = randn_bf16(rng, (num_tokens, cfg.num_kv_heads, cfg.head_dim))
    return q, k, v
