"""Continuous-batching step driver that generates multi-step paged-attention
workloads (host side only; it decides what each step computes and where each
token lives, the GPU library computes it).

Iteration-level scheduling as the pages describe it ("PagedAttention
显存分页与连续批处理(Continuous Batching)实战", continuous batching section:
the step is the scheduling unit, new requests join whenever free blocks allow,
finished requests leave and free their blocks at once; Chunked Prefill section:
long prompts are cut into 512-token slices and mixed with all running decodes
under a max_num_batched_tokens budget; TypeScript engine step: admission while
free blocks >= ceil(prompt / block_size) + 2 and running < max_num_seqs, FCFS,
stopping at the first request that does not fit; "连续批处理：推理吞吐的范式革命",
section 3.2 / "vLLM中的PagedAttention机制与显存优化实践", section 1.2: under
memory pressure the newest running request is preempted, its blocks freed and
it goes back to the head of the waiting queue to be recomputed).

Preemption by swapping ("连续批处理：推理吞吐的范式革命", sections 3.2 and 3.3;
"vLLM中的PagedAttention机制与显存优化实践", sections 1.2 and 2.1): with
`preempt="swap"` the victim's KV blocks that it alone holds (reference count
one) are copied block by block to a host swap space and freed, the request
moves to the swapped queue, and swapped requests are resumed ahead of any new
admission (they have the highest priority), each into freshly allocated
blocks.  `preempt="auto"` follows the pages' rule of thumb: swap a victim
whose cached sequence is at least `swap_min_tokens` long (transfer beats
recomputation there), recompute a shorter one.  Either swap mode falls back
to recomputation when the host swap space is full.

Choices where the pages leave the policy open (documented with the build):
  * each step schedules every running decode first (one token each), then
    prefill slices of at most `chunk` tokens, at most one per request, FCFS,
    until `budget` tokens are scheduled;
  * every prompt is the first L tokens of (a `prefix`-token shared prefix,
    then unique tokens); the prefix K/V is written once before step 0 and kept
    alive by an owner reference; a request shares the prefix blocks it covers
    and copies a shared block before writing into it (copy-on-write);
  * a request with prompt length L decodes positions L, L + 1, ... (q_len 1);
    prompts no longer than the prefix need no prefill;
  * arrivals are Poisson per step; prompt lengths lognormal with the given
    median and sigma, clamped; output lengths geometric on {1, 2, ...};
  * a swapped victim's blocks that are shared prefix blocks are not copied
    out: the prefix stays cached, and the resumed request shares it again;
  * swapped requests resume in the order they were swapped out, stopping at
    the first that does not fit (its private blocks + the 2-block margin);
    no new request is admitted while one is still swapped out;
  * the GPU executes a step in this order: swap-in, swap-out, block copies,
    slot scatter, attention.  A host slot freed by a swap-in may take a
    swap-out of the same step, and a request resumed and preempted again in
    one step is copied out from the blocks it was just copied into.
"""
from __future__ import annotations

import math
from collections import deque
from dataclasses import dataclass, field
from typing import Deque, Dict, List, Optional, Tuple

import numpy as np

from .allocator import BlockAllocator, OutOfBlocks


@dataclass(frozen=True)
class TraceConfig:
    steps: int = 200
    arrival_rate: float = 8.0        # requests per step (Poisson)
    prompt_median: float = 600.0     # lognormal median
    prompt_sigma: float = 1.0
    prompt_min: int = 64
    prompt_max: int = 8192
    output_mean: float = 200.0       # geometric mean
    prefix: int = 500                # shared prompt prefix tokens
    chunk: int = 512                 # prefill slice
    budget: int = 2048               # max_num_batched_tokens
    max_num_seqs: int = 256
    num_blocks: int = 40000
    block_size: int = 16
    num_q_heads: int = 32
    num_kv_heads: int = 8
    head_dim: int = 128
    seed: int = 1005
    preempt: str = "recompute"       # "recompute" | "swap" | "auto"
    swap_blocks: int = 65536         # host swap space, in blocks (4 GiB of 8x128 bf16 K+V)
    swap_min_tokens: int = 2000      # "auto": swap victims with at least this many tokens

    def __post_init__(self):
        if self.preempt not in ("recompute", "swap", "auto"):
            raise ValueError(f"preempt must be recompute, swap or auto, not {self.preempt!r}")


CONTINUOUS_BATCHING_TRACE = TraceConfig()


@dataclass
class Request:
    rid: int
    prompt_len: int
    output_len: int
    arrival_step: int
    table: List[int] = field(default_factory=list)
    computed: int = 0     # positions whose K/V are in the cache
    generated: int = 0
    admitted_step: int = -1
    finished_step: int = -1
    preemptions: int = 0
    swaps: int = 0
    # while swapped out: per logical block, its host swap slot, or -1 for a
    # shared prefix block that stays cached on the device
    host_table: List[int] = field(default_factory=list)

    @property
    def in_prefill(self) -> bool:
        return self.computed < self.prompt_len


@dataclass
class StepPlan:
    """Everything one GPU step needs, as host arrays (int32), executed in
    field order: swap_in, swap_out, copy_pairs, scatter, attention."""

    index: int
    swap_in: np.ndarray           # [n, 2] (host slot, device block)
    swap_out: np.ndarray          # [n, 2] (device block, host slot)
    copy_pairs: np.ndarray        # [n, 2] CoW (src, dst)
    slot_mapping: np.ndarray      # [T]
    block_tables: np.ndarray      # [S, max_blocks], -1 padded
    seq_lens: np.ndarray          # [S]
    query_start_loc: np.ndarray   # [S + 1]
    rids: List[int]
    positions: np.ndarray         # [T] logical position of each new token
    token_rid: np.ndarray         # [T] request of each new token
    num_decode: int
    num_prefill_tokens: int
    stats: Dict[str, float]

    @property
    def num_tokens(self) -> int:
        return int(self.slot_mapping.shape[0])

    @property
    def max_q_len(self) -> int:
        return int(np.diff(self.query_start_loc).max()) if len(self.rids) else 0

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max()) if len(self.rids) else 0


class ContinuousBatchingTrace:
    """Generates StepPlans; see the module docstring for the policy."""

    def __init__(self, cfg: TraceConfig = CONTINUOUS_BATCHING_TRACE):
        self.cfg = cfg
        self.rng = np.random.default_rng(cfg.seed)
        self.alloc = BlockAllocator(cfg.num_blocks, cfg.block_size)
        bs = cfg.block_size
        self.prefix_blocks = [self.alloc.allocate() for _ in range(-(-cfg.prefix // bs))]
        self.waiting: Deque[Request] = deque()
        self.swapped: Deque[Request] = deque()
        self.running: List[Request] = []
        self.finished: List[Request] = []
        self.host = BlockAllocator(cfg.swap_blocks, bs) if cfg.swap_blocks > 0 else None
        self.next_rid = 0
        self.step_index = 0
        self.total_copies = 0
        self.total_swap_in = 0
        self.total_swap_out = 0
        self.total_preempt = {"recompute": 0, "swap": 0}
        self._util_sum = 0.0       # sums over steps, for the summary's means
        self._waste_sum = 0.0
        self._swap_in: List[Tuple[int, int]] = []
        self._swap_out: List[Tuple[int, int]] = []

    # ------------------------------------------------------------- arrivals
    def _arrivals(self) -> None:
        cfg = self.cfg
        n = int(self.rng.poisson(cfg.arrival_rate))
        for _ in range(n):
            L = int(round(self.rng.lognormal(math.log(cfg.prompt_median), cfg.prompt_sigma)))
            L = min(max(L, cfg.prompt_min), cfg.prompt_max)
            out = int(self.rng.geometric(1.0 / cfg.output_mean))
            self.waiting.append(Request(self.next_rid, L, out, self.step_index))
            self.next_rid += 1

    # ------------------------------------------------------------- helpers
    def _blocks_for(self, n_tokens: int) -> int:
        return -(-n_tokens // self.cfg.block_size)

    def _admit(self, req: Request) -> None:
        """Share the prefix blocks the prompt covers; the prefix K/V is cached."""
        bs = self.cfg.block_size
        covered = min(req.prompt_len, self.cfg.prefix)
        req.table = [self.alloc.share(b) for b in self.prefix_blocks[:self._blocks_for(covered)]]
        req.computed = covered
        req.admitted_step = self.step_index
        del bs

    def _release(self, req: Request) -> None:
        self.alloc.free_all(req.table)

    def _swap_victim(self, victim: Request, cow_src: Dict[int, int]) -> bool:
        """Copy the victim's private blocks out to host slots (False when the
        swap space cannot take them).  A block made private by this step's
        copy-on-write still holds nothing, so its logical content is the
        shared source block's."""
        n = -(-victim.computed // self.cfg.block_size)
        logical = []
        for bi in range(n):
            src = cow_src.get(victim.table[bi], victim.table[bi])
            shared = bi < len(self.prefix_blocks) and src == self.prefix_blocks[bi]
            assert shared or self.alloc.refcount(src) == 1, "only prefix blocks are shared"
            logical.append(-1 if shared else src)
        need = sum(1 for b in logical if b >= 0)
        if self.host is None or self.host.free_count < need:
            return False
        victim.host_table = []
        for b in logical:
            if b < 0:
                victim.host_table.append(-1)
            else:
                h = self.host.allocate()
                self._swap_out.append((b, h))
                victim.host_table.append(h)
        return True

    def _preempt_newest(self, protect: Request, cow_src: Dict[int, int]) -> bool:
        """Preempt the most recently admitted running request other than
        `protect` that holds a block of its own (one that only shares prefix
        blocks would free nothing): swap it out (swapped queue) or free its
        blocks for recomputation (head of the waiting queue)."""
        cfg = self.cfg
        for victim in sorted(self.running, key=lambda r: (r.admitted_step, r.rid), reverse=True):
            if victim is protect or all(self.alloc.refcount(b) > 1 for b in victim.table):
                continue
            self.running.remove(victim)
            swap = cfg.preempt == "swap" or (cfg.preempt == "auto"
                                             and victim.computed >= cfg.swap_min_tokens)
            if swap and self._swap_victim(victim, cow_src):
                self._release(victim)
                victim.swaps += 1
                self.swapped.append(victim)
                self.total_preempt["swap"] += 1
            else:
                self._release(victim)
                victim.computed = 0
                victim.generated = 0
                self.waiting.appendleft(victim)
                self.total_preempt["recompute"] += 1
            victim.preemptions += 1
            return True
        return False

    def _resume(self, req: Request) -> None:
        """Swapped request back onto the device: prefix blocks shared again,
        every other block freshly allocated and filled from its host slot."""
        req.table = []
        for bi, h in enumerate(req.host_table):
            if h < 0:
                req.table.append(self.alloc.share(self.prefix_blocks[bi]))
            else:
                b = self.alloc.allocate()
                self._swap_in.append((h, b))
                self.host.free(h)
                req.table.append(b)
        req.host_table = []  # keeps its admission step: its priority does not drop

    def _slots(self, req: Request, lo: int, hi: int, copies: List[Tuple[int, int]]) -> List[int]:
        """Make positions lo..hi-1 writable for req (allocate / copy-on-write)
        and return their slots."""
        bs = self.cfg.block_size
        slots = []
        for pos in range(lo, hi):
            bi = pos // bs
            while bi >= len(req.table):
                req.table.append(self.alloc.allocate())
            blk = self.alloc.make_private(req.table, bi, copies)
            slots.append(blk * bs + pos % bs)
        return slots

    # ------------------------------------------------------------------ step
    def step(self) -> StepPlan:
        cfg = self.cfg
        self._arrivals()
        self._swap_in, self._swap_out = [], []
        # swapped requests first, in swap-out order, with the same margin
        while self.swapped and len(self.running) < cfg.max_num_seqs:
            cand = self.swapped[0]
            need = sum(1 for h in cand.host_table if h >= 0)
            if self.alloc.free_count >= need + 2:
                self.swapped.popleft()
                self._resume(cand)
                self.running.append(cand)
            else:
                break
        # admission: FCFS while the pool keeps a 2-block margin
        while not self.swapped and self.waiting and len(self.running) < cfg.max_num_seqs:
            cand = self.waiting[0]
            if self.alloc.free_count >= self._blocks_for(cand.prompt_len) + 2:
                self.waiting.popleft()
                self._admit(cand)
                self.running.append(cand)
            else:
                break

        copies: List[Tuple[int, int]] = []
        sched: List[Tuple[Request, int, int]] = []  # (request, lo, hi)
        budget = cfg.budget
        # decodes first, one token each; then FCFS prefill slices
        decodes = [r for r in self.running if not r.in_prefill]
        prefills = [r for r in self.running if r.in_prefill]
        for r in decodes:
            if budget <= 0:
                break
            sched.append((r, r.computed, r.computed + 1))
            budget -= 1
        for r in prefills:
            if budget <= 0:
                break
            n = min(cfg.chunk, r.prompt_len - r.computed, budget)
            sched.append((r, r.computed, r.computed + n))
            budget -= n

        # blocks for the scheduled tokens; on exhaustion preempt the newest
        # running request (dropping its work from this step) and retry
        slot_lists: Dict[int, List[int]] = {}
        i = 0
        while i < len(sched):
            r, lo, hi = sched[i]
            try:
                slot_lists[r.rid] = self._slots(r, lo, hi, copies)
                i += 1
            except OutOfBlocks:
                before = {x.rid for x in self.running}
                if not self._preempt_newest(r, {d: s_ for (s_, d) in copies}):
                    raise
                gone = before - {x.rid for x in self.running}
                pos = [k for k, (x, _, _) in enumerate(sched) if x.rid in gone]
                for k in reversed(pos):
                    slot_lists.pop(sched[k][0].rid, None)
                    del sched[k]
                    if k < i:
                        i -= 1
                # copies into blocks the victim held went back to the pool
                copies = [(s_, d) for (s_, d) in copies if self.alloc.refcount(d) > 0]

        # metadata, in schedule order (decodes first)
        bs = cfg.block_size
        S = len(sched)
        max_blocks = max([len(r.table) for r, _, _ in sched], default=1)
        bt = np.full((S, max(max_blocks, 1)), -1, np.int32)
        seq_lens = np.zeros(S, np.int32)
        qsl = np.zeros(S + 1, np.int32)
        slots, positions, token_rid = [], [], []
        for k, (r, lo, hi) in enumerate(sched):
            bt[k, :len(r.table)] = r.table
            seq_lens[k] = hi
            qsl[k + 1] = qsl[k] + (hi - lo)
            slots += slot_lists[r.rid]
            positions += list(range(lo, hi))
            token_rid += [r.rid] * (hi - lo)
        num_decode = sum(1 for r, lo, hi in sched if not r.in_prefill)
        n_prefill = sum(hi - lo for r, lo, hi in sched if r.in_prefill)

        # advance state; finished requests free their blocks at once
        newly_finished = 0
        for r, lo, hi in sched:
            if r.in_prefill:
                r.computed = hi
            else:
                r.computed = hi
                r.generated += 1
                if r.generated >= r.output_len:
                    r.finished_step = self.step_index
                    self.running.remove(r)
                    self._release(r)
                    self.finished.append(r)
                    newly_finished += 1
        self.total_copies += len(copies)
        self.total_swap_in += len(self._swap_in)
        self.total_swap_out += len(self._swap_out)

        used_slots = sum(r.computed for r in self.running)
        alloc_slots = sum(len(r.table) for r in self.running) * bs
        stats = {"running": len(self.running), "waiting": len(self.waiting),
                 "free_blocks": self.alloc.free_count, "copies": len(copies),
                 "finished": newly_finished, "tokens": len(slots),
                 "decode_tokens": num_decode, "prefill_tokens": n_prefill,
                 "block_utilisation": self.alloc.used_count / cfg.num_blocks,
                 "tail_waste_slots": alloc_slots - used_slots,
                 "waste_fraction": (alloc_slots - used_slots) / alloc_slots if alloc_slots else 0.0,
                 "swapped": len(self.swapped), "swap_in_blocks": len(self._swap_in),
                 "swap_out_blocks": len(self._swap_out),
                 "host_free_blocks": self.host.free_count if self.host else 0}
        self._util_sum += stats["block_utilisation"]
        self._waste_sum += stats["waste_fraction"]
        plan = StepPlan(index=self.step_index,
                        swap_in=np.array(self._swap_in, np.int32).reshape(-1, 2),
                        swap_out=np.array(self._swap_out, np.int32).reshape(-1, 2),
                        copy_pairs=np.array(copies, np.int32).reshape(-1, 2),
                        slot_mapping=np.array(slots, np.int32), block_tables=bt,
                        seq_lens=seq_lens, query_start_loc=qsl,
                        rids=[r.rid for r, _, _ in sched],
                        positions=np.array(positions, np.int32),
                        token_rid=np.array(token_rid, np.int32), num_decode=num_decode,
                        num_prefill_tokens=n_prefill, stats=stats)
        self.step_index += 1
        return plan

    def check(self) -> None:
        """Pool and table invariants (raises AssertionError)."""
        self.alloc.check()
        refs: Dict[int, int] = {}
        for b in self.prefix_blocks:
            refs[b] = refs.get(b, 0) + 1
        for r in self.running:
            for b in r.table:
                refs[b] = refs.get(b, 0) + 1
        assert refs == self.alloc.refcounts(), "reference counts do not match the tables"
        bs = self.cfg.block_size
        for r in self.running:
            assert len(r.table) == -(-r.computed // bs), "a table holds a block past the last token"
            assert len(r.table) * bs - r.computed < bs, "more than the last block is partly empty"
        host_refs: Dict[int, int] = {}
        for r in self.swapped:
            assert not r.table and len(r.host_table) == -(-r.computed // bs)
            for h in r.host_table:
                if h >= 0:
                    host_refs[h] = host_refs.get(h, 0) + 1
        if self.host is not None:
            self.host.check()
            assert host_refs == self.host.refcounts(), "host slots do not match the swapped tables"
        else:
            assert not host_refs

    def summary(self) -> Dict[str, float]:
        """Whole-trace counters: preemptions by kind, blocks moved by swapping,
        copy-on-write copies, finished requests; and the per-step means of the
        pool's block utilisation (used / total blocks) and of the internal
        fragmentation (slots the running requests hold but have not filled,
        over the slots they hold: only last blocks are ever partly empty)."""
        n = max(self.step_index, 1)
        return {"mean_block_utilisation": self._util_sum / n,
                "mean_waste_fraction": self._waste_sum / n,
                "steps": self.step_index, "finished": len(self.finished),
                "running": len(self.running), "waiting": len(self.waiting),
                "swapped": len(self.swapped), "copies": self.total_copies,
                "preempt_recompute": self.total_preempt["recompute"],
                "preempt_swap": self.total_preempt["swap"],
                "swap_in_blocks": self.total_swap_in, "swap_out_blocks": self.total_swap_out}
