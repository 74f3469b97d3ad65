"""Host-side physical block allocator for the paged KV cache.

Follows the block manager the pages describe ("PagedAttention 显存分页与连续批处理
(Continuous Batching)实战", TypeScript Block Manager: a pool of physical
blocks with a free list, allocation pops a free block and sets its reference
count to 1, freeing decrements it and returns the block to the pool at zero,
exhaustion is an error; "连续批处理：推理吞吐的范式革命", section 2.1: a
finished request's blocks are reusable at once; section 4.2 and
"vLLM中的PagedAttention机制与显存优化实践", section 1.1: requests share the
blocks of a common prefix by reference, so 10 requests with a 500-token prefix
hold one copy plus 9 references).

The free list is last-in first-out, so a freed block is the next one handed
out ("immediate free/reuse"); on a fresh pool blocks come out in increasing id
order.  Copy-on-write: a request about to write into a block whose reference
count is above one gets a fresh private block, a (src, dst) copy is recorded for
the GPU's block-copy kernel, and the shared block loses one reference.
"""
from __future__ import annotations

from typing import Dict, List, Tuple


class OutOfBlocks(RuntimeError):
    """The pool has no free physical block."""


class BlockAllocator:
    def __init__(self, num_blocks: int, block_size: int):
        if num_blocks <= 0 or block_size <= 0:
            raise ValueError("num_blocks and block_size must be positive")
        self.num_blocks = num_blocks
        self.block_size = block_size
        # top of the stack is the end of the list: the lowest id comes out first
        self._free: List[int] = list(range(num_blocks - 1, -1, -1))
        self._ref: List[int] = [0] * num_blocks
        self.copies_made = 0

    # ---------------------------------------------------------------- queries
    @property
    def free_count(self) -> int:
        return len(self._free)

    @property
    def used_count(self) -> int:
        return self.num_blocks - len(self._free)

    def refcount(self, block: int) -> int:
        return self._ref[block]

    # ------------------------------------------------------------- mutations
    def allocate(self) -> int:
        if not self._free:
            raise OutOfBlocks("no free physical block in the KV-cache pool")
        b = self._free.pop()
        assert self._ref[b] == 0
        self._ref[b] = 1
        return b

    def share(self, block: int) -> int:
        """One more holder of an allocated block (prefix sharing)."""
        if self._ref[block] <= 0:
            raise ValueError(f"block {block} is not allocated")
        self._ref[block] += 1
        return block

    def free(self, block: int) -> None:
        """Drop one reference; the block returns to the pool at zero."""
        if self._ref[block] <= 0:
            raise ValueError(f"block {block} is not allocated")
        self._ref[block] -= 1
        if self._ref[block] == 0:
            self._free.append(block)

    def free_all(self, table: List[int]) -> None:
        for b in table:
            self.free(b)
        table.clear()

    def make_private(self, table: List[int], index: int, copies: List[Tuple[int, int]]) -> int:
        """Copy-on-write of table[index] if it is shared: returns the block the
        caller may write, and appends (src, dst) to copies when a copy is needed."""
        b = table[index]
        if self._ref[b] == 1:
            return b
        new = self.allocate()
        copies.append((b, new))
        self.copies_made += 1
        self._ref[b] -= 1  # cannot reach zero: it was shared
        table[index] = new
        return new

    # ------------------------------------------------------------- checking
    def check(self) -> None:
        """Raise AssertionError if the pool's bookkeeping is inconsistent."""
        free = self._free
        assert len(set(free)) == len(free), "a block is twice in the free list"
        for b in free:
            assert self._ref[b] == 0, f"free block {b} has references"
        allocated = [b for b in range(self.num_blocks) if self._ref[b] > 0]
        assert len(allocated) + len(free) == self.num_blocks, "free + allocated != total"

    def refcounts(self) -> Dict[int, int]:
        return {b: r for b, r in enumerate(self._ref) if r > 0}
