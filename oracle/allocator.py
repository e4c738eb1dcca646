"""Block allocator for a paged KV cache, as a plain Python object.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Rules ("Day 6/90 of Inference Engineering", PagedAttention notes):
  * paragraph 2: the cache manager hands out one block at a time; a sequence
    takes a new block only when its last block is full.
  * paragraph 5: sequences with a common prefix share that prefix's blocks;
    from the token where a sequence diverges it writes into a new block.
  * paragraph 6: a per-sequence block table maps logical block j to the
    physical block holding tokens j·B .. j·B+B-1.

Readings where the page is silent (each one a choice, not a quote):
  * Free list is a stack.  A fresh allocator hands out ``free_order[0]``
    first, then ``free_order[1]``, and so on; a freed block goes on top and
    is the next one handed out.
  * Sharing is by reference count.  ``fork`` gives the child the parent's
    table and token count and adds one reference to each block.
  * Copy-on-write: appending to a sequence whose last block is partly filled
    and shared (count > 1) first takes a new block, records the copy
    (old -> new), drops one reference to the old block and puts the new one
    in the table.  A full shared last block needs no copy: the append takes
    a new block anyway.
  * ``free`` drops one reference to each block of the sequence, in table
    order; blocks that reach zero go back on the free list in that order.
  * Out of blocks: the call fails and leaves the allocator unchanged.
"""

from __future__ import annotations


class OutOfBlocks(Exception):
    pass


class BlockAllocator:
    def __init__(self, num_blocks: int, block_size: int, free_order=None):
        if free_order is None:
            free_order = range(num_blocks)
        order = [int(b) for b in free_order]
        assert sorted(order) == list(range(num_blocks))
        self.num_blocks = num_blocks
        self.block_size = block_size
        self._free = list(reversed(order))  # top of the stack is the end
        self.refcount = [0] * num_blocks
        self.tables: dict[int, list[int]] = {}
        self.lengths: dict[int, int] = {}

    # -- queries ---------------------------------------------------------
    def num_free(self) -> int:
        return len(self._free)

    def block_table(self, seq_id: int) -> list[int]:
        return list(self.tables[seq_id])

    def num_tokens(self, seq_id: int) -> int:
        return self.lengths[seq_id]

    # -- operations ------------------------------------------------------
    def _pop(self) -> int:
        b = self._free.pop()
        assert self.refcount[b] == 0
        self.refcount[b] = 1
        return b

    def add(self, seq_id: int, num_tokens: int) -> None:
        """New sequence holding ``num_tokens`` tokens in ceil(n/B) fresh blocks."""
        if seq_id in self.tables or num_tokens < 0:
            raise KeyError(seq_id)
        need = -(-num_tokens // self.block_size)
        if need > len(self._free):
            raise OutOfBlocks(seq_id)
        self.tables[seq_id] = [self._pop() for _ in range(need)]
        self.lengths[seq_id] = num_tokens

    def fork(self, parent_id: int, child_id: int) -> None:
        if parent_id not in self.tables or child_id in self.tables:
            raise KeyError(child_id)
        table = list(self.tables[parent_id])
        for b in table:
            self.refcount[b] += 1
        self.tables[child_id] = table
        self.lengths[child_id] = self.lengths[parent_id]

    def append_slot(self, seq_id: int):
        """Reserve the slot of the sequence's next token.

        Returns ``(slot, cow_src, cow_dst)``; the copy pair is ``(-1, -1)``
        when no block had to be copied."""
        table = self.tables[seq_id]
        n = self.lengths[seq_id]
        r = n % self.block_size
        cow = (-1, -1)
        if r == 0:
            if not self._free:
                raise OutOfBlocks(seq_id)
            table.append(self._pop())
        else:
            last = table[-1]
            if self.refcount[last] > 1:
                if not self._free:
                    raise OutOfBlocks(seq_id)
                new = self._pop()
                self.refcount[last] -= 1
                table[-1] = new
                cow = (last, new)
        self.lengths[seq_id] = n + 1
        return table[-1] * self.block_size + r, cow[0], cow[1]

    def free(self, seq_id: int) -> None:
        table = self.tables.pop(seq_id)
        del self.lengths[seq_id]
        for b in table:
            assert self.refcount[b] > 0
            self.refcount[b] -= 1
            if self.refcount[b] == 0:
                self._free.append(b)
