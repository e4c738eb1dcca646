"""Populate an allocator with a batch of sequences, optionally sharing one
prefix.

Prefix sharing ("Day 6/90 of Inference Engineering", PagedAttention notes,
paragraph 5): a prefix sequence (id = num_seqs) receives ``prefix_len``
tokens; sequences 0 .. prefix_share-1 fork from it and then each appends its
own remaining tokens one slot at a time, which copies the prefix's last
block first when the prefix ends inside a block; the prefix sequence is then
dropped.  The other sequences get fresh blocks for their ``ctx`` tokens.
"""

from __future__ import annotations

import numpy as np

from .allocator import BlockAllocator


def populate(alloc: BlockAllocator, ctx, prefix_len: int = 0, prefix_share: int = 0) -> np.ndarray:
    """Returns the block copies (int32 ``[n, 2]``, src -> dst, in order) the
    caller must apply to the caches."""
    num_seqs = len(ctx)
    pairs = []
    if prefix_share:
        pid = num_seqs
        alloc.add(pid, prefix_len)
        for s in range(prefix_share):
            alloc.fork(pid, s)
        for s in range(prefix_share):
            for _ in range(int(ctx[s]) - prefix_len):
                _, src, dst = alloc.append_slot(s)
                if src >= 0:
                    pairs.append((src, dst))
        alloc.free(pid)
    for s in range(prefix_share, num_seqs):
        alloc.add(s, int(ctx[s]))
    return np.asarray(pairs, dtype=np.int32).reshape(-1, 2)
