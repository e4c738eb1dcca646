"""Oracle-side set-up and serving loop: allocator + append + decode.

TEST INFRASTRUCTURE ONLY (see the package docstring).

``initial_state`` runs the allocation script of a workload on the oracle's
own :class:`~oracle.allocator.BlockAllocator`:
  * without a shared prefix: sequence s gets ``ctx[s]`` tokens, s = 0, 1, ...
  * with one ("Day 6/90 of Inference Engineering", PagedAttention notes,
    paragraph 5): a prefix sequence (id = S) gets ``prefix_len`` tokens;
    sequences 0 .. prefix_share-1 fork from it, then each in turn appends
    its own ``ctx[s] - prefix_len`` tokens one slot at a time (copy-on-write
    where the prefix ends inside a block); the prefix sequence is freed;
    the remaining sequences are added as above.

``ServingOracle.step`` is one serving decode step (same page, paragraph 2):
every sequence reserves the slot of its next token (taking a new block when
its last one is full), copy-on-write copies are applied, the new keys and
values are written into their slots, and decode runs over the grown
contexts, the new token included.
"""

from __future__ import annotations

import numpy as np

from .allocator import BlockAllocator
from .attention import paged_decode
from .cache import bf16_to_f32, cache_append_inplace, copy_blocks
from .fp8 import quantize


def tables_array(alloc: BlockAllocator, seq_ids, width: int) -> np.ndarray:
    """Block tables of ``seq_ids`` as an int32 array ``[len, width]``; entries
    past a sequence's last block are -1."""
    out = np.full((len(seq_ids), width), -1, dtype=np.int32)
    for i, s in enumerate(seq_ids):
        t = alloc.block_table(s)
        out[i, :len(t)] = t
    return out


def initial_state(num_seqs: int, block_size: int, ctx, num_blocks: int,
                  free_order, prefix_len: int = 0, prefix_share: int = 0):
    """Run the workload's allocation script.  Returns ``(alloc, cow_pairs)``
    where ``cow_pairs`` lists the block copies the script requires, in
    order."""
    alloc = BlockAllocator(num_blocks, block_size, free_order)
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
    return alloc, pairs


class ServingOracle:
    """Serving loop state on the CPU: allocator, caches (mutated in place) and
    context lengths."""

    def __init__(self, alloc: BlockAllocator, k_cache: np.ndarray,
                 v_cache: np.ndarray, num_seqs: int, dtype: str, scale: float,
                 fp8_scales=None):
        """``fp8_scales = (k_scale, v_scale)``: the caches hold E4M3 codes and
        new bf16 tokens are stored quantized (``oracle.fp8``)."""
        self.fp8_scales = fp8_scales
        self.alloc = alloc
        self.k_cache = k_cache
        self.v_cache = v_cache
        self.num_seqs = num_seqs
        self.dtype = dtype
        self.scale = scale

    def context_lens(self) -> np.ndarray:
        return np.array([self.alloc.num_tokens(s) for s in range(self.num_seqs)], dtype=np.int32)

    def tables(self, width: int) -> np.ndarray:
        return tables_array(self.alloc, range(self.num_seqs), width)

    def step(self, q, k_new, v_new, width: int, seqs=None):
        """One decode step.  Returns ``(slots, pairs, out)`` where ``out`` is
        the fp64 decode output of ``seqs`` (all by default)."""
        slots = np.empty(self.num_seqs, dtype=np.int64)
        pairs = []
        for s in range(self.num_seqs):
            slot, src, dst = self.alloc.append_slot(s)
            slots[s] = slot
            if src >= 0:
                pairs.append((src, dst))
        copy_blocks(self.k_cache, self.v_cache, pairs)
        if self.fp8_scales is None:
            cache_append_inplace(self.k_cache, self.v_cache, k_new, v_new, slots)
            out = paged_decode(q, self.k_cache, self.v_cache, self.tables(width),
                               self.context_lens(), self.scale, self.dtype, seqs)
            return slots, pairs, out
        ks, vs = self.fp8_scales
        cache_append_inplace(self.k_cache, self.v_cache, quantize(bf16_to_f32(k_new), ks),
                             quantize(bf16_to_f32(v_new), vs), slots)
        out = paged_decode(q, self.k_cache, self.v_cache, self.tables(width), self.context_lens(),
                           self.scale, "bf16", seqs, cache_dtype="fp8", k_scale=ks, v_scale=vs)
        return slots, pairs, out
