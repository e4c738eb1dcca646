"""Serving decode step on one GPU: allocate, copy-on-write, append, decode.

One step ("Day 6/90 of Inference Engineering", PagedAttention notes,
paragraphs 2, 5 and 6): the host allocator reserves every sequence's next
slot (a new block when the last one is full; a copy when it is shared and
partly filled), the slot mapping and updated block tables go to the device,
pending block copies run, the new keys/values are appended, and paged decode
attends over the grown contexts (the new token included).

The host-side tables live in pinned buffers that the allocator updates in
place; before rewriting them for the next step the host waits for the
previous step's uploads to have executed, so the host runs at most one step
ahead of the device.
"""

from __future__ import annotations

import numpy as np
import torch

from . import ops
from .allocator import BlockAllocator


class ServingEngine:
    def __init__(self, k_cache: torch.Tensor, v_cache: torch.Tensor, allocator: BlockAllocator, seq_ids,
                 num_heads: int, scale: float, max_context_len: int, partition_size: int = 0):
        self.k_cache, self.v_cache = k_cache, v_cache
        self.alloc = allocator
        self.num_heads = num_heads
        self.scale = float(scale)
        self.max_context_len = int(max_context_len)
        n, hkv, b, d = k_cache.shape
        self.num_kv_heads, self.block_size, self.head_dim = hkv, b, d
        dev = k_cache.device
        self.seq_ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        s = self.seq_ids.shape[0]
        self.num_seqs = s
        self.width = -(-self.max_context_len // b)
        pin = dict(pin_memory=True)
        self.tables_h = torch.empty((s, self.width), dtype=torch.int32, **pin)
        self.ctx_h = torch.empty((s,), dtype=torch.int32, **pin)
        self.slots_h = torch.empty((s,), dtype=torch.int64, **pin)
        self.cow_h = torch.empty((s, 2), dtype=torch.int32, **pin)
        self.tables_d = torch.empty((s, self.width), dtype=torch.int32, device=dev)
        self.ctx_d = torch.empty((s,), dtype=torch.int32, device=dev)
        self.slots_d = torch.empty((s,), dtype=torch.int64, device=dev)
        self.cow_d = torch.empty((s, 2), dtype=torch.int32, device=dev)
        self.allocator_tables()
        self.partition_size = ops.decode_partition_size(s, hkv, self.max_context_len, partition_size)
        self.workspace = ops.decode_workspace(s, num_heads, hkv, d, self.max_context_len, self.partition_size, dev)
        self.uploaded = torch.cuda.Event()
        self.uploaded.record()
        self.launches = 0  # kernels this engine has launched
        self.split = -(-self.max_context_len // self.partition_size) > 1

    def allocator_tables(self) -> None:
        """(Re)load the block tables and context lengths from the allocator
        and upload them."""
        self.alloc.block_tables(self.seq_ids, self.tables_h.numpy(), self.ctx_h.numpy())
        self.tables_d.copy_(self.tables_h, non_blocking=True)
        self.ctx_d.copy_(self.ctx_h, non_blocking=True)

    def context_lens(self) -> np.ndarray:
        return self.ctx_h.numpy().copy()

    def step(self, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor, out: torch.Tensor | None = None,
             events=None):
        """One decode step for every sequence: q ``[S, H, D]``, k_new/v_new
        ``[S, Hkv, D]`` on the device.  Returns ``out [S, H, D]``.
        ``events`` (a pair of CUDA events) are recorded around the decode."""
        self.uploaded.synchronize()
        ncow = self.alloc.append_slots(self.seq_ids, self.slots_h.numpy(), self.cow_h.numpy(),
                                       self.tables_h.numpy(), self.ctx_h.numpy())
        self.slots_d.copy_(self.slots_h, non_blocking=True)
        self.tables_d.copy_(self.tables_h, non_blocking=True)
        self.ctx_d.copy_(self.ctx_h, non_blocking=True)
        if ncow:
            self.cow_d[:ncow].copy_(self.cow_h[:ncow], non_blocking=True)
        self.uploaded.record()
        if ncow:
            ops.copy_blocks(self.k_cache, self.v_cache, self.cow_d[:ncow])
            self.launches += 1
        ops.cache_append(k_new, v_new, self.slots_d, self.k_cache, self.v_cache)
        if events is not None:
            events[0].record()
        out = ops.paged_decode(q, self.k_cache, self.v_cache, self.tables_d, self.ctx_d, self.max_context_len,
                               self.scale, out=out, partition_size=self.partition_size, workspace=self.workspace)
        if events is not None:
            events[1].record()
        self.launches += 2 + (1 if self.split else 0)
        return out

    def step_host(self, q_h: torch.Tensor, k_h: torch.Tensor, v_h: torch.Tensor, out_h: torch.Tensor,
                  staging: dict) -> torch.Tensor:
        """Same step with host (pinned) inputs and output: the new tokens are
        copied to the device, the output back to ``out_h``.  ``staging``
        holds reusable device buffers ``q, k, v, out``."""
        staging["q"].copy_(q_h, non_blocking=True)
        staging["k"].copy_(k_h, non_blocking=True)
        staging["v"].copy_(v_h, non_blocking=True)
        self.step(staging["q"], staging["k"], staging["v"], out=staging["out"])
        out_h.copy_(staging["out"], non_blocking=True)
        return out_h
