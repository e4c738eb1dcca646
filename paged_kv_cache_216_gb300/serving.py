"""Serving decode step on one GPU: allocate, copy-on-write, append, decode.

One step ("Day 6/90 of Inference Engineering", PagedAttention notes,
paragraphs 2, 5 and 6): the host allocator reserves every sequence's next
slot (a new block when the last one is full; a copy when it is shared and
partly filled), the slot mapping, context lengths and updated block tables
go to the device in one copy, pending block copies run, the new keys/values
are appended, and paged decode attends over the grown contexts (the new
token included).

The host-side tables live in one pinned buffer that the allocator updates in
place.  Before rewriting it for the next step the host waits for the
previous step's upload to have executed (an event recorded right after the
copy), so the host runs at most one step ahead of the device.

The device part of a step can be captured once into a CUDA graph
(:meth:`ServingEngine.capture`) and replayed every step: one launch instead
of a copy and four kernel launches, with no host gaps between them.  A
captured step reads its new tokens from the engine's staging buffers
(``q_in``, ``k_in``, ``v_in``) and writes ``out``.
"""

from __future__ import annotations

import numpy as np
import torch

from . import ops
from .allocator import BlockAllocator


def _event(timing: bool = False) -> torch.cuda.Event:
    """An event that, recorded during graph capture, becomes a real record
    node of the graph (when this torch supports it)."""
    try:
        return torch.cuda.Event(enable_timing=timing, external=True)
    except TypeError:
        return torch.cuda.Event(enable_timing=timing)


def graphs_supported() -> bool:
    try:
        torch.cuda.Event(external=True)
        return True
    except TypeError:
        return False


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
        # one packed upload: slots int64[S] | context_lens int32[S] | tables int32[S, width]
        t_off = (12 * s + 15) // 16 * 16
        nbytes = t_off + 4 * s * self.width
        self._up_h = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
        self._up_d = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        self.slots_h, self.ctx_h, self.tables_h = self._views(self._up_h, s, t_off)
        self.slots_d, self.ctx_d, self.tables_d = self._views(self._up_d, s, t_off)
        self.cow_h = torch.empty((s, 2), dtype=torch.int32, pin_memory=True)
        self.cow_d = torch.empty((s, 2), dtype=torch.int32, device=dev)
        self.alloc.block_tables(self.seq_ids, self.tables_h.numpy(), self.ctx_h.numpy())
        self._up_d.copy_(self._up_h, non_blocking=True)
        self.partition_size = ops.decode_partition_size(s, hkv, self.max_context_len, partition_size)
        self.workspace = ops.decode_workspace(s, num_heads, hkv, d, self.max_context_len, self.partition_size, dev)
        self.uploaded = _event()
        self.uploaded.record()
        self.launches = 0  # kernels this engine has launched
        self.split = -(-self.max_context_len // self.partition_size) > 1
        self._per_step = 2 + (1 if k_cache.dtype == torch.bfloat16 else 0) + (1 if self.split else 0)
        # staging buffers of captured steps
        self.q_in = torch.empty((s, num_heads, d), dtype=k_cache.dtype, device=dev)
        self.k_in = torch.empty((s, hkv, d), dtype=k_cache.dtype, device=dev)
        self.v_in = torch.empty((s, hkv, d), dtype=k_cache.dtype, device=dev)
        self.out = torch.empty((s, num_heads, d), dtype=k_cache.dtype, device=dev)
        self._pool = None

    @staticmethod
    def _views(buf, s, t_off):
        slots = buf[: 8 * s].view(torch.int64)
        ctx = buf[8 * s: 12 * s].view(torch.int32)
        tables = buf[t_off:].view(torch.int32).view(s, -1)
        return slots, ctx, tables

    def context_lens(self) -> np.ndarray:
        return self.ctx_h.numpy().copy()

    # -- host part ---------------------------------------------------------
    def _reserve(self) -> int:
        """Reserve every sequence's next slot into the pinned upload buffer
        and queue the block copies it requires; returns their number."""
        self.uploaded.synchronize()
        ncow = self.alloc.append_slots(self.seq_ids, self.slots_h.numpy(), self.cow_h.numpy(),
                                       self.tables_h.numpy(), self.ctx_h.numpy())
        if ncow:
            self.cow_d[:ncow].copy_(self.cow_h[:ncow], non_blocking=True)
            ops.copy_blocks(self.k_cache, self.v_cache, self.cow_d[:ncow])
            self.launches += 1
        return ncow

    # -- device part -------------------------------------------------------
    def _device(self, q, k_new, v_new, out, events=None):
        self._up_d.copy_(self._up_h, non_blocking=True)
        self.uploaded.record()
        ops.cache_append(k_new, v_new, self.slots_d, self.k_cache, self.v_cache)
        if events is not None:
            events[0].record()
        out = ops.paged_decode(q, self.k_cache, self.v_cache, self.tables_d, self.ctx_d, self.max_context_len,
                               self.scale, out=out, partition_size=self.partition_size, workspace=self.workspace)
        if events is not None:
            events[1].record()
        return out

    def step(self, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor, out: torch.Tensor | None = None,
             events=None):
        """One decode step for every sequence: q ``[S, H, D]``, k_new/v_new
        ``[S, Hkv, D]`` on the device.  Returns ``out [S, H, D]``.
        ``events`` (a pair of CUDA events) are recorded around the decode."""
        self._reserve()
        self.launches += self._per_step
        return self._device(q, k_new, v_new, out, events)

    def capture(self, events=None) -> torch.cuda.CUDAGraph:
        """Capture the device part of a step (reading ``q_in``, ``k_in``,
        ``v_in``, writing ``out``) as a CUDA graph.  Call after at least one
        eager :meth:`step`.  ``events``, if given, are recorded around the
        decode at every replay (timing events created with ``external``)."""
        if not graphs_supported():
            raise RuntimeError("this torch cannot record events inside a CUDA graph")
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        if self._pool is None:
            self._pool = torch.cuda.graph_pool_handle()
        with torch.cuda.graph(g, pool=self._pool):
            self._device(self.q_in, self.k_in, self.v_in, self.out, events)
        torch.cuda.synchronize()
        return g

    def replay(self, graph: torch.cuda.CUDAGraph, q=None, k_new=None, v_new=None) -> torch.Tensor:
        """One step through a captured graph.  New tokens given here are
        copied into the staging buffers first (they may already be there)."""
        self._reserve()
        for src, dst in ((q, self.q_in), (k_new, self.k_in), (v_new, self.v_in)):
            if src is not None and src.data_ptr() != dst.data_ptr():
                dst.copy_(src, non_blocking=True)
        graph.replay()
        self.launches += self._per_step
        return self.out

    def step_host(self, q_h: torch.Tensor, k_h: torch.Tensor, v_h: torch.Tensor, out_h: torch.Tensor,
                  graph: torch.cuda.CUDAGraph | None = None) -> torch.Tensor:
        """Same step with host (pinned) inputs and output: the new tokens are
        copied into the staging buffers, the output back to ``out_h``."""
        if graph is None:
            self.q_in.copy_(q_h, non_blocking=True)
            self.k_in.copy_(k_h, non_blocking=True)
            self.v_in.copy_(v_h, non_blocking=True)
            self.step(self.q_in, self.k_in, self.v_in, out=self.out)
        else:
            self._reserve()
            self.q_in.copy_(q_h, non_blocking=True)
            self.k_in.copy_(k_h, non_blocking=True)
            self.v_in.copy_(v_h, non_blocking=True)
            graph.replay()
            self.launches += self._per_step
        out_h.copy_(self.out, non_blocking=True)
        return out_h
