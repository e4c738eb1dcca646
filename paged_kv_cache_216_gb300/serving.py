"""Serving decode step on one GPU: allocate, copy-on-write, append, decode.

One step ("Day 6/90 of Inference Engineering", PagedAttention notes,
paragraphs 2, 5 and 6): the host allocator reserves every sequence's next
slot (a new block when the last one is full; a copy when it is shared and
partly filled), the slot mapping, context lengths, block copies, updated
block tables and the decode work list go to the device in one copy, pending
block copies run, the new keys/values are appended, and paged decode attends
over the grown contexts (the new token included).

Pipelining (the native stepper of the C ABI, pa_stepper_*).  The host-side
state lives in one pinned buffer that the allocator updates in place.  It is
copied to one of two device buffers on a side stream, which first waits for
the step that last read that device buffer; the main stream of step i waits
only for its own upload.  So the upload of step i runs while step i-1
decodes, and the main stream carries only append -> decode -> merge.  Before
rewriting the pinned buffer the host waits for the previous upload to
finish, which bounds it to about two steps ahead of the device.  The host
work of a step is one library call before its launches and one after.

The main-stream part of a step can be captured into CUDA graphs
(:meth:`ServingEngine.capture`, one per device buffer) and replayed every
step.
"""

from __future__ import annotations

import ctypes

import numpy as np
import torch

from . import _lib as _libmod
from . import ops
from ._lib import check, lib
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


def _align(x: int, a: int) -> int:
    return (x + a - 1) // a * a


class StepGraphs:
    """Captured main-stream part of a step, one graph per device buffer."""

    def __init__(self, graphs):
        self.graphs = graphs


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
        self.partition_size = ops.decode_partition_size(s, hkv, self.max_context_len, partition_size)
        self.bf16 = k_cache.dtype == torch.bfloat16
        plan_p = self.partition_size if self.bf16 else 0
        offs = (ctypes.c_size_t * 5)()
        total = ctypes.c_size_t(0)
        check(lib().pa_stepper_layout(s, self.max_context_len, b, plan_p, offs, ctypes.byref(total)))
        self._layout = tuple(int(x) for x in offs)
        nbytes = int(total.value)
        self._up_h = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
        self._up_d = [torch.empty(nbytes, dtype=torch.uint8, device=dev) for _ in range(2)]
        self.plan_h, self.slots_h, self.ctx_h, self.cow_h, self.tables_h = self._views(self._up_h)
        self._dv = [self._views(x) for x in self._up_d]
        self._st = ctypes.c_void_p(0)
        check(lib().pa_stepper_create(allocator._h, ctypes.c_void_p(self.seq_ids.ctypes.data), s,
                                      self.max_context_len, b, plan_p, ctypes.c_void_p(self._up_h.data_ptr()),
                                      ctypes.c_void_p(self._up_d[0].data_ptr()),
                                      ctypes.c_void_p(self._up_d[1].data_ptr()), nbytes, ctypes.byref(self._st)))
        self.workspace = ops.decode_workspace(s, num_heads, hkv, d, self.max_context_len, self.partition_size, dev)
        self.up_stream = torch.cuda.Stream(device=dev)
        self._up_ptr = ctypes.c_void_p(self.up_stream.cuda_stream)
        self._bi = ctypes.c_int(0)
        self._nc = ctypes.c_int(0)
        self.k = 0  # device buffer of the next step
        self.launches = 0  # kernels this engine has launched
        self.split = -(-self.max_context_len // self.partition_size) > 1
        self._per_step = 2 + (1 if self.split else 0)  # append + decode (+ merge)
        # staging buffers for steps whose inputs come from elsewhere
        self.q_in = torch.empty((s, num_heads, d), dtype=k_cache.dtype, device=dev)
        self.k_in = torch.empty((s, hkv, d), dtype=k_cache.dtype, device=dev)
        self.v_in = torch.empty((s, hkv, d), dtype=k_cache.dtype, device=dev)
        self.out = torch.empty((s, num_heads, d), dtype=k_cache.dtype, device=dev)
        self._pool = None

    def _views(self, buf):
        s, w = self.num_seqs, self.width
        o_plan, o_slots, o_ctx, o_cow, o_tab = self._layout
        plan = buf[o_plan:o_slots]
        slots = buf[o_slots:o_slots + 8 * s].view(torch.int64)
        ctx = buf[o_ctx:o_ctx + 4 * s].view(torch.int32)
        cow = buf[o_cow:o_cow + 8 * s].view(torch.int32).view(s, 2)
        tables = buf[o_tab:o_tab + 4 * s * w].view(torch.int32).view(s, w)
        return plan, slots, ctx, cow, tables

    def __del__(self):
        st = getattr(self, "_st", None)
        try:
            if st and st.value and _libmod._lib is not None:
                torch.cuda.synchronize()
                _libmod._lib.pa_stepper_destroy(st)
                self._st = ctypes.c_void_p(0)
        except Exception:  # interpreter shutdown
            pass

    def context_lens(self) -> np.ndarray:
        return self.ctx_h.numpy().copy()

    # -- host part ---------------------------------------------------------
    def _prepare(self) -> int:
        """Reserve every sequence's next slot, build the work list, upload
        everything to device buffer ``k`` on the side stream, make the main
        stream wait for it and queue the block copies.  Returns their number."""
        main = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        check(_libmod._lib.pa_stepper_prepare(self._st, self._up_ptr, main, ctypes.byref(self._bi),
                                              ctypes.byref(self._nc)))
        self.k = k = self._bi.value
        ncow = self._nc.value
        if ncow:
            ops.copy_blocks(self.k_cache, self.v_cache, self._dv[k][3][:ncow])
            self.launches += 1
        return ncow

    def _finish(self) -> None:
        check(_libmod._lib.pa_stepper_finish(self._st, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)))
        self.k ^= 1
        self.launches += self._per_step

    # -- main-stream part (capturable) ---------------------------------------
    def _device(self, k, q, k_new, v_new, out, events=None):
        plan, slots, ctx, _, tables = self._dv[k]
        ops.cache_append(k_new, v_new, slots, self.k_cache, self.v_cache)
        if events is not None:
            events[0].record()
        if self.bf16:
            out = ops.paged_decode_planned(q, self.k_cache, self.v_cache, tables, ctx, self.max_context_len,
                                           self.scale, out, plan, self.workspace, self.partition_size)
        else:
            out = ops.paged_decode(q, self.k_cache, self.v_cache, tables, ctx, self.max_context_len, self.scale,
                                   out=out, partition_size=self.partition_size, workspace=self.workspace)
        if events is not None:
            events[1].record()
        return out

    def step(self, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor, out: torch.Tensor | None = None,
             events=None):
        """One decode step for every sequence: q ``[S, H, D]``, k_new/v_new
        ``[S, Hkv, D]`` on the device.  Returns ``out [S, H, D]``.
        ``events`` (a pair of CUDA events) are recorded around the decode."""
        if out is None:
            out = torch.empty_like(q)
        self._prepare()
        out = self._device(self.k, q, k_new, v_new, out, events)
        self._finish()
        return out

    def capture(self, events=None, inputs=None) -> StepGraphs:
        """Capture the main-stream part of a step (append, decode, merge) as
        CUDA graphs, one per device buffer.  ``inputs`` = (q, k_new, v_new,
        out) device tensors the graphs read and write (default: the
        engine's staging buffers ``q_in, k_in, v_in, out``).  ``events``, if
        given, are recorded around the decode at every replay (timing events
        created with ``external``).  Call after at least one eager step."""
        if not graphs_supported():
            raise RuntimeError("this torch cannot record events inside a CUDA graph")
        q, kn, vn, out = inputs if inputs is not None else (self.q_in, self.k_in, self.v_in, self.out)
        if self._pool is None:
            self._pool = torch.cuda.graph_pool_handle()
        torch.cuda.synchronize()
        graphs = []
        for k in range(2):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, pool=self._pool):
                self._device(k, q, kn, vn, out, events)
            graphs.append(g)
        torch.cuda.synchronize()
        return StepGraphs(graphs)

    def replay(self, graphs: StepGraphs, q=None, k_new=None, v_new=None) -> torch.Tensor:
        """One step through captured graphs.  New tokens given here are
        copied into the staging buffers first (graphs captured on other
        inputs need none)."""
        self._prepare()
        for src, dst in ((q, self.q_in), (k_new, self.k_in), (v_new, self.v_in)):
            if src is not None and src.data_ptr() != dst.data_ptr():
                dst.copy_(src, non_blocking=True)
        graphs.graphs[self.k].replay()
        self._finish()
        return self.out

    def step_host(self, q_h: torch.Tensor, k_h: torch.Tensor, v_h: torch.Tensor, out_h: torch.Tensor,
                  graphs: StepGraphs | None = None) -> torch.Tensor:
        """Same step with host (pinned) inputs and output: the new tokens are
        copied into the staging buffers, the output back to ``out_h``.
        ``graphs`` must have been captured on the staging buffers."""
        self._prepare()
        self.q_in.copy_(q_h, non_blocking=True)
        self.k_in.copy_(k_h, non_blocking=True)
        self.v_in.copy_(v_h, non_blocking=True)
        if graphs is None:
            self._device(self.k, self.q_in, self.k_in, self.v_in, self.out)
        else:
            graphs.graphs[self.k].replay()
        self._finish()
        out_h.copy_(self.out, non_blocking=True)
        return out_h
