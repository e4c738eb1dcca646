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
                 num_heads: int, scale: float, max_context_len: int, partition_size: int = 0, prefix_groups=None,
                 kv_scales=None):
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
        self.partition_size = ops.decode_partition_size(
            s, hkv, self.max_context_len, partition_size,
            prefix_groups if k_cache.dtype == torch.bfloat16 else None)
        self.bf16 = k_cache.dtype == torch.bfloat16
        # E4M3 caches: new tokens arrive in bf16 and are stored as codes of
        # x / scale; kv_scales = (k_scale, v_scale).
        self.fp8 = ops.is_fp8(k_cache)
        if self.fp8:
            if kv_scales is None:
                raise ValueError("E4M3 caches need kv_scales=(k_scale, v_scale)")
            self.k_scale, self.v_scale = (float(x) for x in kv_scales)
        tok_dtype = torch.bfloat16 if self.fp8 else k_cache.dtype
        plan_p = self.partition_size if (self.bf16 or self.fp8) else 0
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
        # Groups of the batch that share a prefix's blocks (rows: first
        # position, count, prefix tokens): their shared partitions are
        # attended by work items covering several members each (bf16).
        self.prefix_groups = ops.prefix_groups_array(prefix_groups)
        if self.prefix_groups is not None:
            if not self.bf16:
                raise ValueError("prefix groups need bf16 caches")
            g = self.prefix_groups
            check(lib().pa_stepper_set_prefix_groups(self._st, ctypes.c_void_p(g.ctypes.data), g.shape[0],
                                                     num_heads, hkv))
        self.workspace = ops.decode_workspace(s, num_heads, hkv, d, self.max_context_len, self.partition_size, dev)
        self.up_stream = torch.cuda.Stream(device=dev)
        self._up_ptr = ctypes.c_void_p(self.up_stream.cuda_stream)
        self._bi = ctypes.c_int(0)
        self._nc = ctypes.c_int(0)
        self.k = 0  # device buffer of the next step
        self.launches = 0  # kernels this engine has launched
        self.split = -(-self.max_context_len // self.partition_size) > 1
        self._per_step = 2 + (1 if self.split else 0)  # append + decode (+ merge)
        # staging buffers (one set per device buffer) for steps whose inputs
        # come from elsewhere, and the streams/events of host transfers
        # staging per device buffer: the step's new tokens packed as [q | k | v]
        self._nq, self._nk = s * num_heads * d, s * hkv * d
        self._stg = [torch.empty(self._nq + 2 * self._nk, dtype=tok_dtype, device=dev) for _ in range(2)]
        self.q_in = [x[:self._nq].view(s, num_heads, d) for x in self._stg]
        self.k_in = [x[self._nq:self._nq + self._nk].view(s, hkv, d) for x in self._stg]
        self.v_in = [x[self._nq + self._nk:].view(s, hkv, d) for x in self._stg]
        self.out = [torch.empty((s, num_heads, d), dtype=tok_dtype, device=dev) for _ in range(2)]
        self.down_stream = torch.cuda.Stream(device=dev)
        self._tok_done = [torch.cuda.Event(), torch.cuda.Event()]
        self._step_done = [torch.cuda.Event(), torch.cuda.Event()]
        self._out_read = [torch.cuda.Event(), torch.cuda.Event()]
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
        if self.fp8:
            ops.cache_append_fp8(k_new, v_new, slots, self.k_cache, self.v_cache, self.k_scale, self.v_scale)
        else:
            ops.cache_append(k_new, v_new, slots, self.k_cache, self.v_cache)
        if events is not None:
            events[0].record()
        if self.fp8:
            out = ops.paged_decode_fp8(q, self.k_cache, self.v_cache, tables, ctx, self.max_context_len, self.scale,
                                       self.k_scale, self.v_scale, out=out, partition_size=self.partition_size,
                                       workspace=self.workspace, plan=plan)
        elif self.bf16:
            out = ops.paged_decode_planned(q, self.k_cache, self.v_cache, tables, ctx, self.max_context_len,
                                           self.scale, out, plan, self.workspace, self.partition_size,
                                           prefix_groups=self.prefix_groups)
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

    def capture(self, events=None, inputs=None, parity=None) -> StepGraphs:
        """Capture the main-stream part of a step (append, decode, merge) as
        CUDA graphs, one per device buffer (or only for device buffer
        ``parity``).  ``inputs`` = (q, k_new, v_new, out) device tensors the
        graphs read and write (default: the engine's staging buffers of each
        device buffer).  ``events``, if given, are recorded around the
        decode at every replay (timing events created with ``external``).
        Call after at least one eager step."""
        if not graphs_supported():
            raise RuntimeError("this torch cannot record events inside a CUDA graph")
        if self._pool is None:
            self._pool = torch.cuda.graph_pool_handle()
        torch.cuda.synchronize()
        graphs = []
        for k in range(2):
            if parity is not None and k != parity:
                graphs.append(None)
                continue
            q, kn, vn, out = inputs if inputs is not None else (self.q_in[k], self.k_in[k], self.v_in[k],
                                                                self.out[k])
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, pool=self._pool):
                self._device(k, q, kn, vn, out, events)
            graphs.append(g)
        torch.cuda.synchronize()
        return StepGraphs(graphs)

    def pack_tokens(self, q, k_new, v_new, pin: bool = False) -> torch.Tensor:
        """One step's new tokens packed as the staging layout [q | k | v]
        (on the device, or in pinned host memory with ``pin``): a packed
        step is staged with a single copy."""
        flat = torch.cat([q.reshape(-1), k_new.reshape(-1), v_new.reshape(-1)])
        return flat.pin_memory() if pin else flat

    def _stage(self, k, q=None, k_new=None, v_new=None, packed=None) -> None:
        """Copy the step's new tokens (device or pinned host tensors; one
        packed tensor or three) into staging buffer k on the upload stream,
        after the step's tables, and make the main stream wait for them: the
        copies overlap the previous step's decode."""
        with torch.cuda.stream(self.up_stream):
            if packed is not None:
                self._stg[k].copy_(packed, non_blocking=True)
            for src, dst in ((q, self.q_in[k]), (k_new, self.k_in[k]), (v_new, self.v_in[k])):
                if src is not None and src.data_ptr() != dst.data_ptr():
                    dst.copy_(src, non_blocking=True)
            self._tok_done[k].record(self.up_stream)
        main = torch.cuda.current_stream()
        main.wait_event(self._tok_done[k])
        main.wait_event(self._out_read[k])  # the copy-out of the step that last wrote out[k]

    def replay(self, graphs: StepGraphs, q=None, k_new=None, v_new=None, packed=None) -> torch.Tensor:
        """One step through captured graphs, reading the new tokens from the
        staging buffers (copied there first when given here, as three
        tensors or one from :meth:`pack_tokens`).  Returns the output buffer
        the graph wrote."""
        if graphs.graphs[self.k] is None:
            raise ValueError("these graphs were captured for the other device buffer")
        self._prepare()
        k = self.k
        self._stage(k, q, k_new, v_new, packed)
        graphs.graphs[k].replay()
        self._finish()
        return self.out[k]

    def step_host(self, q_h=None, k_h=None, v_h=None, out_h: torch.Tensor | None = None,
                  graphs: StepGraphs | None = None, packed=None) -> torch.Tensor:
        """Same step with host (pinned) inputs and output: three tensors, or
        one packed by :meth:`pack_tokens` (``pin=True``).  The new tokens are
        copied on the upload stream after the step's tables, the output
        back on a third stream once the step is done, so both transfers
        overlap neighbouring steps; synchronize before reading ``out_h``.
        ``graphs`` must have been captured on the staging buffers."""
        self._prepare()
        k = self.k
        self._stage(k, q_h, k_h, v_h, packed)
        main = torch.cuda.current_stream()
        if graphs is None:
            self._device(k, self.q_in[k], self.k_in[k], self.v_in[k], self.out[k])
        else:
            graphs.graphs[k].replay()
        self._finish()
        self._step_done[k].record(main)
        self.down_stream.wait_event(self._step_done[k])
        with torch.cuda.stream(self.down_stream):
            out_h.copy_(self.out[k], non_blocking=True)
            self._out_read[k].record(self.down_stream)
        return out_h
