"""Tensor-level calls of the C ABI: KV append, block copy, paged decode.

Each function checks shapes/dtypes/devices of its torch tensors, passes raw
device pointers and sizes to libpa.so on the current CUDA stream, and raises
on a non-zero return code.  Nothing here computes any part of the method.
"""

from __future__ import annotations

import ctypes

import numpy as np
import torch

from ._lib import PA_BF16, PA_F32, PA_FP8_E4M3, check, lib

_DTYPES = {torch.bfloat16: PA_BF16, torch.float32: PA_F32, torch.uint8: PA_FP8_E4M3}
_FP8 = getattr(torch, "float8_e4m3fn", None)
if _FP8 is not None:
    _DTYPES[_FP8] = PA_FP8_E4M3


def is_fp8(t: torch.Tensor) -> bool:
    """Whether ``t`` holds E4M3 codes (float8_e4m3fn, or uint8 codes)."""
    return _DTYPES.get(t.dtype) == PA_FP8_E4M3


def _dtype_code(t: torch.Tensor) -> int:
    try:
        return _DTYPES[t.dtype]
    except KeyError:
        raise TypeError(f"unsupported dtype {t.dtype}: bfloat16, float32 or E4M3 codes") from None


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need(cond: bool, msg: str):
    if not cond:
        raise ValueError(msg)


def _cuda_contig(*ts):
    for t in ts:
        _need(t.is_cuda and t.is_contiguous(), "tensors must be contiguous CUDA tensors")


def cache_append(k, v, slot_mapping, k_cache, v_cache, stream=None) -> None:
    """Write new tokens' keys/values ``k, v [T, Hkv, D]`` into slots
    ``slot_mapping [T]`` (int64; negative = skip) of ``k_cache, v_cache
    [N, Hkv, B, D]``, in place."""
    _cuda_contig(k, v, slot_mapping, k_cache, v_cache)
    _need(slot_mapping.dtype == torch.int64, "slot_mapping must be int64")
    _need(k.dtype == v.dtype == k_cache.dtype == v_cache.dtype, "k, v and caches must share a dtype")
    n, hkv, b, d = k_cache.shape
    _need(v_cache.shape == k_cache.shape, "k_cache and v_cache shapes differ")
    t = slot_mapping.shape[0]
    _need(tuple(k.shape) == (t, hkv, d) and tuple(v.shape) == (t, hkv, d), "k, v must be [T, Hkv, D]")
    check(lib().pa_cache_append(_ptr(k), _ptr(v), _ptr(slot_mapping), t, _ptr(k_cache), _ptr(v_cache),
                                n, hkv, d, b, _dtype_code(k_cache), _stream(stream)))


def cache_append_fp8(k, v, slot_mapping, k_cache, v_cache, k_scale: float, v_scale: float, stream=None) -> None:
    """:func:`cache_append` into E4M3 caches (float8_e4m3fn or uint8
    ``[N, Hkv, B, D]``): the bf16 tokens are stored as round-to-nearest-even
    E4M3 codes of x / scale, saturating at ±448."""
    _cuda_contig(k, v, slot_mapping, k_cache, v_cache)
    _need(slot_mapping.dtype == torch.int64, "slot_mapping must be int64")
    _need(k.dtype == v.dtype == torch.bfloat16, "k and v must be bfloat16")
    _need(is_fp8(k_cache) and is_fp8(v_cache), "caches must hold E4M3 codes")
    n, hkv, b, d = k_cache.shape
    _need(v_cache.shape == k_cache.shape, "k_cache and v_cache shapes differ")
    t = slot_mapping.shape[0]
    _need(tuple(k.shape) == (t, hkv, d) and tuple(v.shape) == (t, hkv, d), "k, v must be [T, Hkv, D]")
    check(lib().pa_cache_append_fp8(_ptr(k), _ptr(v), _ptr(slot_mapping), t, _ptr(k_cache), _ptr(v_cache), n, hkv,
                                    d, b, float(k_scale), float(v_scale), _stream(stream)))


def copy_blocks(k_cache, v_cache, pairs, stream=None) -> None:
    """For each (src, dst) row of ``pairs [n, 2]`` (int32, device) copy block
    src to block dst in both caches."""
    _cuda_contig(k_cache, v_cache, pairs)
    _need(pairs.dtype == torch.int32 and pairs.dim() == 2 and pairs.shape[1] == 2, "pairs must be int32 [n, 2]")
    n, hkv, b, d = k_cache.shape
    check(lib().pa_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(pairs), pairs.shape[0], n, hkv, d, b,
                               _dtype_code(k_cache), _stream(stream)))


def decode_partition_size(num_seqs: int, num_kv_heads: int, max_context_len: int, partition_size: int = 0,
                          prefix_groups=None) -> int:
    """The partition size a decode call uses (the library's choice for 0);
    with prefix groups, the one the shared-prefix calls use."""
    g = prefix_groups_array(prefix_groups)
    if g is None:
        return check(lib().pa_decode_partition_size(num_seqs, num_kv_heads, max_context_len, partition_size))
    return check(lib().pa_decode_partition_size_shared_prefix(num_seqs, num_kv_heads, max_context_len,
                                                              partition_size, ctypes.c_void_p(g.ctypes.data),
                                                              g.shape[0]))


def decode_workspace_bytes(num_seqs: int, num_heads: int, head_dim: int, max_context_len: int,
                           partition_size: int) -> int:
    return int(lib().pa_decode_workspace_bytes(num_seqs, num_heads, head_dim, max_context_len, partition_size))


def decode_workspace(num_seqs, num_heads, num_kv_heads, head_dim, max_context_len, partition_size=0,
                     device="cuda"):
    """Allocate (with torch) the workspace pa_decode needs for these sizes;
    None when no workspace is needed."""
    p = decode_partition_size(num_seqs, num_kv_heads, max_context_len, partition_size)
    nbytes = decode_workspace_bytes(num_seqs, num_heads, head_dim, max_context_len, p)
    if nbytes == 0:
        return None
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def paged_decode(q, k_cache, v_cache, block_tables, context_lens, max_context_len: int, scale: float,
                 out=None, partition_size: int = 0, workspace=None, stream=None):
    """out[s, h] = softmax(scale * K_s q[s, h]) V_s over each sequence's
    blocks.  q ``[S, H, D]``; caches ``[N, Hkv, B, D]``; block_tables
    ``[S, max_blocks]`` int32; context_lens ``[S]`` int32 (device);
    ``max_context_len`` a host bound of context_lens.  Returns ``out``."""
    _cuda_contig(q, k_cache, v_cache, block_tables, context_lens)
    _need(q.dtype == k_cache.dtype == v_cache.dtype, "q and caches must share a dtype")
    _need(block_tables.dtype == torch.int32 and context_lens.dtype == torch.int32,
          "block_tables and context_lens must be int32")
    s, h, d = q.shape
    n, hkv, b, d2 = k_cache.shape
    _need(d == d2 and v_cache.shape == k_cache.shape, "head_dim mismatch")
    _need(block_tables.dim() == 2 and block_tables.shape[0] == s and context_lens.shape == (s,),
          "block_tables [S, max_blocks], context_lens [S]")
    if out is None:
        out = torch.empty_like(q)
    _cuda_contig(out)
    _need(out.shape == q.shape and out.dtype == q.dtype, "out must match q")
    if workspace is None:
        workspace = decode_workspace(s, h, hkv, d, max_context_len, partition_size, q.device)
    ws_ptr = _ptr(workspace)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    check(lib().pa_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), block_tables.shape[1],
                          _ptr(context_lens), int(max_context_len), float(scale), _ptr(out), s, h, hkv, d, b, n,
                          int(partition_size), ws_ptr, ws_bytes, _dtype_code(q), _stream(stream)))
    return out


def prefix_groups_array(groups):
    """Prefix groups as the C ABI takes them: a C-contiguous int32 array
    ``[n, 3]`` of (first sequence, number of sequences, shared prefix
    tokens), or None for no groups."""
    if groups is None:
        return None
    g = np.ascontiguousarray(np.asarray(groups, dtype=np.int32).reshape(-1, 3))
    return g if g.shape[0] else None


def _groups_args(groups):
    g = prefix_groups_array(groups)
    return (ctypes.c_void_p(g.ctypes.data) if g is not None else None), (0 if g is None else g.shape[0]), g


def prefill(q, k, v, slot_mapping, query_start, context_lens, block_tables, max_query_len: int,
            max_context_len: int, scale: float, k_cache, v_cache, out=None, stream=None):
    """Append the new tokens ``k, v [T, Hkv, D]`` at ``slot_mapping`` and
    return causal attention ``[T, H, D]`` of their queries ``q``: sequence s
    owns rows ``query_start[s] .. query_start[s+1]-1`` (int32, device) and
    has ``context_lens[s]`` tokens after the append; each new token attends
    the sequence's tokens up to its own position.  bf16."""
    _cuda_contig(q, k, v, slot_mapping, query_start, context_lens, block_tables, k_cache, v_cache)
    _need(q.dtype == k.dtype == v.dtype == k_cache.dtype == v_cache.dtype == torch.bfloat16, "bf16 only")
    _need(slot_mapping.dtype == torch.int64, "slot_mapping must be int64")
    _need(query_start.dtype == context_lens.dtype == block_tables.dtype == torch.int32,
          "query_start, context_lens and block_tables must be int32")
    t, h, d = q.shape
    n, hkv, b, d2 = k_cache.shape
    _need(d == d2 and tuple(k.shape) == (t, hkv, d) and v.shape == k.shape, "shapes")
    s = context_lens.shape[0]
    _need(query_start.shape == (s + 1,) and block_tables.shape[0] == s, "query_start [S+1], block_tables [S, ...]")
    if out is None:
        out = torch.empty_like(q)
    _cuda_contig(out)
    check(lib().pa_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(slot_mapping), t, _ptr(query_start), _ptr(context_lens),
                           _ptr(block_tables), block_tables.shape[1], int(max_query_len), int(max_context_len),
                           float(scale), _ptr(k_cache), _ptr(v_cache), _ptr(out), s, h, hkv, d, b, n, PA_BF16,
                           _stream(stream)))
    return out


def paged_decode_fp8(q, k_cache, v_cache, block_tables, context_lens, max_context_len: int, scale: float,
                     k_scale: float, v_scale: float, out=None, partition_size: int = 0, workspace=None, plan=None,
                     stream=None):
    """:func:`paged_decode` over E4M3 caches written by
    :func:`cache_append_fp8`: keys read as code · k_scale, values as
    code · v_scale; q and out bf16, head_dim 128.  ``plan``: a work list
    from :func:`decode_plan_host` copied to the device (counter at 0), or
    None to build it on the device."""
    _cuda_contig(q, k_cache, v_cache, block_tables, context_lens)
    _need(q.dtype == torch.bfloat16, "q must be bfloat16")
    _need(is_fp8(k_cache) and is_fp8(v_cache), "caches must hold E4M3 codes")
    _need(block_tables.dtype == torch.int32 and context_lens.dtype == torch.int32,
          "block_tables and context_lens must be int32")
    s, h, d = q.shape
    n, hkv, b, d2 = k_cache.shape
    _need(d == d2 and v_cache.shape == k_cache.shape, "head_dim mismatch")
    if out is None:
        out = torch.empty_like(q)
    _cuda_contig(out)
    _need(out.shape == q.shape and out.dtype == q.dtype, "out must match q")
    if workspace is None:
        workspace = decode_workspace(s, h, hkv, d, max_context_len, partition_size, q.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    check(lib().pa_decode_fp8(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), block_tables.shape[1],
                              _ptr(context_lens), int(max_context_len), float(scale), float(k_scale),
                              float(v_scale), _ptr(out), s, h, hkv, d, b, n, int(partition_size), _ptr(plan),
                              _ptr(workspace), ws_bytes, _stream(stream)))
    return out


def paged_decode_shared_prefix(q, k_cache, v_cache, block_tables, context_lens, max_context_len: int, scale: float,
                               prefix_groups, out=None, partition_size: int = 0, workspace=None, stream=None):
    """:func:`paged_decode` for batches where groups of sequences share the
    blocks of a prefix: ``prefix_groups`` rows (first sequence, number of
    sequences, shared prefix tokens).  The whole partitions of each prefix
    are attended by work items that cover several members at once; the
    result is that of :func:`paged_decode`.  bf16 only."""
    _cuda_contig(q, k_cache, v_cache, block_tables, context_lens)
    _need(q.dtype == k_cache.dtype == v_cache.dtype, "q and caches must share a dtype")
    _need(block_tables.dtype == torch.int32 and context_lens.dtype == torch.int32,
          "block_tables and context_lens must be int32")
    s, h, d = q.shape
    n, hkv, b, d2 = k_cache.shape
    _need(d == d2 and v_cache.shape == k_cache.shape, "head_dim mismatch")
    _need(block_tables.dim() == 2 and block_tables.shape[0] == s and context_lens.shape == (s,),
          "block_tables [S, max_blocks], context_lens [S]")
    if out is None:
        out = torch.empty_like(q)
    _cuda_contig(out)
    _need(out.shape == q.shape and out.dtype == q.dtype, "out must match q")
    if workspace is None:
        p = decode_partition_size(s, hkv, max_context_len, partition_size, prefix_groups)
        workspace = decode_workspace(s, h, hkv, d, max_context_len, p, q.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    gp, gn, _keep = _groups_args(prefix_groups)
    check(lib().pa_decode_shared_prefix(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                        block_tables.shape[1], _ptr(context_lens), int(max_context_len),
                                        float(scale), _ptr(out), s, h, hkv, d, b, n, int(partition_size), gp, gn,
                                        _ptr(workspace), ws_bytes, _dtype_code(q), _stream(stream)))
    return out


def decode_plan_bytes(num_seqs: int, max_context_len: int, partition_size: int) -> int:
    return int(lib().pa_decode_plan_bytes(num_seqs, max_context_len, partition_size))


def decode_plan_host(context_lens, max_context_len: int, partition_size: int, plan, prefix_groups=None,
                     num_heads: int = 1, num_kv_heads: int = 1) -> None:
    """Build the decode work list on the host into ``plan`` (a host buffer
    of decode_plan_bytes(...) bytes, numpy or a CPU tensor) from the int32
    host array ``context_lens``; with ``prefix_groups`` (and the decode's
    head counts), the list for :func:`paged_decode_planned` with the same
    groups."""
    ptr = plan.ctypes.data if hasattr(plan, "ctypes") else plan.data_ptr()
    cptr = context_lens.ctypes.data if hasattr(context_lens, "ctypes") else context_lens.data_ptr()
    gp, gn, _keep = _groups_args(prefix_groups)
    if gn:
        check(lib().pa_decode_plan_host_shared_prefix(ctypes.c_void_p(cptr), len(context_lens),
                                                      int(max_context_len), int(partition_size), int(num_heads),
                                                      int(num_kv_heads), gp, gn, ctypes.c_void_p(ptr)))
    else:
        check(lib().pa_decode_plan_host(ctypes.c_void_p(cptr), len(context_lens), int(max_context_len),
                                        int(partition_size), ctypes.c_void_p(ptr)))


def paged_decode_planned(q, k_cache, v_cache, block_tables, context_lens, max_context_len: int, scale: float,
                         out, plan, workspace, partition_size: int, stream=None, prefix_groups=None):
    """:func:`paged_decode` with a work list built by :func:`decode_plan_host`
    and copied to the device (``plan``, uint8, counter at 0; consumed by the
    call).  With ``prefix_groups`` (the groups the list was built with) it
    is :func:`paged_decode_shared_prefix`."""
    s, h, d = q.shape
    n, hkv, b, _ = k_cache.shape
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    gp, gn, _keep = _groups_args(prefix_groups)
    if gn:
        check(lib().pa_decode_planned_shared_prefix(
            _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), block_tables.shape[1], _ptr(context_lens),
            int(max_context_len), float(scale), _ptr(out), s, h, hkv, d, b, n, int(partition_size), gp, gn,
            _ptr(plan), _ptr(workspace), ws_bytes, _dtype_code(q), _stream(stream)))
        return out
    check(lib().pa_decode_planned(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), block_tables.shape[1],
                                  _ptr(context_lens), int(max_context_len), float(scale), _ptr(out), s, h, hkv, d, b,
                                  n, int(partition_size), _ptr(plan), _ptr(workspace), ws_bytes, _dtype_code(q),
                                  _stream(stream)))
    return out


def paged_decode_static_workspace(q, k_cache, v_cache, block_tables, context_lens, max_context_len: int,
                                  scale: float, out, partition_size: int = 0, stream=None):
    """Same as :func:`paged_decode`, for callers that cannot allocate a
    workspace: the split-K scratch is the library's fixed device array
    (``PA_STATIC_WORKSPACE_BYTES``), shared by every call.  ``out`` must be
    given, so this call allocates nothing.  Calls whose kernels overlap on
    the GPU race on the shared array."""
    _cuda_contig(q, k_cache, v_cache, block_tables, context_lens, out)
    _need(q.dtype == k_cache.dtype == v_cache.dtype == out.dtype, "q, caches and out must share a dtype")
    _need(block_tables.dtype == torch.int32 and context_lens.dtype == torch.int32,
          "block_tables and context_lens must be int32")
    s, h, d = q.shape
    n, hkv, b, _ = k_cache.shape
    _need(out.shape == q.shape, "out must match q")
    check(lib().pa_decode_static_workspace(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                           block_tables.shape[1], _ptr(context_lens), int(max_context_len),
                                           float(scale), _ptr(out), s, h, hkv, d, b, n, int(partition_size),
                                           _dtype_code(q), _stream(stream)))
    return out


def get_status(stream=None) -> int:
    """Read and clear the device status word (synchronizes the stream)."""
    v = ctypes.c_uint32(0)
    check(lib().pa_get_status(_stream(stream), ctypes.byref(v)))
    return int(v.value)
