"""Shared set-up for the GPU parity tests: seeded inputs from ``workloads``,
the oracle's view (its own allocator, numpy caches) and the CUDA path's view
(C++ allocator, device tensors) of the same workload."""

from __future__ import annotations

import dataclasses

import numpy as np
import torch

from oracle.attention import paged_decode as oracle_decode
from oracle.cache import copy_blocks as oracle_copy_blocks
from oracle.serving import initial_state, tables_array
from workloads import Workload, context_lens, free_order, pool_blocks, queries, random_pool

BF16_ATOL, BF16_RTOL = 2e-2, 1e-2
F32_ATOL, F32_RTOL = 1e-5, 1e-5


def to_dev(a: np.ndarray, device="cuda") -> torch.Tensor:
    """numpy array (bf16 bit patterns as uint16, or fp32) -> device tensor."""
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def to_bits(t: torch.Tensor) -> np.ndarray:
    """device tensor -> numpy (bf16 as uint16 bit patterns)."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def as_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def assert_close(got: torch.Tensor, ref: np.ndarray, dtype: str, what: str = ""):
    g = as_f64(got)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    atol, rtol = (BF16_ATOL, BF16_RTOL) if dtype == "bf16" else (F32_ATOL, F32_RTOL)
    err = np.abs(g - ref)
    bound = atol + rtol * np.abs(ref)
    bad = ~(err <= bound)
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} of {err.size} outside tolerance; worst at {i}: "
                             f"got {g[i]!r} ref {ref[i]!r} (max abs err {err.max():.3g})")


@dataclasses.dataclass
class DecodeCase:
    w: Workload
    ctx: np.ndarray
    num_blocks: int
    k_pool: np.ndarray  # oracle's caches (CoW copies applied)
    v_pool: np.ndarray
    q: np.ndarray
    tables: np.ndarray  # oracle allocator's tables, -1 padded
    max_ctx: int
    # device side
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    q_d: torch.Tensor
    tables_d: torch.Tensor
    ctx_d: torch.Tensor

    def oracle(self, seqs=None) -> np.ndarray:
        return oracle_decode(self.q, self.k_pool, self.v_pool, self.tables, self.ctx, self.w.scale, self.w.dtype,
                             seqs)


def make_decode_case(w: Workload, ctx: np.ndarray | None = None, prefix_len: int | None = None,
                     device="cuda", extra_blocks: int = 0) -> DecodeCase:
    import paged_kv_cache_216_gb300 as pa
    from paged_kv_cache_216_gb300.prefix import populate

    ctx = context_lens(w) if ctx is None else np.asarray(ctx, dtype=np.int32)
    plen = w.prefix_len if prefix_len is None else prefix_len
    nb = pool_blocks(w, ctx) + w.prefix_share + extra_blocks
    order = free_order(w, nb)
    k_pool = random_pool(w, nb, "k")
    v_pool = random_pool(w, nb, "v")
    q = queries(w)
    width = -(-int(ctx.max()) // w.block_size)
    # CUDA path: C++ allocator, device caches, device block copies
    c = pa.BlockAllocator(nb, w.block_size, order)
    cpairs = populate(c, ctx, plen, w.prefix_share)
    seq_ids = np.arange(w.num_seqs, dtype=np.int64)
    tables_c = np.empty((w.num_seqs, width), dtype=np.int32)
    ctx_c = np.empty(w.num_seqs, dtype=np.int32)
    c.block_tables(seq_ids, tables_c, ctx_c)
    k_cache = to_dev(k_pool, device)
    v_cache = to_dev(v_pool, device)
    if len(cpairs):
        pa.copy_blocks(k_cache, v_cache, to_dev(cpairs, device))
    # oracle: its own allocator and copies on the host arrays
    o, opairs = initial_state(w.num_seqs, w.block_size, ctx, nb, order, plen, w.prefix_share)
    oracle_copy_blocks(k_pool, v_pool, opairs)
    tables_o = tables_array(o, range(w.num_seqs), width)
    assert np.array_equal(tables_o, tables_c) and np.array_equal(ctx_c, ctx)
    return DecodeCase(w=w, ctx=ctx, num_blocks=nb, k_pool=k_pool, v_pool=v_pool, q=q, tables=tables_o,
                      max_ctx=int(ctx.max()), k_cache=k_cache, v_cache=v_cache, q_d=to_dev(q, device),
                      tables_d=to_dev(tables_c, device), ctx_d=to_dev(ctx_c, device))


def run_decode(case: DecodeCase, partition_size: int | None = None, max_ctx: int | None = None):
    import paged_kv_cache_216_gb300 as pa

    w = case.w
    p = w.partition_size if partition_size is None else partition_size
    return pa.paged_decode(case.q_d, case.k_cache, case.v_cache, case.tables_d, case.ctx_d,
                           case.max_ctx if max_ctx is None else max_ctx, w.scale, partition_size=p)
