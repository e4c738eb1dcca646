"""Seeded synthetic decode workloads.

Every array here is drawn from numpy's PCG64 generator seeded through a
``SeedSequence([workload seed, stream tag])`` so that each purpose (context
lengths, free-list order, queries, key pool, value pool, per-step tokens) has
its own independent stream and any size can be regenerated on any machine.

Value distributions follow the decode workloads the method is measured on:
queries, keys and values are N(0, std^2), stored as bf16 (round to nearest
even) or fp32.  Large pools are filled from a seeded N(0, std^2) table, one
random window per (block, head) slab, with a per-slab random sign and low
mantissa pattern so that no two slabs are equal in practice; each element is
still N(0, std^2) up to bf16 rounding.

This module sizes buffers and draws random numbers only.  It does not
allocate blocks, map slots or compute attention.
"""

from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass, field

import numpy as np

# Stream tags: one independent random stream per purpose.
_TAG_CTX = 1
_TAG_FREE = 2
_TAG_Q = 3
_TAG_KPOOL = 4
_TAG_VPOOL = 5
_TAG_STEP = 1000  # + step index


@dataclass(frozen=True)
class Workload:
    """Shape and distribution of one decode workload.

    ``ctx_dist`` is one of ``fixed`` (``ctx_fixed``), ``uniform`` (integers in
    [ctx_lo, ctx_hi]), ``loguniform`` (exp(U(ln lo, ln hi)) rounded) or
    ``geometric`` (support 1, 2, ... with mean ``ctx_mean``, capped at
    ``ctx_hi``).  With ``prefix_len > 0`` the first ``prefix_share``
    sequences share one prefix of that many tokens and draw their lengths
    from [prefix_len + 1, ctx_hi].
    """

    name: str
    dtype: str  # "f32" or "bf16"
    num_seqs: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    seed: int
    std: float = 1.0
    ctx_dist: str = "uniform"
    ctx_lo: int = 1
    ctx_hi: int = 2048
    ctx_mean: float = 0.0
    ctx_fixed: tuple = field(default_factory=tuple)
    partition_size: int = 0  # 0: the library chooses
    pool_fixed: int = 0  # fixed pool size in blocks (0: sized from lengths)
    pool_slack: float = 0.10  # extra fraction of blocks in the pool
    prefix_len: int = 0
    prefix_share: int = 0
    steps: int = 0  # serving loop: decode steps, one appended token each

    @property
    def group(self) -> int:
        return self.num_heads // self.num_kv_heads

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


def _rng(seed: int, tag: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tag])))


WORKLOADS: dict[str, Workload] = {
    # 4 sequences, fp32, pool of 16 blocks in seeded random order.
    "tiny_f32": Workload(
        name="tiny_f32", dtype="f32", num_seqs=4, num_heads=4, num_kv_heads=4,
        head_dim=64, block_size=16, seed=0, ctx_dist="fixed",
        ctx_fixed=(1, 7, 16, 33), pool_fixed=16),
    # Multi-head attention, 32 sequences of uniform length in [1, 2048].
    "mha_bf16": Workload(
        name="mha_bf16", dtype="bf16", num_seqs=32, num_heads=32,
        num_kv_heads=32, head_dim=128, block_size=16, seed=1,
        ctx_dist="uniform", ctx_lo=1, ctx_hi=2048),
    # Grouped-query attention; half the batch shares one 1024-token prefix.
    "gqa_prefix_bf16": Workload(
        name="gqa_prefix_bf16", dtype="bf16", num_seqs=64, num_heads=32,
        num_kv_heads=8, head_dim=128, block_size=16, seed=2,
        ctx_dist="loguniform", ctx_lo=128, ctx_hi=8192, prefix_len=1024,
        prefix_share=32),
    # Long contexts split into 512-token partitions merged by log-sum-exp.
    "long_bf16": Workload(
        name="long_bf16", dtype="bf16", num_seqs=8, num_heads=64,
        num_kv_heads=8, head_dim=128, block_size=32, seed=3, std=0.5,
        ctx_dist="uniform", ctx_lo=32768, ctx_hi=131072, partition_size=512),
}
for _b in (8, 16, 32):
    # Serving loop: 256 sequences, geometric lengths (mean 1024, cap 4096),
    # 20 decode steps that each append one token per sequence.
    WORKLOADS[f"serving_bf16_b{_b}"] = Workload(
        name=f"serving_bf16_b{_b}", dtype="bf16", num_seqs=256, num_heads=32,
        num_kv_heads=8, head_dim=128, block_size=_b, seed=4,
        ctx_dist="geometric", ctx_mean=1024.0, ctx_hi=4096, steps=20)


def context_lens(w: Workload) -> np.ndarray:
    """Initial context length of every sequence (int32, all >= 1)."""
    rng = _rng(w.seed, _TAG_CTX)
    s = w.num_seqs
    if w.ctx_dist == "fixed":
        out = np.asarray(w.ctx_fixed, dtype=np.int64)
        assert out.shape == (s,)
    elif w.ctx_dist == "uniform":
        out = rng.integers(w.ctx_lo, w.ctx_hi + 1, size=s)
    elif w.ctx_dist == "loguniform":
        lo = np.full(s, float(w.ctx_lo))
        lo[: w.prefix_share] = float(w.prefix_len + 1)
        u = rng.uniform(0.0, 1.0, size=s)
        x = np.exp(np.log(lo) + u * (np.log(float(w.ctx_hi)) - np.log(lo)))
        out = np.clip(np.rint(x), lo, w.ctx_hi)
    elif w.ctx_dist == "geometric":
        out = np.minimum(rng.geometric(1.0 / w.ctx_mean, size=s), w.ctx_hi)
    else:
        raise ValueError(w.ctx_dist)
    out = np.asarray(out, dtype=np.int64)
    if w.prefix_share:
        assert np.all(out[: w.prefix_share] > w.prefix_len)
    assert np.all(out >= 1)
    return out.astype(np.int32)


def _cdiv(a, b):
    return -(-a // b)


def pool_blocks(w: Workload, ctx: np.ndarray, extra_steps: int | None = None) -> int:
    """Number of physical blocks in the pool: what the workload holds at its
    peak (shared prefix counted once, plus room for ``extra_steps`` appended
    tokens per sequence), plus ``pool_slack`` of spare blocks."""
    if w.pool_fixed:
        return w.pool_fixed
    b = w.block_size
    steps = w.steps if extra_steps is None else extra_steps
    ctx = np.asarray(ctx, dtype=np.int64)
    if w.prefix_share:
        share = ctx[: w.prefix_share]
        need = _cdiv(w.prefix_len, b) + int(np.sum(_cdiv(share, b) - w.prefix_len // b))
        need += int(np.sum(_cdiv(ctx[w.prefix_share:], b)))
    else:
        need = int(np.sum(_cdiv(ctx, b)))
    if steps:
        need += w.num_seqs * (_cdiv(steps, b) + 1)
    return int(math.ceil(need * (1.0 + w.pool_slack)))


def free_order(w: Workload, num_blocks: int) -> np.ndarray:
    """Seeded permutation of the pool: the order in which a fresh free list
    hands out blocks (element 0 first)."""
    return _rng(w.seed, _TAG_FREE).permutation(num_blocks).astype(np.int32)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    r = r.astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        r[nan] = 0x7FC0
    return r


def normal(shape, std: float, dtype: str, seed: int, tag: int) -> np.ndarray:
    """N(0, std^2) array: float32, or bf16 bits (uint16) for ``bf16``."""
    x = _rng(seed, tag).standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return bf16_bits(x) if dtype == "bf16" else x


def queries(w: Workload, tag_offset: int = 0) -> np.ndarray:
    return normal((w.num_seqs, w.num_heads, w.head_dim), w.std, w.dtype, w.seed, _TAG_Q + tag_offset)


_DIRECT_LIMIT = 1 << 22  # elements drawn directly; above this, table windows


def random_pool(w: Workload, num_blocks: int, which: str) -> np.ndarray:
    """Key ("k") or value ("v") pool ``[num_blocks, Hkv, B, D]`` of
    N(0, std^2) values (bf16 bits or fp32)."""
    tag = _TAG_KPOOL if which == "k" else _TAG_VPOOL
    shape = (num_blocks, w.num_kv_heads, w.block_size, w.head_dim)
    n = int(np.prod(shape))
    if n <= _DIRECT_LIMIT:
        return normal(shape, w.std, w.dtype, w.seed, tag)
    rng = _rng(w.seed, tag)
    slab = w.block_size * w.head_dim
    nslab = num_blocks * w.num_kv_heads
    table_len = (1 << 24) + slab
    table = rng.standard_normal(size=table_len, dtype=np.float32)
    if w.std != 1.0:
        table *= np.float32(w.std)
    if w.dtype == "bf16":
        table = bf16_bits(table)
        flip = np.uint16(0x8000)
        low = np.uint16(0x0007)
    else:
        table = table.view(np.uint32)
        flip = np.uint32(0x80000000)
        low = np.uint32(0x0000001F)
    offs = rng.integers(0, table_len - slab + 1, size=nslab)
    mask = rng.integers(0, 1 << 16, size=nslab).astype(table.dtype)
    mask = (mask & (flip | low))
    win = np.lib.stride_tricks.sliding_window_view(table, slab)
    out = np.empty((nslab, slab), dtype=table.dtype)
    step = 4096
    for i in range(0, nslab, step):
        j = min(nslab, i + step)
        out[i:j] = win[offs[i:j]]
        out[i:j] ^= mask[i:j, None]
    out = out.reshape(shape)
    return out if w.dtype == "bf16" else out.view(np.float32)


def serving_step_tokens(w: Workload, step: int):
    """New token of every sequence at serving step ``step``: its query
    ``[S, H, D]`` and its key and value ``[S, Hkv, D]``."""
    s, h, hk, d = w.num_seqs, w.num_heads, w.num_kv_heads, w.head_dim
    x = normal((s, h + 2 * hk, d), w.std, w.dtype, w.seed, _TAG_STEP + step)
    return (np.ascontiguousarray(x[:, :h]), np.ascontiguousarray(x[:, h:h + hk]),
            np.ascontiguousarray(x[:, h + hk:]))
