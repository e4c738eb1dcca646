"""Decode attention over a paged KV cache, by the plain definition, in fp64.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Definition followed.  For sequence s with context length n = ctx[s] and query
head h, take the KV head kv = h // g (g = H / Hkv query heads per KV head).
The sequence's keys K_s (n x D) are the rows of its cache blocks laid end to
end in block-table order: token t lives in physical block
``block_tables[s][t // B]``, row ``t % B`` ("Day 6/90 of Inference
Engineering", PagedAttention notes, paragraph 6: the block table makes the
scattered blocks read as one contiguous KV cache).  V_s likewise.  Then

    z   = scale · K_s q_{s,h}                 (n scores)
    p   = exp(z - max z) / sum exp(z - max z)
    out = pᵀ V_s                              (D values)

which is the three steps of "PagedAttention Kernel：大模型推理优化的显存管理革新"
section 3.1 (Q·Kᵀ by blocks, softmax, P·V by blocks) written without
blocking.  The method's online softmax and split-K log-sum-exp merge reach
this same value up to rounding.

Cache layout (the pages give none; reading taken): ``[num_blocks, Hkv, B, D]``
for keys and for values.  Stored values are converted to fp64 exactly
(bf16 -> fp32 -> fp64 and fp32 -> fp64 are exact).
"""

from __future__ import annotations

import numpy as np


def to_f64(x: np.ndarray, dtype: str) -> np.ndarray:
    """Exact fp64 value of stored elements.  ``bf16`` arrays hold bit patterns
    (uint16): a bf16 is the top half of an fp32 with the same bits."""
    if dtype == "bf16":
        x = np.asarray(x)
        assert x.dtype == np.uint16
        return (x.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    if dtype == "f32":
        return np.asarray(x, dtype=np.float32).astype(np.float64)
    if dtype == "f64":
        return np.asarray(x, dtype=np.float64)
    raise ValueError(dtype)


def gather_sequence(cache: np.ndarray, table_row: np.ndarray, ctx: int,
                    kv_head: int) -> np.ndarray:
    """Rows 0..ctx-1 of one sequence's keys (or values) for one KV head,
    gathered through its block-table row: ``[ctx, D]`` in storage type."""
    block_size = cache.shape[2]
    nblk = -(-ctx // block_size)
    blocks = np.asarray(table_row[:nblk], dtype=np.int64)
    slabs = cache[blocks, kv_head]  # [nblk, B, D]
    return slabs.reshape(nblk * block_size, cache.shape[3])[:ctx]


def decode_one(q_heads: np.ndarray, k_rows: np.ndarray, v_rows: np.ndarray,
               scale: float) -> np.ndarray:
    """softmax(scale · q Kᵀ) V for a group of query heads sharing one KV head.

    q_heads ``[g, D]``, k_rows and v_rows ``[n, D]``, all fp64; returns
    ``[g, D]`` fp64."""
    z = scale * (q_heads @ k_rows.T)  # [g, n]
    z = z - z.max(axis=1, keepdims=True)
    p = np.exp(z)
    p = p / p.sum(axis=1, keepdims=True)
    return p @ v_rows


def paged_decode(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                 block_tables: np.ndarray, context_lens: np.ndarray,
                 scale: float, dtype: str, seqs=None, cache_dtype: str | None = None,
                 k_scale: float = 1.0, v_scale: float = 1.0) -> np.ndarray:
    """Decode output ``[len(seqs), H, D]`` (fp64) for the listed sequences
    (all by default).

    q ``[S, H, D]``; k_cache, v_cache ``[N, Hkv, B, D]``; block_tables
    ``[S, max_blocks]`` (entries past a sequence's last block are ignored);
    context_lens ``[S]`` (each >= 1).  ``dtype`` is the storage type of q and
    of the caches ("bf16" bit patterns or "f32"); ``cache_dtype="fp8"``
    takes the caches as E4M3 codes read as decode(code) · k_scale (or
    v_scale), see ``oracle.fp8``.
    """
    if cache_dtype == "fp8":
        from .fp8 import decode as fp8_decode

        def kv_f64(rows, which):
            return fp8_decode(rows) * (k_scale if which == "k" else v_scale)
    else:
        def kv_f64(rows, which):
            return to_f64(rows, dtype)
    s_all, h, d = q.shape
    hkv = k_cache.shape[1]
    assert h % hkv == 0 and k_cache.shape[3] == d
    g = h // hkv
    seqs = range(s_all) if seqs is None else list(seqs)
    out = np.empty((len(seqs), h, d), dtype=np.float64)
    for i, s in enumerate(seqs):
        n = int(context_lens[s])
        assert n >= 1
        qs = to_f64(q[s], dtype)
        for kv in range(hkv):
            k_rows = kv_f64(gather_sequence(k_cache, block_tables[s], n, kv), "k")
            v_rows = kv_f64(gather_sequence(v_cache, block_tables[s], n, kv), "v")
            out[i, kv * g:(kv + 1) * g] = decode_one(qs[kv * g:(kv + 1) * g], k_rows, v_rows, scale)
    return out
