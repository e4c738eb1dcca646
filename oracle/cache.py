"""KV append and block copy on a paged cache, element by element.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Append ("Day 6/90 of Inference Engineering", PagedAttention notes,
paragraph 2: each new token's K/V goes into the current cache block): token i
with slot ``slot_mapping[i] = b·B + r`` writes its key for KV head h into
``k_cache[b, h, r, :]`` and its value into ``v_cache[b, h, r, :]``.  A
negative slot means "no write".  Copies are of stored bits, so the result is
exact in any storage type.

Block copy (same page, paragraph 5: a sequence that diverges from a shared
prefix writes to a new block): for each pair (src, dst) the whole block
``src`` of both caches, every KV head, is copied to block ``dst``.  Pairs are
applied in order.

FP8 append (reading of the pages' "fewer bytes moved", see ``oracle.fp8``):
the same scatter, of the codes quantize(x, k_scale) and quantize(x, v_scale)
of the new token's bf16 key and value.
"""

from __future__ import annotations

import numpy as np


def cache_append(k_cache: np.ndarray, v_cache: np.ndarray, k: np.ndarray,
                 v: np.ndarray, slot_mapping: np.ndarray):
    """Return copies of the caches ``[N, Hkv, B, D]`` with tokens ``k, v``
    ``[T, Hkv, D]`` written at ``slot_mapping`` ``[T]``."""
    kc = k_cache.copy()
    vc = v_cache.copy()
    block_size = kc.shape[2]
    for i in range(len(slot_mapping)):
        slot = int(slot_mapping[i])
        if slot < 0:
            continue
        b, r = divmod(slot, block_size)
        for h in range(kc.shape[1]):
            kc[b, h, r, :] = k[i, h, :]
            vc[b, h, r, :] = v[i, h, :]
    return kc, vc


def cache_append_inplace(k_cache: np.ndarray, v_cache: np.ndarray, k: np.ndarray,
                         v: np.ndarray, slot_mapping: np.ndarray) -> None:
    """In-place form of :func:`cache_append` for large pools (same rule,
    written with numpy indexing; slots must be distinct)."""
    slots = np.asarray(slot_mapping, dtype=np.int64)
    keep = slots >= 0
    block_size = k_cache.shape[2]
    b = slots[keep] // block_size
    r = slots[keep] % block_size
    k_cache[b, :, r, :] = k[keep]
    v_cache[b, :, r, :] = v[keep]


def copy_blocks(k_cache: np.ndarray, v_cache: np.ndarray, pairs) -> None:
    """In place: block ``dst`` := block ``src`` in both caches, for each
    (src, dst) pair in order."""
    for src, dst in pairs:
        k_cache[int(dst)] = k_cache[int(src)]
        v_cache[int(dst)] = v_cache[int(src)]


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """fp32 value of bf16 bit patterns (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def cache_append_fp8(k_cache: np.ndarray, v_cache: np.ndarray, k: np.ndarray, v: np.ndarray,
                     slot_mapping: np.ndarray, k_scale: float, v_scale: float):
    """Return copies of the E4M3 caches (uint8 ``[N, Hkv, B, D]``) with the
    bf16 tokens ``k, v`` ``[T, Hkv, D]`` (bit patterns) quantized into their
    slots."""
    from .fp8 import quantize

    kq = quantize(bf16_to_f32(k), k_scale)
    vq = quantize(bf16_to_f32(v), v_scale)
    return cache_append(k_cache, v_cache, kq, vq, slot_mapping)


def quantize_pool_fp8(pool_bits: np.ndarray, scale: float) -> np.ndarray:
    """E4M3 codes of a whole bf16 pool (bit patterns), in place of appending
    every slot one by one; chunked to bound memory."""
    from .fp8 import quantize

    flat = np.asarray(pool_bits).reshape(-1)
    out = np.empty(flat.shape, dtype=np.uint8)
    step = 1 << 24
    for i in range(0, flat.size, step):
        out[i:i + step] = quantize(bf16_to_f32(flat[i:i + step]), scale)
    return out.reshape(np.shape(pool_bits))
