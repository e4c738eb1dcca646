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
