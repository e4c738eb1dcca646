"""Prefill into a paged KV cache: append a prompt's keys and values, then
causal attention of every prompt token, by the plain definition in fp64.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The step before decode on the method's timeline ("Day 6/90 of Inference
Engineering", PagedAttention notes, paragraph 2: the KV cache grows one
block at a time as tokens are produced; a prompt's tokens are written the
same way, many at once).  For sequence s, let n_s new tokens follow c_s
tokens already cached, so its context after the append is
context_lens[s] = c_s + n_s.  New token i (0 <= i < n_s) sits at position
p = c_s + i and attends every token at positions 0..p of the sequence --
the tokens before it and itself, none after (causal attention):

    out[s, i, h] = softmax(scale · K_s[0..p] q[s, i, h]) V_s[0..p]

with K_s, V_s the sequence's rows gathered through its block table after
the append, and query head h reading KV head h // g.  With n_s = 1 this is
the decode step.
"""

from __future__ import annotations

import numpy as np

from .attention import decode_one, gather_sequence, to_f64
from .cache import cache_append


def prefill(q: np.ndarray, k: np.ndarray, v: np.ndarray, slot_mapping: np.ndarray, query_start: np.ndarray,
            context_lens: np.ndarray, block_tables: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
            scale: float, dtype: str):
    """Returns ``(k_cache', v_cache', out)``: copies of the caches with the
    new tokens written at their slots, and ``out [T, H, D]`` fp64.

    q ``[T, H, D]``, k and v ``[T, Hkv, D]`` (storage type ``dtype``), the
    new tokens of all sequences one after another; sequence s owns rows
    ``query_start[s] .. query_start[s + 1] - 1``.  ``context_lens[s]`` counts
    its tokens after the append."""
    kc, vc = cache_append(k_cache, v_cache, k, v, slot_mapping)
    t_all, h, d = q.shape
    hkv = kc.shape[1]
    g = h // hkv
    out = np.full((t_all, h, d), np.nan)
    for s in range(len(context_lens)):
        q0, q1 = int(query_start[s]), int(query_start[s + 1])
        n_new = q1 - q0
        ctx = int(context_lens[s])
        assert 0 <= n_new <= ctx
        for kv in range(hkv):
            k_rows = to_f64(gather_sequence(kc, block_tables[s], ctx, kv), dtype)
            v_rows = to_f64(gather_sequence(vc, block_tables[s], ctx, kv), dtype)
            for i in range(n_new):
                p = ctx - n_new + i  # position of this new token
                qh = to_f64(q[q0 + i, kv * g:(kv + 1) * g], dtype)
                out[q0 + i, kv * g:(kv + 1) * g] = decode_one(qh, k_rows[:p + 1], v_rows[:p + 1], scale)
    return kc, vc, out
