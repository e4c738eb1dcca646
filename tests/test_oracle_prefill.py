"""Pins of the prefill oracle: decode as its one-token case, dense causal
attention on contiguous rows, the first prompt token returning its own
value, invariance to block placement, and planted causal mistakes."""

import numpy as np
import pytest
import scipy.special

import oracle.prefill as pf
from oracle.attention import decode_one, gather_sequence, paged_decode, to_f64
from oracle.cache import cache_append


def _batch(rng, prev, new, hkv=2, g=2, d=8, b=4, nblk=None, shuffle=True):
    """Random fp64 batch: per sequence `prev` cached tokens and `new` prompt
    tokens, tables over a (shuffled) pool, slots of the new tokens."""
    s = len(prev)
    ctx = np.array([p + n for p, n in zip(prev, new)], dtype=np.int32)
    need = sum(-(-int(c) // b) for c in ctx)
    nblk = nblk or need + 3
    perm = rng.permutation(nblk) if shuffle else np.arange(nblk)
    width = max(-(-int(c) // b) for c in ctx)
    tables = np.full((s, width), -1, dtype=np.int32)
    it = iter(perm.tolist())
    for i in range(s):
        nb = -(-int(ctx[i]) // b)
        tables[i, :nb] = [next(it) for _ in range(nb)]
    kc = rng.standard_normal((nblk, hkv, b, d))
    vc = rng.standard_normal((nblk, hkv, b, d))
    qs = np.concatenate([[0], np.cumsum(new)]).astype(np.int32)
    t = int(qs[-1])
    q = rng.standard_normal((t, hkv * g, d))
    k = rng.standard_normal((t, hkv, d))
    v = rng.standard_normal((t, hkv, d))
    slots = np.empty(t, dtype=np.int64)
    for i in range(s):
        for j in range(new[i]):
            pos = prev[i] + j
            slots[qs[i] + j] = tables[i, pos // b] * b + pos % b
    return q, k, v, slots, qs, ctx, tables, kc, vc


def _wrong_no_self(q, k, v, slots, qs, ctx, tables, kc, vc, scale, dtype):
    """Each token attends only the tokens before it (off by one)."""
    kc2, vc2 = cache_append(kc, vc, k, v, slots)
    out = np.full(q.shape, np.nan)
    g = q.shape[1] // kc.shape[1]
    for s in range(len(ctx)):
        n_new = int(qs[s + 1] - qs[s])
        for kv in range(kc.shape[1]):
            kr = gather_sequence(kc2, tables[s], int(ctx[s]), kv)
            vr = gather_sequence(vc2, tables[s], int(ctx[s]), kv)
            for i in range(n_new):
                p = int(ctx[s]) - n_new + i
                m = max(p, 1)
                out[qs[s] + i, kv * g:(kv + 1) * g] = decode_one(q[qs[s] + i, kv * g:(kv + 1) * g], kr[:m], vr[:m],
                                                                 scale)
    return kc2, vc2, out


def _wrong_positions(q, k, v, slots, qs, ctx, tables, kc, vc, scale, dtype):
    """Positions counted from the start of the prompt, ignoring the cached
    tokens before it."""
    kc2, vc2 = cache_append(kc, vc, k, v, slots)
    out = np.full(q.shape, np.nan)
    g = q.shape[1] // kc.shape[1]
    for s in range(len(ctx)):
        n_new = int(qs[s + 1] - qs[s])
        for kv in range(kc.shape[1]):
            kr = gather_sequence(kc2, tables[s], int(ctx[s]), kv)
            vr = gather_sequence(vc2, tables[s], int(ctx[s]), kv)
            for i in range(n_new):
                out[qs[s] + i, kv * g:(kv + 1) * g] = decode_one(q[qs[s] + i, kv * g:(kv + 1) * g], kr[:i + 1],
                                                                 vr[:i + 1], scale)
    return kc2, vc2, out


def pin_one_token_is_decode(fn):
    rng = np.random.default_rng(1)
    prev, new = [5, 0, 12], [1, 1, 1]
    q, k, v, slots, qs, ctx, tables, kc, vc = _batch(rng, prev, new)
    kc2, vc2, out = fn(q, k, v, slots, qs, ctx, tables, kc, vc, 0.3, "f64")
    want = paged_decode(q, kc2, vc2, tables, ctx, 0.3, "f64")
    assert np.array_equal(out, want)


def pin_dense_causal_attention(fn):
    """Contiguous rows: scores masked above the diagonal, scipy softmax."""
    rng = np.random.default_rng(2)
    prev, new = [3, 0], [6, 9]
    q, k, v, slots, qs, ctx, tables, kc, vc = _batch(rng, prev, new, hkv=2, g=2)
    kc2, vc2, out = fn(q, k, v, slots, qs, ctx, tables, kc, vc, 0.45, "f64")
    for s in range(2):
        n, c = new[s], int(ctx[s])
        for kv in range(2):
            K = to_f64(gather_sequence(kc2, tables[s], c, kv), "f64")
            V = to_f64(gather_sequence(vc2, tables[s], c, kv), "f64")
            for hh in (2 * kv, 2 * kv + 1):
                Q = q[qs[s]:qs[s] + n, hh]  # [n, d]
                z = 0.45 * Q @ K.T  # [n, c]
                pos = prev[s] + np.arange(n)
                z[np.arange(c)[None, :] > pos[:, None]] = -np.inf
                P = scipy.special.softmax(z, axis=1)
                np.testing.assert_allclose(out[qs[s]:qs[s] + n, hh], P @ V, rtol=0, atol=1e-12)


def pin_first_token_of_fresh_prompt(fn):
    rng = np.random.default_rng(3)
    q, k, v, slots, qs, ctx, tables, kc, vc = _batch(rng, [0, 0], [4, 1])
    _, _, out = fn(q, k, v, slots, qs, ctx, tables, kc, vc, 0.3, "f64")
    for s in range(2):
        for hh in range(4):
            assert np.array_equal(out[qs[s], hh], v[qs[s], hh // 2])


def pin_block_placement_invariance(fn):
    rng = np.random.default_rng(4)
    prev, new = [7, 2, 0], [5, 11, 3]
    q, k, v, slots, qs, ctx, tables, kc, vc = _batch(rng, prev, new, shuffle=False)
    _, _, out = fn(q, k, v, slots, qs, ctx, tables, kc, vc, 0.3, "f64")
    perm = rng.permutation(kc.shape[0])  # block b moves to perm[b]
    kc_p = np.empty_like(kc)
    vc_p = np.empty_like(vc)
    kc_p[perm] = kc
    vc_p[perm] = vc
    tables_p = np.where(tables >= 0, perm[np.maximum(tables, 0)], -1).astype(np.int32)
    b = kc.shape[2]
    slots_p = perm[slots // b] * b + slots % b
    _, _, out_p = fn(q, k, v, slots_p, qs, ctx, tables_p, kc_p, vc_p, 0.3, "f64")
    assert np.array_equal(out, out_p)


PINS = [pin_one_token_is_decode, pin_dense_causal_attention, pin_first_token_of_fresh_prompt,
        pin_block_placement_invariance]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_prefill_oracle_pins(pin):
    pin(pf.prefill)


def test_prefill_appends_like_the_cache_oracle():
    rng = np.random.default_rng(5)
    q, k, v, slots, qs, ctx, tables, kc, vc = _batch(rng, [2, 9], [7, 4])
    kc2, vc2, _ = pf.prefill(q, k, v, slots, qs, ctx, tables, kc, vc, 0.3, "f64")
    want_k, want_v = cache_append(kc, vc, k, v, slots)
    assert np.array_equal(kc2, want_k) and np.array_equal(vc2, want_v)


@pytest.mark.parametrize("wrong", [_wrong_no_self, _wrong_positions], ids=lambda f: f.__name__)
def test_planted_causal_mistakes_fail_a_pin(wrong):
    failed = 0
    for pin in PINS:
        try:
            pin(wrong)
        except AssertionError:
            failed += 1
    assert failed >= 1
