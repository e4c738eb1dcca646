"""Pins of the append, block-copy, allocator and serving-loop oracles."""

import numpy as np
import pytest
import scipy.special

from oracle.allocator import BlockAllocator, OutOfBlocks
from oracle.cache import cache_append, cache_append_inplace, copy_blocks
from oracle.serving import ServingOracle, initial_state, tables_array
from tests._golden import allocator_trace, append_layout


def test_append_matches_hand_derived_layout():
    shape, slots, k, v, k_want, v_want = append_layout()
    kc = np.zeros(shape, dtype=np.float32)
    vc = np.zeros(shape, dtype=np.float32)
    kc2, vc2 = cache_append(kc, vc, k, v, slots)
    assert np.array_equal(kc2, k_want)
    assert np.array_equal(vc2, v_want)
    assert not kc.any()  # the input is not modified


def test_append_inplace_matches_loop_form():
    rng = np.random.default_rng(20)
    kc = rng.integers(0, 1 << 16, size=(7, 3, 8, 16)).astype(np.uint16)
    vc = rng.integers(0, 1 << 16, size=(7, 3, 8, 16)).astype(np.uint16)
    k = rng.integers(0, 1 << 16, size=(9, 3, 16)).astype(np.uint16)
    v = rng.integers(0, 1 << 16, size=(9, 3, 16)).astype(np.uint16)
    slots = rng.permutation(56)[:9].astype(np.int64)
    slots[[2, 5]] = -1
    a, b = cache_append(kc, vc, k, v, slots)
    kc2, vc2 = kc.copy(), vc.copy()
    cache_append_inplace(kc2, vc2, k, v, slots)
    assert np.array_equal(a, kc2) and np.array_equal(b, vc2)


def test_copy_blocks_copies_whole_blocks_in_order():
    rng = np.random.default_rng(21)
    kc = rng.standard_normal((5, 2, 4, 3))
    vc = rng.standard_normal((5, 2, 4, 3))
    k0, v0 = kc.copy(), vc.copy()
    copy_blocks(kc, vc, [(1, 3), (3, 4)])
    assert np.array_equal(kc[3], k0[1]) and np.array_equal(vc[3], v0[1])
    assert np.array_equal(kc[4], k0[1]) and np.array_equal(vc[4], v0[1])  # in order
    for b in (0, 1, 2):
        assert np.array_equal(kc[b], k0[b]) and np.array_equal(vc[b], v0[b])


def _check_expect(alloc, kv):
    for key, val in kv.items():
        if key == "free":
            assert alloc.num_free() == val, key
        elif key.startswith("table."):
            assert alloc.block_table(int(key[6:])) == val, key
        elif key.startswith("len."):
            assert alloc.num_tokens(int(key[4:])) == val, key
        elif key.startswith("ref."):
            assert alloc.refcount[int(key[4:])] == val, key
        else:
            raise KeyError(key)


def test_allocator_matches_hand_derived_trace():
    (n, b, order), steps = allocator_trace()
    alloc = BlockAllocator(n, b, order)
    for st in steps:
        if st[0] == "expect":
            _check_expect(alloc, st[1])
            continue
        _, op, args, res = st
        if res == "oom":
            before = (alloc.num_free(), list(alloc.refcount), dict(alloc.lengths))
            with pytest.raises(OutOfBlocks):
                getattr(alloc, {"append": "append_slot"}.get(op, op))(*args)
            assert before == (alloc.num_free(), list(alloc.refcount), dict(alloc.lengths))
        elif op == "append":
            assert alloc.append_slot(*args) == res
        else:
            getattr(alloc, op)(*args)


def test_allocator_invariants_under_random_operations():
    """Refcount of each block = number of tables holding it; free and held
    blocks partition the pool; live tokens occupy distinct slots."""
    rng = np.random.default_rng(22)
    b = 4
    alloc = BlockAllocator(40, b, rng.permutation(40))
    live = []
    nxt = 0
    for _ in range(3000):
        r = rng.random()
        try:
            if r < 0.15 or not live:
                alloc.add(nxt, int(rng.integers(0, 9)))
                live.append(nxt)
                nxt += 1
            elif r < 0.25:
                alloc.fork(live[rng.integers(len(live))], nxt)
                live.append(nxt)
                nxt += 1
            elif r < 0.35:
                s = live.pop(rng.integers(len(live)))
                alloc.free(s)
            else:
                alloc.append_slot(live[rng.integers(len(live))])
        except OutOfBlocks:
            pass
        counts = np.zeros(40, dtype=int)
        for s in live:
            t = alloc.block_table(s)
            assert len(t) == -(-alloc.num_tokens(s) // b)
            for blk in t:
                counts[blk] += 1
        assert list(counts) == alloc.refcount
        assert alloc.num_free() + int(np.count_nonzero(counts)) == 40
    # distinct slots for the last token of every sequence that owns its last block
    owners = {}
    for s in live:
        t = alloc.block_table(s)
        if t and alloc.refcount[t[-1]] == 1:
            slot = t[-1] * b + (alloc.num_tokens(s) - 1) % b
            assert slot not in owners
            owners[slot] = s


def test_initial_state_shares_the_prefix_blocks():
    ctx = np.array([40, 33, 50, 12, 7], dtype=np.int32)
    alloc, pairs = initial_state(5, 8, ctx, 40, np.arange(40), prefix_len=32, prefix_share=3)
    assert pairs == []  # 32 = 4 full blocks of 8: divergence on a block boundary
    t = [alloc.block_table(s) for s in range(5)]
    assert t[0][:4] == t[1][:4] == t[2][:4]
    for blk in t[0][:4]:
        assert alloc.refcount[blk] == 3  # the prefix sequence itself was freed
    assert [alloc.num_tokens(s) for s in range(5)] == list(ctx)
    # a prefix that ends inside a block forces one copy per sharing sequence
    alloc2, pairs2 = initial_state(5, 8, ctx, 40, np.arange(40), prefix_len=30, prefix_share=3)
    assert len(pairs2) == 3
    assert len({p[0] for p in pairs2}) == 1  # all copied the same partly filled block
    t2 = [alloc2.block_table(s) for s in range(5)]
    assert t2[0][:3] == t2[1][:3] == t2[2][:3] and len({t2[s][3] for s in range(3)}) == 3


def test_serving_loop_equals_attention_over_token_history():
    """A few serving steps with copy-on-write: every step's oracle output
    equals dense attention (scipy softmax) over each sequence's full token
    history kept contiguously by the test."""
    rng = np.random.default_rng(23)
    b, hkv, d, h, s = 4, 2, 8, 4, 3
    ctx = np.array([6, 9, 11], dtype=np.int32)
    nblk = 24
    alloc, pairs = initial_state(s, b, ctx, nblk, rng.permutation(nblk), prefix_len=6, prefix_share=2)
    kc = rng.standard_normal((nblk, hkv, b, d))
    vc = rng.standard_normal((nblk, hkv, b, d))
    copy_blocks(kc, vc, pairs)
    hist_k, hist_v = [], []
    for i in range(s):
        t = alloc.block_table(i)
        n = alloc.num_tokens(i)
        hist_k.append(kc[t].transpose(1, 0, 2, 3).reshape(hkv, -1, d)[:, :n])
        hist_v.append(vc[t].transpose(1, 0, 2, 3).reshape(hkv, -1, d)[:, :n])
    # the two sharing sequences really have the same first 6 rows
    assert np.array_equal(hist_k[0][:, :6], hist_k[1][:, :6])
    srv = ServingOracle(alloc, kc, vc, s, "f64", 0.4)
    ncow = 0
    for step in range(6):
        q = rng.standard_normal((s, h, d))
        kn = rng.standard_normal((s, hkv, d))
        vn = rng.standard_normal((s, hkv, d))
        _, pairs, out = srv.step(q, kn, vn, width=8)
        ncow += len(pairs)
        for i in range(s):
            hist_k[i] = np.concatenate([hist_k[i], kn[i][:, None]], axis=1)
            hist_v[i] = np.concatenate([hist_v[i], vn[i][:, None]], axis=1)
            for hh in range(h):
                p = scipy.special.softmax(0.4 * hist_k[i][hh // 2] @ q[i, hh])
                np.testing.assert_allclose(out[i, hh], hist_v[i][hh // 2].T @ p, rtol=0, atol=1e-12)
    assert ncow == 0  # prefix 6 ended mid-block: the copies happened in initial_state
    assert list(srv.context_lens()) == [12, 15, 17]
