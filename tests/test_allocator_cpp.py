"""The C++ block allocator (through the C ABI) against the hand-derived trace
and, bit for bit, against the oracle's allocator under random operations."""

import numpy as np
import pytest

from oracle.allocator import BlockAllocator as OracleAllocator
from oracle.allocator import OutOfBlocks as OracleOOM
from oracle.serving import initial_state
from tests._golden import allocator_trace
from tests._lib_fixture import ensure_built
from workloads import WORKLOADS, context_lens, free_order, pool_blocks


@pytest.fixture(scope="module")
def pkg():
    ensure_built()
    import paged_kv_cache_216_gb300 as pkg

    return pkg


def test_cpp_allocator_matches_hand_derived_trace(pkg):
    (n, b, order), steps = allocator_trace()
    a = pkg.BlockAllocator(n, b, order)
    for st in steps:
        if st[0] == "expect":
            for key, val in st[1].items():
                if key == "free":
                    assert a.num_free() == val, key
                elif key.startswith("table."):
                    assert a.block_table(int(key[6:])) == val, key
                elif key.startswith("len."):
                    assert a.num_tokens(int(key[4:])) == val, key
                elif key.startswith("ref."):
                    assert a.refcount(int(key[4:])) == val, key
            continue
        _, op, args, res = st
        fn = {"append": a.append_slot, "add": a.add, "fork": a.fork, "free": a.free}[op]
        if res == "oom":
            free_before = a.num_free()
            with pytest.raises(pkg.OutOfBlocks):
                fn(*args)
            assert a.num_free() == free_before
        elif op == "append":
            assert fn(*args) == res
        else:
            fn(*args)


def test_cpp_allocator_equals_oracle_under_random_operations(pkg):
    rng = np.random.default_rng(30)
    nb, b = 64, 8
    order = rng.permutation(nb).astype(np.int32)
    c = pkg.BlockAllocator(nb, b, order)
    o = OracleAllocator(nb, b, order)
    live, nxt = [], 0
    for _ in range(4000):
        r = rng.random()
        if r < 0.12 or not live:
            op, args = "add", (nxt, int(rng.integers(0, 30)))
        elif r < 0.22:
            op, args = "fork", (live[rng.integers(len(live))], nxt)
        elif r < 0.32:
            op, args = "free", (live[rng.integers(len(live))],)
        else:
            op, args = "append_slot", (live[rng.integers(len(live))],)
        try:
            want = getattr(o, op)(*args)
            oom = False
        except OracleOOM:
            oom = True
        if oom:
            with pytest.raises(pkg.OutOfBlocks):
                getattr(c, op)(*args)
        else:
            got = getattr(c, op)(*args)
            assert got == want
            if op in ("add", "fork"):
                live.append(nxt)
                nxt += 1
            elif op == "free":
                live.remove(args[0])
        assert c.num_free() == o.num_free()
    for s in live:
        assert c.block_table(s) == o.block_table(s)
        assert c.num_tokens(s) == o.num_tokens(s)
    for blk in range(nb):
        assert c.refcount(blk) == o.refcount[blk]


def test_batched_append_equals_single_appends_and_updates_tables(pkg):
    rng = np.random.default_rng(31)
    nb, b = 200, 4
    order = rng.permutation(nb).astype(np.int32)
    ctx = rng.integers(1, 20, size=12)
    a1 = pkg.BlockAllocator(nb, b, order)
    a2 = pkg.BlockAllocator(nb, b, order)
    for s, n in enumerate(ctx):
        a1.add(s, int(n))
        a2.add(s, int(n))
    a1.fork(3, 12)
    a2.fork(3, 12)  # a shared, partly filled last block -> copy-on-write
    ids = np.arange(13, dtype=np.int64)
    width = 16
    tables = np.full((13, width), -1, dtype=np.int32)
    lens = np.zeros(13, dtype=np.int32)
    a1.block_tables(ids, tables, lens)
    for step in range(9):
        slots = np.empty(13, dtype=np.int64)
        pairs = np.empty((13, 2), dtype=np.int32)
        nc = a1.append_slots(ids, slots, pairs, tables, lens)
        want_pairs = []
        for i, s in enumerate(ids):
            slot, src, dst = a2.append_slot(int(s))
            assert slots[i] == slot
            if src >= 0:
                want_pairs.append((src, dst))
        assert [tuple(p) for p in pairs[:nc]] == want_pairs
        if step == 0 and ctx[3] % b:
            assert nc >= 1
        full = np.full((13, width), -1, dtype=np.int32)
        lens2 = np.zeros(13, dtype=np.int32)
        a2.block_tables(ids, full, lens2)
        assert np.array_equal(tables, full) and np.array_equal(lens, lens2)


def test_batched_append_is_all_or_nothing_on_oom(pkg):
    a = pkg.BlockAllocator(4, 4, np.arange(4, dtype=np.int32))
    a.add(0, 4)
    a.add(1, 8)
    a.add(2, 3)  # 4 blocks used: 0 and 1 are full, 2 is not
    ids = np.array([2, 0, 1], dtype=np.int64)
    slots = np.zeros(3, dtype=np.int64)
    pairs = np.zeros((3, 2), dtype=np.int32)
    with pytest.raises(pkg.OutOfBlocks):
        a.append_slots(ids, slots, pairs)
    assert a.num_tokens(2) == 3 and a.num_tokens(0) == 4 and a.num_free() == 0


def test_error_codes(pkg):
    a = pkg.BlockAllocator(8, 4)
    with pytest.raises(pkg.PAError) as e:
        a.free(5)
    assert e.value.code == -4  # unknown sequence
    a.add(1, 3)
    with pytest.raises(pkg.PAError) as e:
        a.add(1, 3)
    assert e.value.code == -4
    with pytest.raises(pkg.PAError) as e:
        pkg.BlockAllocator(4, 4, np.array([0, 1, 1, 2], dtype=np.int32))
    assert e.value.code == -1
    with pytest.raises(pkg.PAError) as e:
        a.append_slots(np.array([1, 1], dtype=np.int64), np.zeros(2, np.int64), np.zeros((2, 2), np.int32))
    assert e.value.code == -1  # the same sequence twice in one batch


@pytest.mark.parametrize("name", ["gqa_prefix_bf16", "serving_bf16_b16", "mha_bf16"])
def test_workload_set_up_matches_oracle(pkg, name):
    """The product-side set-up script (C++ allocator) and the oracle's give
    identical tables for every workload, including a mid-block prefix."""
    from paged_kv_cache_216_gb300.prefix import populate

    w = WORKLOADS[name]
    for prefix_len in ([w.prefix_len, w.prefix_len - 5] if w.prefix_share else [0]):
        ctx = context_lens(w)
        nb = pool_blocks(w, ctx) + w.prefix_share
        order = free_order(w, nb)
        o, opairs = initial_state(w.num_seqs, w.block_size, ctx, nb, order, prefix_len, w.prefix_share)
        c = pkg.BlockAllocator(nb, w.block_size, order)
        cpairs = populate(c, ctx, prefix_len, w.prefix_share)
        assert [tuple(p) for p in cpairs] == opairs
        for s in range(w.num_seqs):
            assert c.block_table(s) == o.block_table(s)
        assert c.num_free() == o.num_free()
