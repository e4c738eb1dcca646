"""The host-built decode work list (pa_decode_plan_host): every (sequence,
partition) pair exactly once, full partitions first, partial ones from the
longest remainder down, empty contexts last, counter 0 (no GPU needed)."""

import numpy as np
import pytest

from tests._lib_fixture import ensure_built


@pytest.fixture(scope="module")
def ops():
    ensure_built()
    from paged_kv_cache_216_gb300 import ops

    return ops


def _parse(buf):
    hdr = buf[:256].view(np.int32)
    n = int(hdr[1])
    ent = buf[256:256 + 8 * n].view(np.int32).reshape(n, 2)
    return int(hdr[0]), ent[:, 0] & 0xFFFF, ent[:, 0] >> 16, ent[:, 1]


@pytest.mark.parametrize("P", [32, 64, 512])
def test_plan_lists_every_pair_longest_first(ops, P):
    rng = np.random.default_rng(P)
    ctx = rng.integers(0, 3000, size=97).astype(np.int32)
    ctx[[3, 10]] = 0
    ctx[5] = 2 * P  # a context of whole partitions only
    mx = int(ctx.max())
    nbytes = ops.decode_plan_bytes(len(ctx), mx, P)
    assert nbytes == 256 + 8 * len(ctx) * (-(-mx // P))
    buf = np.full(nbytes, 0xAB, dtype=np.uint8)
    ops.decode_plan_host(ctx, mx, P, buf)
    counter, s, part, c = _parse(buf)
    assert counter == 0
    want = {(i, p) for i in range(len(ctx)) for p in range(-(-int(ctx[i]) // P))}
    want |= {(i, 0) for i in range(len(ctx)) if ctx[i] == 0}
    got = list(zip(s.tolist(), part.tolist()))
    assert len(got) == len(want) and set(got) == want
    assert np.array_equal(c, ctx[s])
    size = np.where(c == 0, -1, np.minimum(c - part * P, P))  # tokens of each entry; empties last
    full = size == P
    nf = int(full.sum())
    assert full[:nf].all() and not full[nf:].any()
    rest = size[nf:]
    assert np.all(rest[:-1] >= rest[1:])  # non-increasing: longest partial first, empties at the end


def test_plan_rejects_bad_arguments(ops):
    from paged_kv_cache_216_gb300._lib import PAError

    buf = np.zeros(4096, dtype=np.uint8)
    with pytest.raises(PAError):
        ops.decode_plan_host(np.array([5, 900], dtype=np.int32), 800, 64, buf)  # longer than the bound
    with pytest.raises(PAError):
        ops.decode_plan_host(np.array([5, 9], dtype=np.int32), 800, 48, buf)  # not a multiple of 32


def _skip_of(groups, n, P, max_ctx):
    """Shared partitions of each sequence: whole partitions of its group's
    prefix, none when no context can span two partitions."""
    skip = np.zeros(n, dtype=np.int64)
    if -(-max_ctx // P) > 1:
        for first, count, prefix in groups:
            skip[first:first + count] = prefix // P
    return skip


def _parse_shared(buf):
    """(ordinary entries (s, part, ctx), shared entries (table seq, part, s0, nm))."""
    hdr = buf[:256].view(np.int32)
    n = int(hdr[1])
    ent = buf[256:256 + 8 * n].view(np.int32).reshape(n, 2)
    sh = ent[:, 1] < 0
    nsh = int(sh.sum())
    assert sh[:nsh].all() and not sh[nsh:].any()  # shared items head the list
    x, y = ent[:nsh, 0], ent[:nsh, 1]
    shared = [(int(a & 0xFFFF), int(a >> 16), int((b >> 8) & 0xFFFF), int(b & 0xFF)) for a, b in zip(x, y)]
    o = ent[nsh:]
    return int(hdr[0]), o[:, 0] & 0xFFFF, o[:, 0] >> 16, o[:, 1], shared


@pytest.mark.parametrize("P,g", [(32, 4), (64, 1), (64, 8)])
def test_plan_shares_prefix_partitions(ops, P, g):
    """With prefix groups the list starts with one shared item per (group,
    shared partition, run of 128/g consecutive members: one tensor-core tile
    of query rows), then holds every other (sequence, partition) pair
    exactly once, longest first."""
    rng = np.random.default_rng(100 + P + g)
    ctx = rng.integers(150, 900, size=23).astype(np.int32)
    ctx[1] = 3 * P  # ends exactly at its group's shared part
    ctx[6] = 0  # an empty member
    ctx[9] = P // 2  # a member shorter than its group's shared part
    groups = [(0, 4, 3 * P + 5), (5, 6, 2 * P), (12, 1, P - 1), (14, 3, 200)]
    mx = int(ctx.max())
    buf = np.full(ops.decode_plan_bytes(len(ctx), mx, P), 0xCD, dtype=np.uint8)
    ops.decode_plan_host(ctx, mx, P, buf, prefix_groups=groups, num_heads=8 * g, num_kv_heads=8)
    counter, s, part, c, shared = _parse_shared(buf)
    assert counter == 0
    skip = _skip_of(groups, len(ctx), P, mx)
    nm = 128 // g
    want_shared = set()
    for first, count, prefix in groups:
        for p in range(prefix // P):
            for s0 in range(first, first + count, nm):
                want_shared.add((first, p, s0, min(nm, first + count - s0)))
    assert len(shared) == len(want_shared) and set(shared) == want_shared
    want = {(i, p) for i in range(len(ctx)) for p in range(int(skip[i]), -(-int(ctx[i]) // P))}
    want |= {(i, 0) for i in range(len(ctx)) if ctx[i] == 0}
    got = list(zip(s.tolist(), part.tolist()))
    assert len(got) == len(want) and set(got) == want
    assert not any(i == 1 for i, _ in got)  # all of its partitions are shared
    assert np.array_equal(c, ctx[s])
    size = np.where(c == 0, -1, np.minimum(c - part * P, P))
    nf = int((size == P).sum())
    assert (size[:nf] == P).all() and np.all(size[nf:-1] >= size[nf + 1:])
    # no groups: the plain list
    buf2 = np.full_like(buf, 0xCD)
    ops.decode_plan_host(ctx, mx, P, buf2, prefix_groups=[])
    plain = np.full_like(buf, 0xCD)
    ops.decode_plan_host(ctx, mx, P, plain)
    assert np.array_equal(buf2, plain)


def test_plan_with_one_partition_shares_nothing(ops):
    """When no context spans two partitions there are no partial slots for
    shared partitions: groups change nothing."""
    ctx = np.array([40, 64, 10], dtype=np.int32)
    a = np.zeros(ops.decode_plan_bytes(3, 64, 64), dtype=np.uint8)
    b = np.zeros_like(a)
    ops.decode_plan_host(ctx, 64, 64, a, prefix_groups=[(0, 3, 64)], num_heads=8, num_kv_heads=2)
    ops.decode_plan_host(ctx, 64, 64, b)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("groups", [
    [(0, 3, 100), (2, 2, 100)],  # overlapping
    [(3, 2, 100), (0, 2, 100)],  # not ascending
    [(0, 0, 100)],  # empty
    [(8, 3, 100)],  # past the batch
    [(0, 2, 5000)],  # prefix longer than the length bound
    [(0, 2, -1)],
])
def test_plan_rejects_bad_prefix_groups(ops, groups):
    from paged_kv_cache_216_gb300._lib import PAError

    buf = np.zeros(ops.decode_plan_bytes(10, 1000, 64), dtype=np.uint8)
    with pytest.raises(PAError):
        ops.decode_plan_host(np.full(10, 500, dtype=np.int32), 1000, 64, buf, prefix_groups=groups)


def test_plan_rejects_too_many_prefix_groups(ops):
    from paged_kv_cache_216_gb300._lib import PA_MAX_PREFIX_GROUPS, PAError

    n = PA_MAX_PREFIX_GROUPS + 1
    groups = [(i, 1, 64) for i in range(n)]
    buf = np.zeros(ops.decode_plan_bytes(n, 1000, 64), dtype=np.uint8)
    with pytest.raises(PAError, match="UNSUPPORTED|more than"):
        ops.decode_plan_host(np.full(n, 500, dtype=np.int32), 1000, 64, buf, prefix_groups=groups)
