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
