"""The algorithmic work bench.py divides by, checked against brute-force
counts on the CPU: KV bytes of a decode step (every context token's key and
value row per KV head; a prefix group's shared partitions once per group),
the E4M3 byte count, prefill FLOPs (each new token's keys up to its own
position), and DRAM counters reported only for the captured kernel
version."""

import os
import sys
from types import SimpleNamespace

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _w(hkv=8, d=128, eb=2):
    return SimpleNamespace(num_kv_heads=hkv, head_dim=d, elem_bytes=eb)


def _brute_rows(ctx, groups, P):
    """(sequence or group, position) pairs read once each: a group's members
    share the positions below the whole-partition part of the prefix."""
    seen = set()
    owner = {s: ("seq", s) for s in range(len(ctx))}
    shared_len = {}
    for gi, (first, count, prefix) in enumerate(groups or ()):
        for s in range(first, first + count):
            owner[s] = ("grp", gi)
            shared_len[s] = prefix // P * P
    for s, c in enumerate(ctx):
        for t in range(int(c)):
            if s in shared_len and t < shared_len[s]:
                seen.add((owner[s], t))
            else:
                seen.add((("seq", s), t))
    return len(seen)


@pytest.mark.parametrize("seed", range(5))
def test_kv_bytes_counts_every_row_once(seed):
    rng = np.random.default_rng(seed)
    ctx = rng.integers(0, 3000, size=12)
    w = _w()
    assert bench.kv_bytes(ctx, w) == _brute_rows(ctx, None, 512) * 8 * 128 * 2 * 2
    # E4M3 storage: one byte per element
    assert bench.kv_bytes(ctx, w, elem_bytes=1) * 2 == bench.kv_bytes(ctx, w)


@pytest.mark.parametrize("seed", range(5))
def test_kv_bytes_with_prefix_groups(seed):
    rng = np.random.default_rng(100 + seed)
    P = 512
    ctx = rng.integers(0, 4000, size=10)
    prefix = int(rng.integers(0, 3000))
    groups = [(2, 5, prefix)]
    w = _w(hkv=4, d=64)
    want = _brute_rows(ctx, groups, P) * 4 * 64 * 2 * 2
    assert bench.kv_bytes(ctx, w, groups, P) == want


def test_prefill_flops_brute_force():
    sh = dict(num_seqs=3, cached=5, new=7, num_heads=4, num_kv_heads=2, head_dim=64, block_size=8)
    b = bench.prefill_batch(seed=3, **sh)
    keys = sum(sh["cached"] + i + 1 for _ in range(sh["num_seqs"]) for i in range(sh["new"]))
    assert bench.prefill_flops(b) == keys * sh["num_heads"] * sh["head_dim"] * 4
    # the batch is what the count assumes: slots of the new tokens after the cached ones
    B = sh["block_size"]
    for s in range(sh["num_seqs"]):
        for i in range(sh["new"]):
            p = sh["cached"] + i
            assert b["slots"][s * sh["new"] + i] == b["tables"][s, p // B] * B + p % B


def test_ragged_prefill_batch_and_flops():
    sh = dict(num_seqs=3, cached=[0, 9, 30], new=[4, 17, 1], num_heads=4, num_kv_heads=2, head_dim=64, block_size=8)
    b = bench.prefill_batch(seed=4, **sh)
    keys = sum(c + i + 1 for c, n in zip(sh["cached"], sh["new"]) for i in range(n))
    assert bench.prefill_flops(b) == keys * sh["num_heads"] * sh["head_dim"] * 4
    assert list(b["qs"]) == [0, 4, 21, 22] and list(b["ctx"]) == [4, 26, 31]
    assert b["q"].shape == (22, 4, 64) and b["k"].shape == (22, 2, 64)
    B = sh["block_size"]
    used = set()
    for s, (c, n) in enumerate(zip(sh["cached"], sh["new"])):
        nb = -(-(c + n) // B)
        used |= set(b["tables"][s, :nb].tolist())
        for i in range(n):
            p = c + i
            assert b["slots"][b["qs"][s] + i] == b["tables"][s, p // B] * B + p % B
    assert len(used) == sum(-(-(c + n) // B) for c, n in zip(sh["cached"], sh["new"]))  # no block shared
    # the bench's ragged batch: 8 prompts, lengths in their stated ranges
    r = bench.PREFILL_RAGGED_SHAPE
    assert len(r["cached"]) == len(r["new"]) == r["num_seqs"] == 8
    assert all(0 <= c <= 4096 for c in r["cached"]) and all(64 <= n <= 2048 for n in r["new"])


def test_dram_counters_only_for_the_captured_kernel(monkeypatch):
    v = bench.decode_traffic("mha_bf16")
    assert v is None or v > 0
    if v is not None:
        # another version of the sources: the stored counters are not reported
        monkeypatch.setattr(bench, "DECODE_SOURCES", ("bench.py",))
        assert bench.decode_traffic("mha_bf16") is None


def test_kernel_hash_ignores_comments_only():
    """The hash that gates the committed DRAM counters changes with the code
    and not with its comments (string literals are code)."""
    import bench

    a = 'int f() {  // sum\n  /* two\n lines */ return g("a // b");\n}\n'
    b = 'int f() {\n\n  return g("a // b");  // other words\n}\n'
    c = 'int f() {\n  return g("a // c");\n}\n'
    assert bench.strip_comments(a) == bench.strip_comments(b)
    assert bench.strip_comments(a) != bench.strip_comments(c)
    src = {"x": a}
    assert bench.decode_kernel_hash(("x",), src.get) == bench.decode_kernel_hash(("x",), {"x": b}.get)
