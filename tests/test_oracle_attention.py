"""Pins of the decode oracle against what the mathematics fixes.

Each test would fail under a plausible mistake in ``oracle.attention``:
a wrong gather (block order, row/column order, block size), a wrong GQA head
mapping, a missing or wrong scale, swapped K and V, a missing max
subtraction, reading rows past the context, or inexact bf16 conversion.
"""

import math

import numpy as np
import pytest
import scipy.special

from oracle.attention import paged_decode, to_f64
from oracle.allocator import BlockAllocator
from oracle.serving import tables_array
from workloads import WORKLOADS, context_lens, free_order, queries, random_pool


def _identity_pool(kd, block_size):
    """Lay contiguous per-sequence rows ``kd [S, Hkv, M*B, D]`` out as a pool in
    which sequence s owns blocks s*M .. s*M+M-1 (identity block tables)."""
    s, hkv, n, d = kd.shape
    m = n // block_size
    pool = kd.reshape(s, hkv, m, block_size, d).transpose(0, 2, 1, 3, 4)
    return np.ascontiguousarray(pool.reshape(s * m, hkv, block_size, d))


def test_bf16_conversion_is_exact():
    bits = np.array([0x3F80, 0xC000, 0x3E80, 0x7F7F, 0x0001, 0x8000, 0x4049], dtype=np.uint16)
    want = [1.0, -2.0, 0.25, (2 - 2 ** -7) * 2.0 ** 127, 2.0 ** -133, -0.0, 3.140625]
    got = to_f64(bits, "bf16")
    for g, w in zip(got, want):
        assert g == w and math.copysign(1, g) == math.copysign(1, w)


def test_identity_tables_match_dense_attention():
    """(a) With identity block tables paged decode is ordinary attention on
    the contiguous keys/values (scipy softmax on contiguous arrays)."""
    rng = np.random.default_rng(10)
    s, h, hkv, d, b = 3, 6, 2, 16, 4
    m = 5
    ctx = np.array([1, 9, 20], dtype=np.int32)  # 20 = M*B: a full last block
    q = rng.standard_normal((s, h, d))
    kd = rng.standard_normal((s, hkv, m * b, d))
    vd = rng.standard_normal((s, hkv, m * b, d))
    tables = np.arange(s * m, dtype=np.int32).reshape(s, m)
    scale = 0.3
    out = paged_decode(q, _identity_pool(kd, b), _identity_pool(vd, b), tables, ctx, scale, "f64")
    g = h // hkv
    for i in range(s):
        n = ctx[i]
        for hh in range(h):
            kv = hh // g
            p = scipy.special.softmax(scale * (kd[i, kv, :n] @ q[i, hh]))
            want = vd[i, kv, :n].T @ p
            np.testing.assert_allclose(out[i, hh], want, rtol=0, atol=1e-12)


def test_block_permutation_invariance_is_bitwise():
    """(b) Relabelling physical blocks (and the tables with them) changes no
    bit of the result."""
    w = WORKLOADS["tiny_f32"]
    rng = np.random.default_rng(11)
    nblk, hkv, b, d = 16, 4, 16, 64
    kc = rng.standard_normal((nblk, hkv, b, d)).astype(np.float32)
    vc = rng.standard_normal((nblk, hkv, b, d)).astype(np.float32)
    q = rng.standard_normal((4, 4, d)).astype(np.float32)
    ctx = np.array([1, 7, 16, 33], dtype=np.int32)
    tables = rng.permutation(nblk)[:12].reshape(4, 3).astype(np.int32)
    perm = rng.permutation(nblk)
    kc2 = np.empty_like(kc)
    vc2 = np.empty_like(vc)
    kc2[perm] = kc
    vc2[perm] = vc
    tables2 = perm[tables].astype(np.int32)
    a = paged_decode(q, kc, vc, tables, ctx, w.scale, "f32")
    c = paged_decode(q, kc2, vc2, tables2, ctx, w.scale, "f32")
    assert np.array_equal(a, c)


def test_single_token_returns_its_value_exactly():
    """(c) ctx = 1: the softmax of one score is exactly 1, so out = V_0."""
    rng = np.random.default_rng(12)
    kc = rng.standard_normal((4, 2, 8, 32))
    vc = rng.standard_normal((4, 2, 8, 32))
    q = rng.standard_normal((2, 4, 32)) * 50.0
    tables = np.array([[3, 0], [1, 2]], dtype=np.int32)
    out = paged_decode(q, kc, vc, tables, np.array([1, 1]), 0.7, "f64")
    for s in range(2):
        for h in range(4):
            assert np.array_equal(out[s, h], vc[tables[s, 0], h // 2, 0])


def test_constant_values_and_gqa_head_mapping():
    """(d) All value rows of KV head kv equal c_kv: every query head h in
    that head's group returns c_{h // g}; a group mapping h % g fails."""
    rng = np.random.default_rng(13)
    nblk, hkv, b, d, h = 8, 4, 4, 8, 16
    c = rng.standard_normal((hkv, d))
    vc = np.broadcast_to(c[None, :, None, :], (nblk, hkv, b, d)).copy()
    kc = rng.standard_normal((nblk, hkv, b, d))
    q = rng.standard_normal((2, h, d))
    tables = np.array([[5, 1, 7, 0], [2, 6, 3, 4]], dtype=np.int32)
    out = paged_decode(q, kc, vc, tables, np.array([13, 4]), 0.5, "f64")
    for s in range(2):
        for hh in range(h):
            np.testing.assert_allclose(out[s, hh], c[hh // 4], rtol=0, atol=1e-12)


def test_two_token_closed_form():
    """Two tokens with scores scale*a and 0 give the logistic weights
    sigma(scale*a) and sigma(-scale*a) on their (distinct) value rows."""
    d = 8
    a = 3.0
    scale = 1.0 / math.sqrt(d)
    kc = np.zeros((2, 1, 2, d))
    vc = np.zeros((2, 1, 2, d))
    kc[1, 0, 0, 0] = 1.0  # token 0: k = e0
    kc[1, 0, 1, 1] = 1.0  # token 1: k = e1 (q has no e1 part -> score 0)
    vc[1, 0, 0, 2] = 1.0  # token 0: v = e2
    vc[1, 0, 1, 3] = 1.0  # token 1: v = e3
    q = np.zeros((1, 1, d))
    q[0, 0, 0] = a
    out = paged_decode(q, kc, vc, np.array([[1]]), np.array([2]), scale, "f64")[0, 0]
    w0 = 1.0 / (1.0 + math.exp(-scale * a))
    want = np.zeros(d)
    want[2] = w0
    want[3] = 1.0 - w0
    np.testing.assert_allclose(out, want, rtol=0, atol=1e-15)


def test_large_scores_do_not_overflow():
    """Scores near 1e3 would overflow exp without the max subtraction; the
    result is still the logistic closed form (here exactly the first row)."""
    d = 4
    kc = np.zeros((1, 1, 4, d))
    vc = np.zeros((1, 1, 4, d))
    kc[0, 0, 0, 0] = 1.0
    kc[0, 0, 1, 0] = 0.999
    vc[0, 0, 0] = [1, 0, 0, 0]
    vc[0, 0, 1] = [0, 1, 0, 0]
    q = np.zeros((1, 1, d))
    q[0, 0, 0] = 2000.0
    out = paged_decode(q, kc, vc, np.array([[0]]), np.array([2]), 1.0, "f64")[0, 0]
    w1 = 1.0 / (1.0 + math.exp(2000.0 * 0.001))
    np.testing.assert_allclose(out, [1 - w1, w1, 0, 0], rtol=0, atol=1e-15)
    assert np.all(np.isfinite(out))


def test_rows_past_context_and_unused_table_entries_are_ignored():
    """Rows past ctx in the last block, and table entries past the last
    block (even invalid ones), do not change the result."""
    rng = np.random.default_rng(14)
    nblk, hkv, b, d = 6, 1, 4, 8
    kc = rng.standard_normal((nblk, hkv, b, d))
    vc = rng.standard_normal((nblk, hkv, b, d))
    q = rng.standard_normal((1, 1, d))
    tab = np.array([[4, 2, 5, 0]], dtype=np.int32)
    base = paged_decode(q, kc, vc, tab, np.array([6]), 0.4, "f64")
    kc2, vc2 = kc.copy(), vc.copy()
    kc2[2, 0, 2:] = 1e6  # rows 6, 7 of the sequence: past ctx
    vc2[2, 0, 2:] = np.nan
    kc2[5] = np.nan
    tab2 = np.array([[4, 2, -7, 99]], dtype=np.int32)
    got = paged_decode(q, kc2, vc2, tab2, np.array([6]), 0.4, "f64")
    assert np.array_equal(base, got)
    # and the result is the dense softmax over exactly those 6 rows
    rows_k = np.concatenate([kc[4, 0], kc[2, 0, :2]])
    rows_v = np.concatenate([vc[4, 0], vc[2, 0, :2]])
    p = scipy.special.softmax(0.4 * rows_k @ q[0, 0])
    np.testing.assert_allclose(base[0, 0], rows_v.T @ p, rtol=0, atol=1e-12)


def test_output_is_convex_combination_of_values():
    rng = np.random.default_rng(15)
    kc = rng.standard_normal((10, 2, 8, 16)) * 3
    vc = rng.standard_normal((10, 2, 8, 16))
    q = rng.standard_normal((3, 4, 16))
    tables = rng.permutation(10)[:9].reshape(3, 3).astype(np.int32)
    ctx = np.array([24, 3, 17])
    out = paged_decode(q, kc, vc, tables, ctx, 0.25, "f64")
    for s in range(3):
        nb = -(-ctx[s] // 8)
        for kv in range(2):
            rows = vc[tables[s, :nb], kv].reshape(-1, 16)[:ctx[s]]
            lo, hi = rows.min(axis=0), rows.max(axis=0)
            for hh in (2 * kv, 2 * kv + 1):
                assert np.all(out[s, hh] >= lo - 1e-12) and np.all(out[s, hh] <= hi + 1e-12)


def test_shared_prefix_equals_unshared_copies():
    """(e) Sequences that share prefix blocks through the allocator give
    bit-identical results to sequences holding private copies."""
    rng = np.random.default_rng(16)
    b, hkv, d, h = 4, 2, 8, 4
    shared = BlockAllocator(32, b, rng.permutation(32))
    shared.add(100, 10)  # prefix of 10 tokens: the divergence is mid-block
    for s in range(3):
        shared.fork(100, s)
    pairs = []
    for s in range(3):
        for _ in range(3 + 2 * s):
            _, src, dst = shared.append_slot(s)
            if src >= 0:
                pairs.append((src, dst))
    assert len(pairs) == 3  # each child copied the partly filled block once
    kc = rng.standard_normal((32, hkv, b, d))
    vc = rng.standard_normal((32, hkv, b, d))
    for src, dst in pairs:  # the copy happens before any child's new token lands
        kc[dst] = kc[src]
        vc[dst] = vc[src]
    # the private twin: same logical token rows, own blocks
    seq_rows_k, seq_rows_v = [], []
    for s in range(3):
        t = shared.block_table(s)
        n = shared.num_tokens(s)
        seq_rows_k.append(kc[t].transpose(1, 0, 2, 3).reshape(hkv, -1, d)[:, :n])
        seq_rows_v.append(vc[t].transpose(1, 0, 2, 3).reshape(hkv, -1, d)[:, :n])
    priv = BlockAllocator(32, b)
    kp = np.zeros_like(kc)
    vp = np.zeros_like(vc)
    for s in range(3):
        n = shared.num_tokens(s)
        priv.add(s, n)
        t = priv.block_table(s)
        for j, blk in enumerate(t):
            rows = slice(j * b, min(n, (j + 1) * b))
            cnt = rows.stop - rows.start
            kp[blk, :, :cnt] = seq_rows_k[s][:, rows]
            vp[blk, :, :cnt] = seq_rows_v[s][:, rows]
    q = rng.standard_normal((3, h, d))
    ctx = np.array([shared.num_tokens(s) for s in range(3)])
    a = paged_decode(q, kc, vc, tables_array(shared, range(3), 8), ctx, 0.35, "f64")
    c = paged_decode(q, kp, vp, tables_array(priv, range(3), 8), ctx, 0.35, "f64")
    assert np.array_equal(a, c)
    # and the shared prefix really is shared: its first two full blocks
    assert shared.block_table(0)[:2] == shared.block_table(1)[:2] == shared.block_table(2)[:2]


def test_brute_force_scalar_loops_on_tiny_workload():
    """Scalar triple loop with math.exp, token by token through the
    (block, row) address, on the fp32 tiny workload."""
    w = WORKLOADS["tiny_f32"]
    ctx = context_lens(w)
    nblk = 16
    kc = random_pool(w, nblk, "k")
    vc = random_pool(w, nblk, "v")
    q = queries(w)
    order = free_order(w, nblk)
    alloc = BlockAllocator(nblk, w.block_size, order)
    for s in range(w.num_seqs):
        alloc.add(s, int(ctx[s]))
    tables = tables_array(alloc, range(w.num_seqs), 4)
    out = paged_decode(q, kc, vc, tables, ctx, w.scale, "f32")
    for s in range(w.num_seqs):
        for hh in range(w.num_heads):
            scores = []
            for t in range(ctx[s]):
                blk = tables[s][t // w.block_size]
                acc = 0.0
                for dd in range(w.head_dim):
                    acc += float(q[s, hh, dd]) * float(kc[blk, hh, t % w.block_size, dd])
                scores.append(acc * w.scale)
            mx = max(scores)
            e = [math.exp(x - mx) for x in scores]
            tot = sum(e)
            for dd in range(0, w.head_dim, 7):
                val = 0.0
                for t in range(ctx[s]):
                    blk = tables[s][t // w.block_size]
                    val += e[t] / tot * float(vc[blk, hh, t % w.block_size, dd])
                assert abs(out[s, hh, dd] - val) <= 1e-12 * max(1.0, abs(val))


@pytest.mark.parametrize("name", ["mha_bf16", "gqa_prefix_bf16"])
def test_bf16_inputs_are_exact_in_fp64(name):
    """Stored bf16 values enter the fp64 computation unchanged: the oracle
    on bf16 bits equals the oracle on the same values given as fp32."""
    w = WORKLOADS[name].replace(num_seqs=2, ctx_dist="uniform", ctx_lo=5, ctx_hi=40,
                                prefix_len=0, prefix_share=0)
    ctx = context_lens(w)
    kc = random_pool(w, 8, "k")
    vc = random_pool(w, 8, "v")
    q = queries(w)
    tables = np.array([[0, 3, 5], [7, 1, 2]], dtype=np.int32)
    a = paged_decode(q, kc, vc, tables, ctx, w.scale, "bf16")
    f32 = lambda x: to_f64(x, "bf16").astype(np.float32)  # noqa: E731
    c = paged_decode(f32(q), f32(kc), f32(vc), tables, ctx, w.scale, "f32")
    assert np.array_equal(a, c)
