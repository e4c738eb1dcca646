"""Shared-prefix decode on the GPU against the fp64 oracle.

The result is defined as that of plain paged decode over each sequence's
own block table (the oracle's definition): only which work items read the
shared blocks differs.  Tolerance as for decode: |gpu - ref| <= 2e-2 +
1e-2 |ref| (bf16 storage, fp32 accumulation).
"""

import numpy as np
import pytest
import torch

from oracle.attention import paged_decode as oracle_decode
from tests._cases import as_f64, assert_close, make_decode_case, to_dev
from tests._lib_fixture import ensure_built
from workloads import WORKLOADS, normal

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    ensure_built()
    import paged_kv_cache_216_gb300 as pa

    return pa


def _grouped(seed, S, H, Hkv, D, B, groups, ctx, shared_blocks=None):
    """Seeded batch whose groups share their prefix blocks: group
    (first, count, prefix) members hold the same physical blocks for their
    first ``shared_blocks`` (default ceil(prefix / B)) table entries, every
    other block is the sequence's own; the pool is shuffled."""
    ctx = np.asarray(ctx, dtype=np.int32)
    width = -(-int(ctx.max()) // B)
    rng = np.random.default_rng(seed)
    need = int(sum(-(-int(c) // B) for c in ctx)) + 8
    N = need + 5
    perm = rng.permutation(N).astype(np.int32)
    nxt = iter(perm.tolist())
    tables = np.full((S, width), -1, dtype=np.int32)
    member = {}
    for gi, (first, count, prefix) in enumerate(groups):
        nsh = -(-prefix // B) if shared_blocks is None else shared_blocks[gi]
        shared = [next(nxt) for _ in range(nsh)]
        for s in range(first, first + count):
            member[s] = shared
    for s in range(S):
        nb = -(-int(ctx[s]) // B)
        shared = member.get(s, [])
        row = shared[:nb] + [next(nxt) for _ in range(max(0, nb - len(shared)))]
        tables[s, :len(row)] = row
    k = normal((N, Hkv, B, D), 1.0, "bf16", seed, 11)
    v = normal((N, Hkv, B, D), 1.0, "bf16", seed, 12)
    q = normal((S, H, D), 1.0, "bf16", seed, 13)
    return dict(q=q, k=k, v=v, tables=tables, ctx=ctx, N=N, scale=1.0 / np.sqrt(D))


def _run(pa, c, groups, P, plain=False):
    q, kc, vc = to_dev(c["q"]), to_dev(c["k"]), to_dev(c["v"])
    tab, ctx = to_dev(c["tables"]), to_dev(c["ctx"])
    mx = int(c["ctx"].max())
    if plain:
        return pa.paged_decode(q, kc, vc, tab, ctx, mx, c["scale"], partition_size=P)
    return pa.paged_decode_shared_prefix(q, kc, vc, tab, ctx, mx, c["scale"], groups, partition_size=P)


def _oracle(c):
    return oracle_decode(c["q"], c["k"], c["v"], c["tables"], c["ctx"], c["scale"], "bf16")


# name: (seed, S, H, Hkv, D, B, P, groups, context-length range of the batch)
CASES = {
    # GQA g = 4, one group of 5 of 7 sequences, 4 shared partitions
    "g4_d128_b16": (31, 7, 16, 4, 128, 16, 64, [(0, 5, 256)], (256, 700)),
    # MHA g = 1, head_dim 64, two groups with sequences outside both
    "g1_d64_b32": (32, 8, 4, 4, 64, 32, 64, [(1, 3, 128), (4, 2, 320)], (320, 900)),
    # g = 8 with 12 members: 96 of the 128 rows of a tile, block size 8
    "g8_d128_b8": (33, 13, 16, 2, 128, 8, 32, [(0, 12, 96)], (96, 400)),
    # g = 8 with 20 members: 160 rows, two tiles per shared partition
    "g8_two_tiles": (37, 23, 16, 2, 128, 16, 64, [(1, 20, 128)], (128, 420)),
    # g = 4 with 40 members: 160 rows, two tiles (the second one partly empty)
    "g4_40_members": (38, 44, 8, 2, 128, 16, 64, [(2, 40, 192)], (192, 480)),
    # a one-member group and a prefix that is not a whole number of partitions
    "g2_ragged_groups": (34, 9, 8, 4, 128, 16, 128, [(0, 1, 256), (2, 4, 384), (6, 3, 200)], (384, 1100)),
    # the GQA prefix workload's shape at a smaller batch: 1024-token prefix, P = 512
    "g4_p512": (35, 9, 32, 8, 128, 16, 512, [(0, 6, 1024)], (1025, 2600)),
    # 20 members of g = 4: 80 rows in two tiles
    "g4_80_rows": (36, 22, 8, 2, 128, 32, 64, [(0, 20, 192)], (192, 500)),
    # the library's partition choice (P 0): 128 for plain decode of this
    # batch, lengthened to 1024 (the whole prefix) with the group
    "g4_auto_partition": (39, 9, 32, 8, 128, 16, 0, [(0, 6, 1024)], (1025, 2600)),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_shared_prefix_matches_oracle(pa, name):
    seed, S, H, Hkv, D, B, P, groups, (lo, hi) = CASES[name]
    rng = np.random.default_rng(seed)
    ctx = rng.integers(lo, hi + 1, size=S)
    for first, count, prefix in groups:  # members hold at least the prefix
        ctx[first:first + count] = np.maximum(ctx[first:first + count], prefix)
    c = _grouped(seed, S, H, Hkv, D, B, groups, ctx)
    out = _run(pa, c, groups, P)
    ref = _oracle(c)
    torch.cuda.synchronize()
    assert_close(out, ref, "bf16", name)
    plain = _run(pa, c, groups, P, plain=True)
    assert_close(out, as_f64(plain), "bf16", f"{name} vs plain decode")
    assert pa.get_status() == 0


def test_member_contexts_at_and_inside_the_shared_part(pa):
    """Members whose context ends exactly where the shared partitions end
    (every partition shared, also a single one), and members whose context
    ends inside the shared part (masked there)."""
    S, P, B = 8, 64, 16
    groups = [(0, 4, 256), (4, 3, 64)]
    ctx = np.array([256, 300, 100, 64 + 7, 64, 65, 500, 333], dtype=np.int32)
    c = _grouped(40, S, 8, 2, 128, B, groups, ctx)
    out = _run(pa, c, groups, P)
    ref = _oracle(c)
    torch.cuda.synchronize()
    assert_close(out, ref, "bf16", "edge contexts")
    assert pa.get_status() == 0


def test_empty_member_gets_zero_row(pa):
    groups = [(0, 3, 128)]
    ctx = np.array([300, 200, 150, 90], dtype=np.int32)
    c = _grouped(41, 4, 8, 4, 128, 16, groups, ctx)
    c["ctx"] = ctx.copy()
    c["ctx"][1] = 0
    out = _run(pa, c, groups, 64)
    torch.cuda.synchronize()
    assert torch.all(out[1] == 0)
    keep = [0, 2, 3]
    ref = oracle_decode(c["q"], c["k"], c["v"], c["tables"], c["ctx"], c["scale"], "bf16", keep)
    assert_close(out[keep], ref, "bf16", "other sequences")
    assert pa.get_status() == pa._lib.PA_STATUS_BAD_CONTEXT


def test_host_plan_equals_device_plan_bitwise(pa):
    """The host-built list without the shared partitions and the device
    planner give bit-identical outputs (same kernels, same per-item work)."""
    from paged_kv_cache_216_gb300 import ops

    seed, S, H, Hkv, D, B, P, groups, (lo, hi) = CASES["g2_ragged_groups"]
    rng = np.random.default_rng(seed)
    ctx = rng.integers(lo, hi + 1, size=S).astype(np.int32)
    c = _grouped(seed, S, H, Hkv, D, B, groups, ctx)
    dev = _run(pa, c, groups, P)
    mx = int(ctx.max())
    plan_h = np.zeros(ops.decode_plan_bytes(S, mx, P), dtype=np.uint8)
    ops.decode_plan_host(ctx, mx, P, plan_h, prefix_groups=groups, num_heads=H, num_kv_heads=Hkv)
    plan_d = torch.from_numpy(plan_h).cuda()
    q, kc, vc = to_dev(c["q"]), to_dev(c["k"]), to_dev(c["v"])
    ws = ops.decode_workspace(S, H, Hkv, D, mx, P, q.device)
    out = torch.empty_like(q)
    ops.paged_decode_planned(q, kc, vc, to_dev(c["tables"]), to_dev(ctx), mx, c["scale"], out, plan_d, ws, P,
                             prefix_groups=groups)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), dev.view(torch.int16))
    assert pa.get_status() == 0


def test_groups_shorter_than_a_partition_fall_back_to_plain_decode(pa):
    groups = [(0, 4, 60)]
    ctx = np.array([300, 200, 150, 90, 77], dtype=np.int32)
    c = _grouped(42, 5, 8, 4, 128, 16, groups, ctx)
    out = _run(pa, c, groups, 64)
    plain = _run(pa, c, groups, 64, plain=True)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), plain.view(torch.int16))
    assert pa.get_status() == 0


def test_gqa_prefix_workload_full_size(pa):
    """The GQA prefix-sharing batch at full size (64 sequences, 32 of them on
    one 1024-token prefix): sampled sequences against the oracle, every
    output against plain decode."""
    w = WORKLOADS["gqa_prefix_bf16"]
    case = make_decode_case(w)
    groups = [(0, w.prefix_share, w.prefix_len // w.block_size * w.block_size)]
    out = pa.paged_decode_shared_prefix(case.q_d, case.k_cache, case.v_cache, case.tables_d, case.ctx_d,
                                        case.max_ctx, w.scale, groups)
    plain = pa.paged_decode(case.q_d, case.k_cache, case.v_cache, case.tables_d, case.ctx_d, case.max_ctx, w.scale)
    torch.cuda.synchronize()
    assert_close(out, as_f64(plain), "bf16", "vs plain decode")
    rng = np.random.default_rng(5)
    seqs = sorted(set(rng.choice(w.prefix_share, 3, replace=False).tolist()) | {40, int(np.argmax(case.ctx))})
    assert_close(out[seqs], case.oracle(seqs), "bf16", "sampled vs oracle")
    assert pa.get_status() == 0


def test_serving_engine_with_prefix_groups(pa):
    """Serving steps of a batch whose first sequences fork from one prompt
    that ends inside a block (each member's first append copies that
    block): the engine decodes with the group's shared blocks and matches
    the oracle's serving loop step by step."""
    from oracle.cache import copy_blocks
    from oracle.serving import ServingOracle, initial_state
    from paged_kv_cache_216_gb300.prefix import populate
    from tests._cases import to_bits
    from workloads import context_lens, free_order, pool_blocks, random_pool, serving_step_tokens

    w = WORKLOADS["gqa_prefix_bf16"].replace(num_seqs=9, num_heads=16, num_kv_heads=4, ctx_lo=150, ctx_hi=700,
                                             prefix_len=200, prefix_share=5, partition_size=64, steps=6)
    ctx = context_lens(w)
    nb = pool_blocks(w, ctx, extra_steps=w.steps) + w.prefix_share
    order = free_order(w, nb)
    k_pool, v_pool = random_pool(w, nb, "k"), random_pool(w, nb, "v")
    alloc = pa.BlockAllocator(nb, w.block_size, order)
    cpairs = populate(alloc, ctx, w.prefix_len, w.prefix_share)
    kd, vd = to_dev(k_pool), to_dev(v_pool)
    if len(cpairs):
        pa.copy_blocks(kd, vd, to_dev(cpairs))
    shared = w.prefix_len // w.block_size * w.block_size  # tokens in blocks still shared after the copies
    groups = [(0, w.prefix_share, shared)]
    eng = pa.ServingEngine(kd, vd, alloc, np.arange(w.num_seqs), w.num_heads, w.scale, int(ctx.max()) + w.steps,
                           w.partition_size, prefix_groups=groups)
    o, opairs = initial_state(w.num_seqs, w.block_size, ctx, nb, order, w.prefix_len, w.prefix_share)
    copy_blocks(k_pool, v_pool, opairs)
    orc = ServingOracle(o, k_pool, v_pool, w.num_seqs, w.dtype, w.scale)
    for step in range(w.steps):
        q, k, v = serving_step_tokens(w, step)
        out = eng.step(to_dev(q), to_dev(k), to_dev(v))
        slots, _, ref = orc.step(q, k, v, eng.width)
        torch.cuda.synchronize()
        assert np.array_equal(eng.slots_h.numpy(), slots)
        assert np.array_equal(to_bits(eng.k_cache), orc.k_cache)
        assert_close(out, ref, "bf16", f"step {step}")
    assert pa.get_status() == 0
