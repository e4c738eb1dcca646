"""Paged decode on the GPU against the fp64 oracle, element by element.

Tolerances: bf16 storage with fp32 accumulation |gpu - ref| <= 2e-2 +
1e-2 |ref|; fp32 storage 1e-5 + 1e-5 |ref|.
"""

import numpy as np
import pytest
import torch

from tests._cases import as_f64, assert_close, make_decode_case, run_decode, to_dev
from tests._lib_fixture import ensure_built
from workloads import WORKLOADS, Workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    ensure_built()
    import paged_kv_cache_216_gb300 as pa

    return pa


def test_tiny_f32_workload(pa):
    case = make_decode_case(WORKLOADS["tiny_f32"])
    out = run_decode(case)
    assert_close(out, case.oracle(), "f32", "tiny_f32")
    assert pa.get_status() == 0


# Reduced versions of each workload: several tiles, partitions and ragged tails.
SMALL = {
    "mha_small": WORKLOADS["mha_bf16"].replace(num_seqs=6, num_heads=4, num_kv_heads=4, ctx_hi=700),
    "gqa_prefix_small": WORKLOADS["gqa_prefix_bf16"].replace(num_seqs=6, num_heads=16, num_kv_heads=4,
                                                             ctx_lo=40, ctx_hi=900, prefix_len=100,
                                                             prefix_share=3),
    "long_small": WORKLOADS["long_bf16"].replace(num_seqs=3, num_heads=16, num_kv_heads=2, ctx_lo=1100,
                                                 ctx_hi=3000),
    "serving_b8_small": WORKLOADS["serving_bf16_b8"].replace(num_seqs=9, num_heads=8, num_kv_heads=2,
                                                             ctx_mean=150.0, ctx_hi=600, steps=0),
    "d64_g2_b32": Workload(name="d64", dtype="bf16", num_seqs=5, num_heads=4, num_kv_heads=2, head_dim=64,
                           block_size=32, seed=21, ctx_lo=1, ctx_hi=800),
    "f32_g8_d128_b8": Workload(name="f32big", dtype="f32", num_seqs=3, num_heads=16, num_kv_heads=2, head_dim=128,
                               block_size=8, seed=22, ctx_lo=1, ctx_hi=700),
}


@pytest.mark.parametrize("name", sorted(SMALL))
@pytest.mark.parametrize("partition", [0, 64, 4096])
def test_small_workloads(pa, name, partition):
    w = SMALL[name]
    case = make_decode_case(w)
    out = run_decode(case, partition_size=partition)
    assert_close(out, case.oracle(), w.dtype, f"{name} P={partition}")
    assert pa.get_status() == 0


@pytest.mark.parametrize("b", [8, 16, 32])
@pytest.mark.parametrize("g", [1, 4, 8])
def test_context_length_edges(pa, b, g):
    """Lengths at block, 32-token chunk and partition boundaries."""
    ctx = np.array([1, 2, 7, 8, 9, 15, 16, 17, 31, 32, 33, 63, 64, 65, 511, 512, 513, 1023, 1024, 1025],
                   dtype=np.int32)
    w = Workload(name="edges", dtype="bf16", num_seqs=len(ctx), num_heads=2 * g, num_kv_heads=2, head_dim=128,
                 block_size=b, seed=23 + b + g, ctx_dist="fixed", ctx_fixed=tuple(ctx))
    case = make_decode_case(w, ctx=ctx)
    ref = case.oracle()
    for partition in (512, 64, 0):
        assert_close(run_decode(case, partition_size=partition), ref, "bf16", f"B={b} g={g} P={partition}")


def test_many_items_per_cta_wrap_the_pipeline(pa):
    """Small partitions over many (sequence, KV head) pairs give every
    persistent CTA a dozen or more work items, so its stage and query rings
    wrap many times."""
    w = Workload(name="wrap", dtype="bf16", num_seqs=64, num_heads=32, num_kv_heads=8, head_dim=128,
                 block_size=16, seed=25, ctx_lo=200, ctx_hi=420)
    case = make_decode_case(w)
    for partition in (32, 64, 4096):
        assert_close(run_decode(case, partition_size=partition), case.oracle(), "bf16", f"P={partition}")
    assert pa.get_status() == 0


@pytest.mark.parametrize("name", ["gqa_prefix_small", "serving_b8_small", "long_small"])
def test_host_plan_gives_identical_output(pa, name):
    """pa_decode_planned with the host-built work list equals pa_decode
    (device-built list) bit for bit: every item is computed the same way
    whichever CTA takes it, and partitions merge in a fixed order."""
    from paged_kv_cache_216_gb300 import ops

    w = SMALL[name]
    case = make_decode_case(w)
    p = ops.decode_partition_size(w.num_seqs, w.num_kv_heads, case.max_ctx, 64)
    ref = ops.paged_decode(case.q_d, case.k_cache, case.v_cache, case.tables_d, case.ctx_d, case.max_ctx, w.scale,
                           partition_size=p)
    plan_h = np.zeros(ops.decode_plan_bytes(w.num_seqs, case.max_ctx, p), dtype=np.uint8)
    ops.decode_plan_host(case.ctx, case.max_ctx, p, plan_h)
    ws = ops.decode_workspace(w.num_seqs, w.num_heads, w.num_kv_heads, w.head_dim, case.max_ctx, p)
    out = torch.empty_like(case.q_d)
    for _ in range(2):  # a fresh copy of the list each call
        plan_d = torch.from_numpy(plan_h).cuda()
        ops.paged_decode_planned(case.q_d, case.k_cache, case.v_cache, case.tables_d, case.ctx_d, case.max_ctx,
                                 w.scale, out, plan_d, ws, p)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert pa.get_status() == 0


def test_split_and_unsplit_agree(pa):
    w = SMALL["long_small"]
    case = make_decode_case(w)
    a = as_f64(run_decode(case, partition_size=32))
    c = as_f64(run_decode(case, partition_size=4096))
    np.testing.assert_allclose(a, c, atol=2e-2, rtol=1e-2)


def test_single_token_returns_value_row(pa):
    w = Workload(name="one", dtype="bf16", num_seqs=3, num_heads=8, num_kv_heads=2, head_dim=128, block_size=16,
                 seed=24, ctx_dist="fixed", ctx_fixed=(1, 1, 1))
    case = make_decode_case(w, ctx=np.array([1, 1, 1], dtype=np.int32))
    out = run_decode(case)
    for s in range(3):
        blk = case.tables[s, 0]
        for h in range(8):
            v_row = case.v_pool[blk, h // 4, 0]
            got = out[s, h].cpu().view(torch.int16).numpy().view(np.uint16)
            assert np.array_equal(got, v_row)  # softmax of one score is 1: out = V_0 exactly


@pytest.mark.parametrize("b", [8, 16])
def test_garbage_past_context_does_not_leak(pa, b):
    """Rows past the context in the last block (never written in serving)
    hold NaN/Inf: the output must not see them."""
    w = SMALL["serving_b8_small"].replace(block_size=b)
    case = make_decode_case(w)
    ref = case.oracle()
    kd = case.k_cache.view(torch.int16)
    vd = case.v_cache.view(torch.int16)
    for s, n in enumerate(case.ctx):
        nb = -(-int(n) // w.block_size)
        last = int(case.tables[s, nb - 1])
        r = int(n) - (nb - 1) * w.block_size
        if r < w.block_size:
            kd[last, :, r:] = 0x7FC0  # NaN
            vd[last, :, r:] = 0x7F80  # +Inf
    out = run_decode(case, partition_size=64)
    assert torch.isfinite(out.float()).all()
    assert_close(out, ref, "bf16", "garbage tail")


def test_bad_context_and_block_are_flagged_not_faulted(pa):
    w = SMALL["mha_small"]
    case = make_decode_case(w)
    pa.get_status()
    ctx = case.ctx.copy()
    ctx[1] = 0
    out = pa.paged_decode(case.q_d, case.k_cache, case.v_cache, case.tables_d, to_dev(ctx), case.max_ctx, w.scale)
    st = pa.get_status()
    assert st & pa._lib.PA_STATUS_BAD_CONTEXT
    assert (out[1].float() == 0).all()
    others = [s for s in range(w.num_seqs) if s != 1]
    assert_close(out[others], case.oracle(others), "bf16", "other sequences")
    tables = case.tables.copy()
    tables[0, 0] = case.num_blocks + 5
    pa.paged_decode(case.q_d, case.k_cache, case.v_cache, to_dev(tables), case.ctx_d, case.max_ctx, w.scale)
    assert pa.get_status() & pa._lib.PA_STATUS_BAD_BLOCK


# Full-size workloads in the launch configuration the benchmark uses; the
# oracle checks a sample of sequences, every output is checked finite.
FULL_SAMPLES = {"mha_bf16": [0, 7, 31], "gqa_prefix_bf16": [0, 31, 32, 63], "long_bf16": [2, 5]}


@pytest.mark.parametrize("name", sorted(FULL_SAMPLES))
def test_full_size_workloads_sampled(pa, name):
    w = WORKLOADS[name]
    case = make_decode_case(w)
    out = run_decode(case)
    assert torch.isfinite(out.float()).all()
    seqs = FULL_SAMPLES[name]
    if name == "long_bf16":
        seqs = sorted({int(np.argmax(case.ctx)), int(np.argmin(case.ctx))} | set(seqs))
    assert_close(out[seqs], case.oracle(seqs), "bf16", name)
    assert pa.get_status() == 0
    if name == "gqa_prefix_bf16":
        # sharing sequences really read the same physical prefix blocks
        m = w.prefix_len // w.block_size
        assert (case.tables[: w.prefix_share, :m] == case.tables[0, :m]).all()
