"""The serving loop (allocate -> copy-on-write -> append -> decode) on the GPU
against the oracle's own serving loop: slots, block tables and caches
bit-exact, decode outputs within the bf16 tolerance."""

import numpy as np
import pytest
import torch

from oracle.allocator import BlockAllocator as OracleAllocator
from oracle.serving import ServingOracle, initial_state
from tests._cases import assert_close, to_bits, to_dev
from tests._lib_fixture import ensure_built
from workloads import WORKLOADS, context_lens, free_order, pool_blocks, random_pool, serving_step_tokens

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    ensure_built()
    import paged_kv_cache_216_gb300 as pa

    return pa


def _engine_and_oracle(pa, w, steps, fork_pairs=()):
    """Both sides' serving state.  ``fork_pairs`` = (parent, child): the child
    is forked from the parent instead of being added, so the first append of
    the step copies their shared partly filled last block."""
    from paged_kv_cache_216_gb300.prefix import populate

    ctx = context_lens(w)
    for parent, child in fork_pairs:
        ctx[child] = ctx[parent]
    nb = pool_blocks(w, ctx, extra_steps=steps) + len(fork_pairs) + w.prefix_share
    order = free_order(w, nb)
    k_pool = random_pool(w, nb, "k")
    v_pool = random_pool(w, nb, "v")
    children = {c for _, c in fork_pairs}
    # CUDA path
    c = pa.BlockAllocator(nb, w.block_size, order)
    o = OracleAllocator(nb, w.block_size, order)
    if fork_pairs:
        for s in range(w.num_seqs):
            if s not in children:
                c.add(s, int(ctx[s]))
                o.add(s, int(ctx[s]))
        for parent, child in fork_pairs:
            c.fork(parent, child)
            o.fork(parent, child)
        cpairs = np.zeros((0, 2), np.int32)
        opairs = []
    else:
        cpairs = populate(c, ctx, w.prefix_len, w.prefix_share)
        o, opairs = initial_state(w.num_seqs, w.block_size, ctx, nb, order, w.prefix_len, w.prefix_share)
    kd, vd = to_dev(k_pool), to_dev(v_pool)
    if len(cpairs):
        pa.copy_blocks(kd, vd, to_dev(cpairs))
    eng = pa.ServingEngine(kd, vd, c, np.arange(w.num_seqs), w.num_heads, w.scale,
                           int(ctx.max()) + steps, w.partition_size)
    from oracle.cache import copy_blocks

    copy_blocks(k_pool, v_pool, opairs)
    orc = ServingOracle(o, k_pool, v_pool, w.num_seqs, w.dtype, w.scale)
    return eng, orc


def test_serving_small_with_copy_on_write(pa):
    w = WORKLOADS["serving_bf16_b16"].replace(num_seqs=7, num_heads=8, num_kv_heads=2, ctx_mean=60.0,
                                              ctx_hi=200, prefix_len=37, prefix_share=0)
    steps = 6
    eng, orc = _engine_and_oracle(pa, w, steps, fork_pairs=[(0, 1), (4, 6)])
    total_cow = 0
    for step in range(steps):
        q, k, v = serving_step_tokens(w, step)
        out = eng.step(to_dev(q), to_dev(k), to_dev(v))
        slots, pairs, ref = orc.step(q, k, v, eng.width)
        torch.cuda.synchronize()
        assert np.array_equal(eng.slots_h.numpy(), slots)
        assert np.array_equal(eng.ctx_h.numpy(), orc.context_lens())
        assert np.array_equal(eng.tables_h.numpy(), orc.tables(eng.width))
        total_cow += len(pairs)
        assert np.array_equal(to_bits(eng.k_cache), orc.k_cache)
        assert np.array_equal(to_bits(eng.v_cache), orc.v_cache)
        assert_close(out, ref, "bf16", f"step {step}")
    assert total_cow >= 1  # a shared partly filled block was copied
    assert pa.get_status() == 0


@pytest.mark.parametrize("b", [8, 16, 32])
def test_serving_full_size(pa, b):
    """The serving workload at full size (256 sequences, 20 steps): every
    step's slots, tables and appended rows exact; decode outputs of sampled
    sequences checked against the oracle on three of the steps."""
    w = WORKLOADS[f"serving_bf16_b{b}"]
    eng, orc = _engine_and_oracle(pa, w, w.steps)
    rng = np.random.default_rng(b)
    for step in range(w.steps):
        q, k, v = serving_step_tokens(w, step)
        out = eng.step(to_dev(q), to_dev(k), to_dev(v))
        check = step in (0, w.steps // 2, w.steps - 1)
        seqs = sorted(set(rng.choice(w.num_seqs, 3, replace=False).tolist()) | {int(np.argmax(orc.context_lens()))}) \
            if check else []
        slots, pairs, ref = orc.step(q, k, v, eng.width, seqs=seqs)
        torch.cuda.synchronize()
        assert not pairs
        assert np.array_equal(eng.slots_h.numpy(), slots)
        assert np.array_equal(eng.tables_h.numpy(), orc.tables(eng.width))
        blk = torch.from_numpy(slots // b).cuda()
        row = torch.from_numpy(slots % b).cuda()
        got_k = to_bits(eng.k_cache[blk, :, row])
        assert np.array_equal(got_k, k)
        got_v = to_bits(eng.v_cache[blk, :, row])
        assert np.array_equal(got_v, v)
        if check:
            assert torch.isfinite(out.float()).all()
            assert_close(out[seqs], ref, "bf16", f"B={b} step {step}")
    assert pa.get_status() == 0


def test_serving_graph_replay_matches_oracle(pa):
    """The captured step (upload, append, plan, decode, merge as one CUDA
    graph) replayed step after step gives the oracle's slots, caches and
    outputs; the copy-on-write of a fork runs eagerly just before the first
    replay."""
    from paged_kv_cache_216_gb300.serving import graphs_supported

    if not graphs_supported():
        pytest.skip("this torch cannot record events inside a CUDA graph")
    # one eager decode first: it sets up the library's per-device state
    z = torch.zeros((1, 2, 128), dtype=torch.bfloat16, device="cuda")
    zc = torch.zeros((2, 2, 8, 128), dtype=torch.bfloat16, device="cuda")
    pa.paged_decode(z, zc, zc, torch.zeros((1, 1), dtype=torch.int32, device="cuda"),
                    torch.ones(1, dtype=torch.int32, device="cuda"), 1, 1.0)
    w = WORKLOADS["serving_bf16_b8"].replace(num_seqs=6, num_heads=16, num_kv_heads=2, ctx_mean=400.0,
                                             ctx_hi=1500, partition_size=128)
    ctx = context_lens(w)
    parent = int(np.argmax(ctx % w.block_size != 0))  # a partly filled last block to share
    child = (parent + 1) % w.num_seqs
    steps = 7
    eng, orc = _engine_and_oracle(pa, w, steps, fork_pairs=[(parent, child)])
    graph = eng.capture()
    ncow = 0
    for step in range(steps):
        q, k, v = serving_step_tokens(w, step)
        out = eng.replay(graph, to_dev(q), to_dev(k), to_dev(v)).clone()
        slots, pairs, ref = orc.step(q, k, v, eng.width)
        ncow += len(pairs)
        torch.cuda.synchronize()
        assert np.array_equal(eng.slots_h.numpy(), slots)
        assert np.array_equal(eng.tables_h.numpy(), orc.tables(eng.width))
        assert np.array_equal(to_bits(eng.k_cache), orc.k_cache)
        assert np.array_equal(to_bits(eng.v_cache), orc.v_cache)
        assert_close(out, ref, "bf16", f"graph step {step}")
    assert ncow == 1
    assert pa.get_status() == 0


@pytest.mark.parametrize("use_graph", [False, True])
def test_serving_host_buffers_match_oracle(pa, use_graph):
    """Steps driven from pinned host buffers (tokens uploaded on the side
    stream, output copied back on a third) give the oracle's outputs."""
    from paged_kv_cache_216_gb300.serving import graphs_supported

    if use_graph and not graphs_supported():
        pytest.skip("this torch cannot record events inside a CUDA graph")
    w = WORKLOADS["serving_bf16_b16"].replace(num_seqs=5, num_heads=16, num_kv_heads=4, ctx_mean=300.0,
                                              ctx_hi=1200)
    steps = 5
    eng, orc = _engine_and_oracle(pa, w, steps + 1)  # + the eager first step
    q0, k0, v0 = serving_step_tokens(w, 99)
    eng.step(to_dev(q0), to_dev(k0), to_dev(v0))  # an eager step first
    orc.step(q0, k0, v0, eng.width, seqs=[])
    graphs = eng.capture() if use_graph else None

    def pinned(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).pin_memory()

    outs, refs = [], []
    for step in range(steps):
        q, k, v = serving_step_tokens(w, step)
        out_h = torch.empty((w.num_seqs, w.num_heads, w.head_dim), dtype=torch.bfloat16).pin_memory()
        if use_graph:  # one packed host buffer per step
            eng.step_host(out_h=out_h, graphs=graphs, packed=eng.pack_tokens(pinned(q), pinned(k), pinned(v), pin=True))
        else:
            eng.step_host(pinned(q), pinned(k), pinned(v), out_h, graphs=graphs)
        outs.append(out_h)
        refs.append(orc.step(q, k, v, eng.width)[2])
    torch.cuda.synchronize()
    for step, (o, r) in enumerate(zip(outs, refs)):
        assert_close(o, r, "bf16", f"host step {step}")
    assert pa.get_status() == 0
