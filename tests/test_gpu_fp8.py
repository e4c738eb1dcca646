"""FP8 (E4M3) KV storage on the GPU against the oracle.

Append: the stored codes must equal the oracle's quantization bit for bit
(NaN inputs: any NaN code).  Decode: within the bf16 tolerance of the
fp64 oracle over the same codes, |gpu - ref| <= 2e-2 + 1e-2 |ref|; the
kernel's only roundings are q to fp16 (exact in range), the softmax
weights to fp16 (relative 2^-11) and fp32 accumulation.
"""

import numpy as np
import pytest
import torch

from oracle import fp8 as ofp8
from oracle.attention import paged_decode as oracle_decode
from oracle.cache import bf16_to_f32, cache_append_fp8, quantize_pool_fp8
from tests._cases import assert_close, make_decode_case, to_bits, to_dev
from tests._lib_fixture import ensure_built
from workloads import WORKLOADS, Workload, bf16_bits, context_lens, free_order, pool_blocks, random_pool

pytestmark = pytest.mark.gpu

K_SCALE, V_SCALE = 0.05, 0.0173


@pytest.fixture(scope="module")
def pa():
    ensure_built()
    import paged_kv_cache_216_gb300 as pa

    return pa


def _codes(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.uint8).numpy()


def _fp8_cache(shape, device="cuda"):
    dt = getattr(torch, "float8_e4m3fn", torch.uint8)
    return torch.zeros(shape, dtype=torch.uint8, device=device).view(dt)


def _quantize_on_gpu(pa, pool_d: torch.Tensor, scale_k: float, scale_v: float, v_pool_d: torch.Tensor):
    """Both bf16 pools [N, Hkv, B, D] into E4M3 caches through the append
    kernel, one slot per token row."""
    n, hkv, b, d = pool_d.shape
    kt = pool_d.permute(0, 2, 1, 3).reshape(n * b, hkv, d).contiguous()
    vt = v_pool_d.permute(0, 2, 1, 3).reshape(n * b, hkv, d).contiguous()
    slots = torch.arange(n * b, dtype=torch.int64, device=pool_d.device)
    kc, vc = _fp8_cache(pool_d.shape), _fp8_cache(pool_d.shape)
    pa.cache_append_fp8(kt, vt, slots, kc, vc, scale_k, scale_v)
    return kc, vc


def test_append_fp8_is_bit_exact(pa):
    """Random tokens plus zeros, signed zeros, values that underflow, tie
    exactly between two codes, saturate, and infinities/NaN, into random
    slots of a pool (untouched slots keep their codes)."""
    rng = np.random.default_rng(50)
    n, hkv, b, d, t = 9, 3, 16, 128, 40
    x = rng.standard_normal((t, hkv, d)).astype(np.float32)
    scale = 0.25  # a power of two: x / scale is exact, ties stay ties
    pos = ofp8.DECODE[:0x7F]
    mids = ((pos[:-1] + pos[1:]) / 2)  # exact midpoints between codes
    x[0, 0, :len(mids[:128])] = (mids[:128] * scale).astype(np.float32)
    x[1, 0, :8] = np.array([0.0, -0.0, 1e-8, -1e-8, 500.0, -1e6, np.inf, -np.inf], dtype=np.float32)
    x[1, 1, 0] = np.nan
    kbits = bf16_bits(x)
    vbits = bf16_bits(rng.standard_normal((t, hkv, d)).astype(np.float32) * np.float32(3.0))
    slots = rng.permutation(n * b)[:t].astype(np.int64)
    slots[[5, 11]] = -1
    init = rng.integers(0, 0x7F, size=(n, hkv, b, d)).astype(np.uint8)
    kc = torch.from_numpy(init.copy()).cuda()
    vc = torch.from_numpy(init.copy()).cuda()
    pa.cache_append_fp8(to_dev(kbits), to_dev(vbits), torch.from_numpy(slots).cuda(), kc, vc, scale, 0.0173)
    torch.cuda.synchronize()
    want_k, want_v = cache_append_fp8(init, init, kbits, vbits, slots, scale, 0.0173)
    got_k, got_v = _codes(kc), _codes(vc)
    nan_k = (want_k & 0x7F) == 0x7F
    assert np.array_equal((got_k & 0x7F) == 0x7F, nan_k)
    assert np.array_equal(got_k[~nan_k], want_k[~nan_k])
    assert np.array_equal(got_v, want_v)
    assert pa.get_status() == 0


SMALL = {
    "mha_g1_b16": WORKLOADS["mha_bf16"].replace(num_seqs=6, num_heads=4, num_kv_heads=4, ctx_hi=700),
    "gqa_g4_b16": WORKLOADS["gqa_prefix_bf16"].replace(num_seqs=6, num_heads=16, num_kv_heads=4, ctx_lo=40,
                                                       ctx_hi=900, prefix_len=100, prefix_share=3),
    "long_g8_b32": WORKLOADS["long_bf16"].replace(num_seqs=3, num_heads=16, num_kv_heads=2, ctx_lo=1100,
                                                  ctx_hi=3000),
    "serving_g4_b8": WORKLOADS["serving_bf16_b8"].replace(num_seqs=9, num_heads=8, num_kv_heads=2, ctx_mean=150.0,
                                                          ctx_hi=600, steps=0),
    "g2_b32": Workload(name="g2", dtype="bf16", num_seqs=5, num_heads=4, num_kv_heads=2, head_dim=128,
                       block_size=32, seed=61, ctx_lo=1, ctx_hi=800),
    # 8-token blocks with an odd number of KV heads: one head per work item
    # (with an even number the kernel takes two heads per item)
    "odd_hkv_b8": Workload(name="odd", dtype="bf16", num_seqs=5, num_heads=6, num_kv_heads=3, head_dim=128,
                           block_size=8, seed=62, ctx_lo=1, ctx_hi=700),
}


def _fp8_case(pa, w, ctx=None):
    case = make_decode_case(w, ctx=ctx)
    kc, vc = _quantize_on_gpu(pa, case.k_cache, K_SCALE, V_SCALE, case.v_cache)
    k_codes = quantize_pool_fp8(case.k_pool, K_SCALE)
    v_codes = quantize_pool_fp8(case.v_pool, V_SCALE)
    torch.cuda.synchronize()
    assert np.array_equal(_codes(kc), k_codes) and np.array_equal(_codes(vc), v_codes)
    return case, kc, vc, k_codes, v_codes


def _oracle(case, k_codes, v_codes, seqs=None):
    return oracle_decode(case.q, k_codes, v_codes, case.tables, case.ctx, case.w.scale, "bf16", seqs,
                         cache_dtype="fp8", k_scale=K_SCALE, v_scale=V_SCALE)


@pytest.mark.parametrize("name", sorted(SMALL))
@pytest.mark.parametrize("partition", [0, 64, 4096])
def test_fp8_decode_small_workloads(pa, name, partition):
    w = SMALL[name]
    case, kc, vc, k_codes, v_codes = _fp8_case(pa, w)
    out = pa.paged_decode_fp8(case.q_d, kc, vc, case.tables_d, case.ctx_d, case.max_ctx, w.scale, K_SCALE, V_SCALE,
                              partition_size=partition)
    torch.cuda.synchronize()
    assert_close(out, _oracle(case, k_codes, v_codes), "bf16", f"{name} P={partition}")
    assert pa.get_status() == 0


@pytest.mark.parametrize("b", [8, 16, 32])
@pytest.mark.parametrize("g", [1, 4, 8])
def test_fp8_context_edges(pa, b, g):
    """Lengths at every block, 64-token stage and partition edge."""
    edges = sorted({1, b - 1, b, b + 1, 63, 64, 65, 127, 128, 129, 2 * b + 3, 191, 256, 300})
    w = Workload(name=f"edges_b{b}_g{g}", dtype="bf16", num_seqs=len(edges), num_heads=2 * g, num_kv_heads=2,
                 head_dim=128, block_size=b, seed=70 + b + g, ctx_dist="fixed", ctx_fixed=tuple(edges))
    case, kc, vc, k_codes, v_codes = _fp8_case(pa, w)
    for partition in (64, 128):
        out = pa.paged_decode_fp8(case.q_d, kc, vc, case.tables_d, case.ctx_d, case.max_ctx, w.scale, K_SCALE,
                                  V_SCALE, partition_size=partition)
        torch.cuda.synchronize()
        assert_close(out, _oracle(case, k_codes, v_codes), "bf16", f"B={b} g={g} P={partition}")
    assert pa.get_status() == 0


@pytest.mark.parametrize("b", [8, 16])
def test_fp8_nan_codes_past_the_context_are_ignored(pa, b):
    w = SMALL["serving_g4_b8"].replace(block_size=b)
    case, kc, vc, k_codes, v_codes = _fp8_case(pa, w)
    kb, vb = kc.view(torch.uint8), vc.view(torch.uint8)
    for s in range(w.num_seqs):  # NaN codes in the unused rows of every last block
        n = int(case.ctx[s])
        if n % b:
            blk = int(case.tables[s, (n - 1) // b])
            kb[blk, :, n % b:] = 0x7F
            vb[blk, :, n % b:] = 0xFF
    out = pa.paged_decode_fp8(case.q_d, kc, vc, case.tables_d, case.ctx_d, case.max_ctx, w.scale, K_SCALE, V_SCALE,
                              partition_size=64)
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all()
    assert_close(out, _oracle(case, k_codes, v_codes), "bf16", "NaN tail")
    assert pa.get_status() == 0


def test_fp8_host_plan_equals_device_plan_bitwise(pa):
    from paged_kv_cache_216_gb300 import ops

    w = SMALL["long_g8_b32"]
    case, kc, vc, _, _ = _fp8_case(pa, w)
    p = 512
    dev = pa.paged_decode_fp8(case.q_d, kc, vc, case.tables_d, case.ctx_d, case.max_ctx, w.scale, K_SCALE, V_SCALE,
                              partition_size=p)
    plan_h = np.zeros(ops.decode_plan_bytes(w.num_seqs, case.max_ctx, p), dtype=np.uint8)
    ops.decode_plan_host(case.ctx, case.max_ctx, p, plan_h)
    host = pa.paged_decode_fp8(case.q_d, kc, vc, case.tables_d, case.ctx_d, case.max_ctx, w.scale, K_SCALE,
                               V_SCALE, partition_size=p, plan=torch.from_numpy(plan_h).cuda())
    torch.cuda.synchronize()
    assert torch.equal(dev.view(torch.int16), host.view(torch.int16))
    assert pa.get_status() == 0


def test_fp8_serving_loop_matches_oracle(pa):
    """Serving steps with E4M3 caches and a fork whose shared partly filled
    block is copied on the first append: slots, tables and stored codes
    exact, outputs within tolerance, every step."""
    from oracle.allocator import BlockAllocator as OracleAllocator
    from oracle.serving import ServingOracle
    from workloads import serving_step_tokens

    w = WORKLOADS["serving_bf16_b16"].replace(num_seqs=7, num_heads=8, num_kv_heads=2, ctx_mean=200.0, ctx_hi=700)
    steps = 6
    ctx = context_lens(w)
    parent = int(np.argmax(ctx % w.block_size != 0))
    child = (parent + 1) % w.num_seqs
    ctx[child] = ctx[parent]
    nb = pool_blocks(w, ctx, extra_steps=steps) + 1
    order = free_order(w, nb)
    k_codes = quantize_pool_fp8(random_pool(w, nb, "k"), K_SCALE)
    v_codes = quantize_pool_fp8(random_pool(w, nb, "v"), V_SCALE)
    c = pa.BlockAllocator(nb, w.block_size, order)
    o = OracleAllocator(nb, w.block_size, order)
    for s in range(w.num_seqs):
        if s != child:
            c.add(s, int(ctx[s]))
            o.add(s, int(ctx[s]))
    c.fork(parent, child)
    o.fork(parent, child)
    kc = torch.from_numpy(k_codes.copy()).cuda().view(getattr(torch, "float8_e4m3fn", torch.uint8))
    vc = torch.from_numpy(v_codes.copy()).cuda().view(getattr(torch, "float8_e4m3fn", torch.uint8))
    eng = pa.ServingEngine(kc, vc, c, np.arange(w.num_seqs), w.num_heads, w.scale, int(ctx.max()) + steps, 128,
                           kv_scales=(K_SCALE, V_SCALE))
    orc = ServingOracle(o, k_codes, v_codes, w.num_seqs, "bf16", w.scale, fp8_scales=(K_SCALE, V_SCALE))
    ncow = 0
    for step in range(steps):
        q, k, v = serving_step_tokens(w, step)
        out = eng.step(to_dev(q), to_dev(k), to_dev(v))
        slots, pairs, ref = orc.step(q, k, v, eng.width)
        ncow += len(pairs)
        torch.cuda.synchronize()
        assert np.array_equal(eng.slots_h.numpy(), slots)
        assert np.array_equal(eng.tables_h.numpy(), orc.tables(eng.width))
        assert np.array_equal(_codes(eng.k_cache), orc.k_cache)
        assert np.array_equal(_codes(eng.v_cache), orc.v_cache)
        assert_close(out, ref, "bf16", f"fp8 step {step}")
    assert ncow == 1
    assert pa.get_status() == 0


def _sub_pool_oracle(case_tables, ctx, q, k_bits, v_bits, seqs, scale):
    """Oracle output of the listed sequences from only their own blocks,
    quantized here (a full-size pool is too large to quantize on the CPU in
    a test)."""
    b = k_bits.shape[2]
    blocks = sorted({int(x) for s in seqs for x in case_tables[s, :-(-int(ctx[s]) // b)]})
    remap = {blk: i for i, blk in enumerate(blocks)}
    kq = ofp8.quantize(bf16_to_f32(k_bits[blocks]), K_SCALE)
    vq = ofp8.quantize(bf16_to_f32(v_bits[blocks]), V_SCALE)
    tables = np.zeros((len(seqs), case_tables.shape[1]), dtype=np.int32)
    for i, s in enumerate(seqs):
        n = -(-int(ctx[s]) // b)
        tables[i, :n] = [remap[int(x)] for x in case_tables[s, :n]]
    return oracle_decode(q[seqs], kq, vq, tables, ctx[seqs], scale, "bf16", cache_dtype="fp8", k_scale=K_SCALE,
                         v_scale=V_SCALE)


@pytest.mark.parametrize("name", ["long_bf16", "serving_bf16_b16"])
def test_fp8_full_size_sampled(pa, name):
    """A full-size workload with E4M3 caches: sampled sequences (the
    longest included) against the oracle over their own quantized blocks."""
    w = WORKLOADS[name]
    case = make_decode_case(w)
    kc, vc = _quantize_on_gpu(pa, case.k_cache, K_SCALE, V_SCALE, case.v_cache)
    del case.k_cache, case.v_cache
    torch.cuda.empty_cache()
    out = pa.paged_decode_fp8(case.q_d, kc, vc, case.tables_d, case.ctx_d, case.max_ctx, w.scale, K_SCALE, V_SCALE,
                              partition_size=w.partition_size)
    torch.cuda.synchronize()
    rng = np.random.default_rng(3)
    seqs = sorted(set(rng.choice(w.num_seqs, 2, replace=False).tolist()) | {int(np.argmax(case.ctx))})
    ref = _sub_pool_oracle(case.tables, case.ctx, case.q, case.k_pool, case.v_pool, seqs, w.scale)
    assert_close(out[seqs], ref, "bf16", f"{name} fp8 sampled")
    assert pa.get_status() == 0
