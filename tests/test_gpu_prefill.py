"""Prefill on the GPU against the oracle: the appended cache bit for bit,
the causal attention of every new token within the bf16 tolerance
(|gpu - ref| <= 2e-2 + 1e-2 |ref|)."""

import numpy as np
import pytest
import torch

from oracle.attention import decode_one, gather_sequence, to_f64
from oracle.cache import cache_append
from oracle.prefill import prefill as oracle_prefill
from tests._cases import assert_close, to_bits, to_dev
from tests._lib_fixture import ensure_built
from workloads import normal

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    ensure_built()
    import paged_kv_cache_216_gb300 as pa

    return pa


def _batch(seed, prev, new, H, Hkv, D, B):
    """Seeded bf16 batch: sequence s has prev[s] cached tokens and new[s]
    new ones; tables over a shuffled pool; slots of the new tokens."""
    rng = np.random.default_rng(seed)
    S = len(prev)
    ctx = np.array([p + n for p, n in zip(prev, new)], dtype=np.int32)
    need = sum(-(-int(c) // B) for c in ctx)
    N = need + 7
    perm = rng.permutation(N)
    width = max(-(-int(c) // B) for c in ctx)
    tables = np.full((S, width), -1, dtype=np.int32)
    it = iter(perm.tolist())
    for s in range(S):
        nb = -(-int(ctx[s]) // B)
        tables[s, :nb] = [next(it) for _ in range(nb)]
    qs = np.concatenate([[0], np.cumsum(new)]).astype(np.int32)
    T = int(qs[-1])
    slots = np.empty(T, dtype=np.int64)
    for s in range(S):
        for j in range(new[s]):
            pos = prev[s] + j
            slots[qs[s] + j] = tables[s, pos // B] * B + pos % B
    kc = normal((N, Hkv, B, D), 1.0, "bf16", seed, 21)
    vc = normal((N, Hkv, B, D), 1.0, "bf16", seed, 22)
    q = normal((T, H, D), 1.0, "bf16", seed, 23)
    k = normal((T, Hkv, D), 1.0, "bf16", seed, 24)
    v = normal((T, Hkv, D), 1.0, "bf16", seed, 25)
    return dict(q=q, k=k, v=v, slots=slots, qs=qs, ctx=ctx, tables=tables, kc=kc, vc=vc, scale=1.0 / np.sqrt(D))


def _run(pa, b, max_query_len=None):
    kc, vc = to_dev(b["kc"]), to_dev(b["vc"])
    out = pa.prefill(to_dev(b["q"]), to_dev(b["k"]), to_dev(b["v"]), torch.from_numpy(b["slots"]).cuda(),
                     torch.from_numpy(b["qs"]).cuda(), torch.from_numpy(b["ctx"]).cuda(),
                     torch.from_numpy(b["tables"]).cuda(),
                     int(np.diff(b["qs"]).max()) if max_query_len is None else max_query_len, int(b["ctx"].max()),
                     b["scale"], kc, vc)
    torch.cuda.synchronize()
    return out, kc, vc


CASES = {
    # (prev cached tokens, new tokens, H, Hkv, D, B)
    "g4_d128_b16": ([0, 5, 100, 1000], [1, 37, 64, 130], 16, 4, 128, 16),
    "g1_d64_b32": ([0, 33], [200, 65], 4, 4, 64, 32),
    "g8_d128_b8": ([7, 0, 300], [9, 17, 1], 16, 2, 128, 8),
    "g2_long_prompt": ([2000], [700], 8, 4, 128, 16),
    "g4_fresh_prompts": ([0, 0, 0], [1, 2, 63], 8, 2, 128, 32),
    # one query head per KV head on the tcgen05 path (query boxes of 128 tokens x 1 head)
    "g1_d128_b32": ([0, 100], [150, 33], 4, 4, 128, 32),
    # a sequence with no new tokens between two that have some
    "g4_no_new_tokens": ([12, 40, 0], [3, 0, 70], 8, 2, 128, 16),
    # head_dim 64 with grouped heads: ragged prompts, full and partial tiles, 8-token blocks
    "g4_d64_b8": ([0, 77, 300], [70, 33, 129], 16, 4, 64, 8),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_prefill_matches_oracle(pa, name):
    prev, new, H, Hkv, D, B = CASES[name]
    b = _batch(sum(new) + len(prev), prev, new, H, Hkv, D, B)
    out, kc, vc = _run(pa, b)
    kc_o, vc_o, ref = oracle_prefill(b["q"], b["k"], b["v"], b["slots"], b["qs"], b["ctx"], b["tables"], b["kc"],
                                     b["vc"], b["scale"], "bf16")
    assert np.array_equal(to_bits(kc), kc_o) and np.array_equal(to_bits(vc), vc_o)
    assert_close(out, ref, "bf16", name)
    assert pa.get_status() == 0


def _poison_past_context(b, B):
    """Rows of each sequence's last block past its context hold NaN (keys)
    and +Inf (values), as rows never written may: masked keys must not let
    them into any output."""
    for s, ctx in enumerate(b["ctx"]):
        if ctx % B:
            blk = b["tables"][s, (int(ctx) - 1) // B]
            b["kc"][blk, :, ctx % B:, :] = 0x7FC0  # bf16 NaN
            b["vc"][blk, :, ctx % B:, :] = 0x7F80  # bf16 +Inf


@pytest.mark.parametrize("name", ["g4_d128_b16", "g8_d128_b8", "g1_d64_b32", "g4_d64_b8", "g2_long_prompt"])
def test_prefill_ignores_non_finite_rows_past_the_context(pa, name):
    prev, new, H, Hkv, D, B = CASES[name]
    b = _batch(sum(new) + 3 * len(prev), prev, new, H, Hkv, D, B)
    _poison_past_context(b, B)
    out, kc, vc = _run(pa, b)
    kc_o, vc_o, ref = oracle_prefill(b["q"], b["k"], b["v"], b["slots"], b["qs"], b["ctx"], b["tables"], b["kc"],
                                     b["vc"], b["scale"], "bf16")
    assert np.array_equal(to_bits(kc), kc_o) and np.array_equal(to_bits(vc), vc_o)
    assert np.isfinite(out.float().cpu().numpy()).all()
    assert_close(out, ref, "bf16", name + " with non-finite rows past the context")
    assert pa.get_status() == 0


def test_prefill_of_one_token_per_sequence_is_decode(pa):
    """n_s = 1 everywhere: the rows equal paged decode over the appended
    cache (both within tolerance of the same oracle values)."""
    prev, new = [10, 77, 0, 300], [1, 1, 1, 1]
    b = _batch(91, prev, new, 16, 4, 128, 16)
    out, kc, vc = _run(pa, b)
    dec = pa.paged_decode(to_dev(b["q"]), kc, vc, torch.from_numpy(b["tables"]).cuda(),
                          torch.from_numpy(b["ctx"]).cuda(), int(b["ctx"].max()), b["scale"])
    torch.cuda.synchronize()
    _, _, ref = oracle_prefill(b["q"], b["k"], b["v"], b["slots"], b["qs"], b["ctx"], b["tables"], b["kc"], b["vc"],
                               b["scale"], "bf16")
    assert_close(out, ref, "bf16", "prefill")
    assert_close(dec, ref, "bf16", "decode")


def test_prefill_larger_max_query_len_and_bad_lengths(pa):
    """A host bound above the longest prompt changes nothing; a sequence whose
    lengths are inconsistent (more new tokens than context) is skipped with
    PA_STATUS_BAD_CONTEXT while the others are computed."""
    prev, new, H, Hkv, D, B = CASES["g4_d128_b16"]
    b = _batch(7, prev, new, H, Hkv, D, B)
    out, _, _ = _run(pa, b, max_query_len=512)
    _, _, ref = oracle_prefill(b["q"], b["k"], b["v"], b["slots"], b["qs"], b["ctx"], b["tables"], b["kc"], b["vc"],
                               b["scale"], "bf16")
    assert_close(out, ref, "bf16", "max_query_len 512")
    assert pa.get_status() == 0
    bad = dict(b)
    bad["ctx"] = b["ctx"].copy()
    bad["ctx"][1] = 10  # 37 new tokens cannot fit in a context of 10
    out2, _, _ = _run(pa, bad)
    assert pa.get_status() == pa._lib.PA_STATUS_BAD_CONTEXT
    rows = np.r_[b["qs"][0]:b["qs"][1], b["qs"][2]:b["qs"][4]]
    assert_close(out2[rows], ref[rows], "bf16", "other sequences")


def _check_sampled_tokens(b, out, kc, prev, tokens, H, Hkv):
    """Tokens tokens[s] (indices among sequence s's new tokens) of every
    sequence against the oracle's per-token definition, every KV head."""
    kc_o, vc_o = cache_append(b["kc"], b["vc"], b["k"], b["v"], b["slots"])
    assert np.array_equal(to_bits(kc), kc_o)
    g = H // Hkv
    for s, idx in enumerate(tokens):
        for i in idx:
            row = int(b["qs"][s]) + i
            p = prev[s] + i
            for kv in range(Hkv):
                kr = to_f64(gather_sequence(kc_o, b["tables"][s], p + 1, kv), "bf16")
                vr = to_f64(gather_sequence(vc_o, b["tables"][s], p + 1, kv), "bf16")
                ref = decode_one(to_f64(b["q"][row, kv * g:(kv + 1) * g], "bf16"), kr, vr, b["scale"])
                assert_close(out[row, kv * g:(kv + 1) * g], ref, "bf16", f"s{s} i{i} kv{kv}")


def test_prefill_bench_shape_sampled(pa):
    """The benchmark's prefill batch (8 sequences, 512 cached + 512 new
    tokens, 32/8 heads): sampled tokens (first, last, random) of every
    sequence against the oracle's per-token definition."""
    S, prev_n, new_n, H, Hkv, D, B = 8, 512, 512, 32, 8, 128, 16
    b = _batch(5, [prev_n] * S, [new_n] * S, H, Hkv, D, B)
    out, kc, vc = _run(pa, b)
    rng = np.random.default_rng(6)
    tokens = [sorted({0, new_n - 1, int(rng.integers(new_n))}) for _ in range(S)]
    _check_sampled_tokens(b, out, kc, [prev_n] * S, tokens, H, Hkv)
    assert pa.get_status() == 0


# Ragged batches of more work items (sequence, KV head, pair of 128-row
# tiles) than CTAs, not a multiple of them: with these lengths the kernel
# takes one snake over all CTAs for the first (its busiest CTA would get 32
# chunk units against 52 in the count-aware order) and the count-aware
# order for the second (44 against 52).
RAGGED = {
    "plain_order": ([1688, 112, 1352, 2027, 333], [113, 74, 10, 613, 31]),
    "count_aware_order": ([0, 300, 1200, 50, 2000, 700], [900, 64, 513, 1024, 200, 777]),
}


@pytest.mark.parametrize("name", sorted(RAGGED))
def test_prefill_ragged_many_items_sampled(pa, name):
    """One token of every pair of tiles of every sequence (its first and a
    random one), plus each sequence's last, so that every work item is
    checked against the oracle."""
    prev, new = RAGGED[name]
    H, Hkv, D, B = 32, 8, 128, 16
    b = _batch(7, prev, new, H, Hkv, D, B)
    out, kc, vc = _run(pa, b)
    rng = np.random.default_rng(8)
    per_pair = 256 // (H // Hkv)  # new tokens per pair of tiles
    tokens = []
    for n in new:
        idx = {n - 1}
        for t0 in range(0, n, per_pair):
            idx |= {t0, int(rng.integers(t0, min(n, t0 + per_pair)))}
        tokens.append(sorted(idx))
    _check_sampled_tokens(b, out, kc, prev, tokens, H, Hkv)
    assert pa.get_status() == 0


@pytest.mark.parametrize("cap", [7, 50])
def test_prefill_over_several_launches(pa, cap):
    """A batch attended by several kernel launches, each over a contiguous
    range of the work items (the path of batches with more items than one
    launch lists), here forced with a small bound on the items of a launch:
    the same result as one launch, and the oracle's."""
    prev, new, H, Hkv, D, B = CASES["g4_d128_b16"]  # 48 work items
    b = _batch(21, prev, new, H, Hkv, D, B)
    one, _, _ = _run(pa, b)
    assert pa.lib().pa_prefill_test_items_per_launch(cap) == 0
    try:
        out, kc, vc = _run(pa, b)
    finally:
        assert pa.lib().pa_prefill_test_items_per_launch(0) == 0
    kc_o, vc_o, ref = oracle_prefill(b["q"], b["k"], b["v"], b["slots"], b["qs"], b["ctx"], b["tables"], b["kc"],
                                     b["vc"], b["scale"], "bf16")
    assert np.array_equal(to_bits(kc), kc_o) and np.array_equal(to_bits(vc), vc_o)
    assert_close(out, ref, "bf16", f"{cap} items per launch")
    assert torch.equal(out, one)
    assert pa.get_status() == 0
    assert pa.lib().pa_prefill_test_items_per_launch(-1) == -1


@pytest.mark.parametrize("name", ["g4_d128_b16", "g4_d64_b8"])
def test_prefill_output_16_byte_aligned(pa, name):
    """Output rows written into a view 16 bytes past a 32-byte boundary: full
    tiles go out by TMA store from their staging buffer, a sequence's last
    (partial) tile by 16-byte stores of each row; the elements on either side
    of the view stay untouched."""
    prev, new, H, Hkv, D, B = CASES[name]
    b = _batch(sum(new) + 5 * len(prev), prev, new, H, Hkv, D, B)
    T = int(b["qs"][-1])
    n = T * H * D
    sentinel = -7.0
    base = torch.full((8 + n + 8,), sentinel, dtype=torch.bfloat16, device="cuda")
    out = base[8:8 + n].view(T, H, D)
    assert out.data_ptr() % 32 == 16
    kc, vc = to_dev(b["kc"]), to_dev(b["vc"])
    got = pa.prefill(to_dev(b["q"]), to_dev(b["k"]), to_dev(b["v"]), torch.from_numpy(b["slots"]).cuda(),
                     torch.from_numpy(b["qs"]).cuda(), torch.from_numpy(b["ctx"]).cuda(),
                     torch.from_numpy(b["tables"]).cuda(), int(np.diff(b["qs"]).max()), int(b["ctx"].max()),
                     b["scale"], kc, vc, out=out)
    torch.cuda.synchronize()
    assert got.data_ptr() == out.data_ptr()
    _, _, ref = oracle_prefill(b["q"], b["k"], b["v"], b["slots"], b["qs"], b["ctx"], b["tables"], b["kc"], b["vc"],
                               b["scale"], "bf16")
    assert_close(out, ref, "bf16", name + " (16-byte aligned output)")
    assert bool((base[:8] == sentinel).all()) and bool((base[8 + n:] == sentinel).all())
    assert pa.get_status() == 0
