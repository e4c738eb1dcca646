"""KV append and block copy on the GPU: bit-exact against the oracle over the
whole pool (untouched slots must stay unchanged)."""

import numpy as np
import pytest
import torch

from oracle.cache import cache_append as oracle_append
from oracle.cache import copy_blocks as oracle_copy
from tests._cases import to_bits, to_dev
from tests._lib_fixture import ensure_built
from workloads import Workload, normal, random_pool

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    ensure_built()
    import paged_kv_cache_216_gb300 as pa

    return pa


@pytest.mark.parametrize("dtype,d,b,hkv,t", [
    ("bf16", 128, 16, 8, 256), ("bf16", 128, 8, 8, 256), ("bf16", 128, 32, 8, 256),
    ("bf16", 64, 16, 4, 37), ("f32", 64, 16, 4, 57), ("f32", 128, 8, 2, 33), ("bf16", 128, 16, 32, 1),
])
def test_append_bit_exact(pa, dtype, d, b, hkv, t):
    w = Workload(name="t", dtype=dtype, num_seqs=t, num_heads=hkv, num_kv_heads=hkv, head_dim=d, block_size=b,
                 seed=40 + d + b)
    nb = (t // b) + 7
    kc = random_pool(w, nb, "k")
    vc = random_pool(w, nb, "v")
    k = normal((t, hkv, d), 1.0, dtype, w.seed, 70)
    v = normal((t, hkv, d), 1.0, dtype, w.seed, 71)
    rng = np.random.default_rng(w.seed)
    slots = rng.permutation(nb * b)[:t].astype(np.int64)
    slots[rng.random(t) < 0.1] = -1  # skipped tokens
    kd, vd = to_dev(kc), to_dev(vc)
    pa.cache_append(to_dev(k), to_dev(v), to_dev(slots), kd, vd)
    want_k, want_v = oracle_append(kc, vc, k, v, slots)
    assert np.array_equal(to_bits(kd), want_k)
    assert np.array_equal(to_bits(vd), want_v)
    assert pa.get_status() == 0


def test_append_out_of_range_slot_is_skipped_and_flagged(pa):
    w = Workload(name="t", dtype="bf16", num_seqs=4, num_heads=2, num_kv_heads=2, head_dim=128, block_size=16,
                 seed=5)
    kc = random_pool(w, 3, "k")
    vc = random_pool(w, 3, "v")
    k = normal((3, 2, 128), 1.0, "bf16", 5, 72)
    slots = np.array([5, 48, 47], dtype=np.int64)  # 48 = 3 blocks * 16: out of range
    kd, vd = to_dev(kc), to_dev(vc)
    pa.get_status()
    pa.cache_append(to_dev(k), to_dev(k), to_dev(slots), kd, vd)
    assert pa.get_status() & pa._lib.PA_STATUS_BAD_SLOT
    keep = slots.copy()
    keep[1] = -1
    want_k, _ = oracle_append(kc, vc, k, k, keep)
    assert np.array_equal(to_bits(kd), want_k)


@pytest.mark.parametrize("dtype,d,b,hkv", [("bf16", 128, 16, 8), ("f32", 64, 32, 4), ("bf16", 64, 8, 2)])
def test_copy_blocks_bit_exact(pa, dtype, d, b, hkv):
    w = Workload(name="t", dtype=dtype, num_seqs=1, num_heads=hkv, num_kv_heads=hkv, head_dim=d, block_size=b,
                 seed=9)
    nb = 40
    kc = random_pool(w, nb, "k")
    vc = random_pool(w, nb, "v")
    rng = np.random.default_rng(9)
    perm = rng.permutation(nb)
    pairs = np.stack([perm[:12], perm[12:24]], axis=1).astype(np.int32)  # dsts distinct, never a src
    kd, vd = to_dev(kc), to_dev(vc)
    pa.copy_blocks(kd, vd, to_dev(pairs))
    oracle_copy(kc, vc, [tuple(p) for p in pairs])
    assert np.array_equal(to_bits(kd), kc) and np.array_equal(to_bits(vd), vc)
    assert pa.get_status() == 0


def test_copy_blocks_bad_id_is_skipped_and_flagged(pa):
    w = Workload(name="t", dtype="bf16", num_seqs=1, num_heads=2, num_kv_heads=2, head_dim=128, block_size=16,
                 seed=10)
    kc = random_pool(w, 6, "k")
    kd, vd = to_dev(kc), to_dev(kc)
    pa.get_status()
    pa.copy_blocks(kd, vd, torch.tensor([[1, 2], [0, 9]], dtype=torch.int32, device="cuda"))
    assert pa.get_status() & pa._lib.PA_STATUS_BAD_BLOCK
    oracle_copy(kc, kc.copy(), [(1, 2)])
    assert np.array_equal(to_bits(kd), kc)
