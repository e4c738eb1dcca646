"""The decode kernel's bounded waits, made to run out on purpose.

Every pipeline wait of the bf16 decode kernel gives up after a time limit,
raises PA_STATUS_TIMEOUT and winds the CTA down (the defensive checks that
"PagedAttention Kernel：大模型推理优化的显存管理革新", section 5.1, asks
for).  pa_decode_test_withhold sets a 1 ms limit and has every CTA's copy
warp withhold one chunk: nothing is ever copied for it and its barrier is
never armed, so the wait for it runs out.  No copy is in flight for the
withheld chunk and no wait is unbounded, so nothing can fault or hang.  The
tests check that the call comes back in milliseconds with the time-out bit
set, and that a normal decode right after matches the oracle.
"""

import time

import pytest
import torch

from tests._cases import assert_close, make_decode_case
from tests._lib_fixture import ensure_built
from workloads import Workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    ensure_built()
    import paged_kv_cache_216_gb300 as pa

    return pa


@pytest.fixture(scope="module")
def case(pa):
    w = Workload(name="timeout", dtype="bf16", num_seqs=8, num_heads=32, num_kv_heads=8, head_dim=128,
                 block_size=16, seed=71, ctx_lo=200, ctx_hi=1500)
    return make_decode_case(w)


def _withhold(pa, case, out, withheld_chunk, wait_limit_us):
    from paged_kv_cache_216_gb300.ops import _ptr, _stream

    w = case.w
    p = pa.decode_partition_size(w.num_seqs, w.num_kv_heads, case.max_ctx, 0)
    ws = pa.decode_workspace(w.num_seqs, w.num_heads, w.num_kv_heads, w.head_dim, case.max_ctx, p)
    n, hkv, b, d = case.k_cache.shape
    rc = pa.lib().pa_decode_test_withhold(
        _ptr(case.q_d), _ptr(case.k_cache), _ptr(case.v_cache), _ptr(case.tables_d), case.tables_d.shape[1],
        _ptr(case.ctx_d), case.max_ctx, w.scale, _ptr(out), w.num_seqs, w.num_heads, hkv, d, b, n, p, _ptr(ws),
        ws.numel(), withheld_chunk, wait_limit_us, _stream())
    return rc, ws


@pytest.mark.parametrize("withheld_chunk", [0, 1, 3])
def test_withheld_chunk_times_out_and_the_context_stays_usable(pa, case, withheld_chunk):
    from paged_kv_cache_216_gb300._lib import PA_STATUS_TIMEOUT

    assert pa.get_status() == 0
    out = torch.empty_like(case.q_d)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    rc, ws = _withhold(pa, case, out, withheld_chunk, 1000)
    assert rc == 0, pa.lib().pa_last_error()
    status = pa.get_status()  # synchronizes the stream
    elapsed = time.perf_counter() - t0
    assert status & PA_STATUS_TIMEOUT, f"status {status:#x}"
    assert elapsed < 1.0, f"a 1 ms wait limit took {elapsed:.3f} s to come back"
    del ws
    # the context is intact: a normal decode right after matches the oracle
    got = pa.paged_decode(case.q_d, case.k_cache, case.v_cache, case.tables_d, case.ctx_d, case.max_ctx,
                          case.w.scale)
    torch.cuda.synchronize()
    assert_close(got, case.oracle(), "bf16", "decode after a timed-out call")
    assert pa.get_status() == 0


def test_withhold_hook_refuses_bad_limits(pa, case):
    out = torch.empty_like(case.q_d)
    rc, _ = _withhold(pa, case, out, 0, 0)
    assert rc == -1 and b"wait_limit_us" in pa.lib().pa_last_error()
    rc, _ = _withhold(pa, case, out, -1, 1000)
    assert rc == -1 and b"withheld_chunk" in pa.lib().pa_last_error()
