"""The prefill kernel's bounded waits, made to run out on purpose.

Every pipeline wait of the tcgen05 prefill kernel gives up after 2 s, raises
PA_STATUS_TIMEOUT, lets its copies and products in flight finish and exits
(the defensive checks that "PagedAttention Kernel：大模型推理优化的显存管理革新",
section 5.1, asks for).  pa_prefill_test_withhold has the key producer of
every CTA skip one of its chunks: nothing is ever copied for it and its
barrier is never armed, so the MMA thread's wait for it runs out, the abort
flag stops the other roles, and the copies already issued are waited for
(the withheld one within the same limit).  No wait is unbounded and no copy
is in flight for the withheld chunk, so nothing can fault or hang.  The test
checks that the call comes back with the time-out bit set and that a normal
prefill right after matches the oracle.
"""

import time

import numpy as np
import pytest

from oracle.prefill import prefill as oracle_prefill
from tests._cases import assert_close, to_bits
from tests.test_gpu_prefill import CASES, _batch, _run

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    from tests._lib_fixture import ensure_built

    ensure_built()
    import paged_kv_cache_216_gb300 as pa

    return pa


def test_prefill_withheld_chunk_times_out_and_the_context_stays_usable(pa):
    from paged_kv_cache_216_gb300._lib import PA_STATUS_TIMEOUT

    prev, new, H, Hkv, D, B = CASES["g4_d128_b16"]
    assert pa.get_status() == 0
    assert pa.lib().pa_prefill_test_withhold(1) == 0
    try:
        b = _batch(91, prev, new, H, Hkv, D, B)
        t0 = time.perf_counter()
        _run(pa, b)
        status = pa.get_status()
        elapsed = time.perf_counter() - t0
    finally:
        assert pa.lib().pa_prefill_test_withhold(-1) == 0
    assert status & PA_STATUS_TIMEOUT, f"status {status:#x}"
    assert elapsed < 30.0, f"waits of 2 s took {elapsed:.1f} s to wind down"
    # the context is intact: a normal prefill right after matches the oracle
    b = _batch(92, prev, new, H, Hkv, D, B)
    out, kc, vc = _run(pa, b)
    kc_o, vc_o, ref = oracle_prefill(b["q"], b["k"], b["v"], b["slots"], b["qs"], b["ctx"], b["tables"], b["kc"],
                                     b["vc"], b["scale"], "bf16")
    assert np.array_equal(to_bits(kc), kc_o) and np.array_equal(to_bits(vc), vc_o)
    assert_close(out, ref, "bf16", "prefill after a timed-out call")
    assert pa.get_status() == 0


def test_prefill_withhold_hook_refuses_below_minus_one(pa):
    assert pa.lib().pa_prefill_test_withhold(-2) == -1
    assert b"chunk" in pa.lib().pa_last_error()
