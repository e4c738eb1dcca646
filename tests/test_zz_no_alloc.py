"""pa_decode_static_workspace: paged decode for callers that cannot allocate.

Some callers cannot call cudaMalloc to give pa_decode its split-K workspace:
their device memory is reserved up front by another allocator, or their loop
must not make calls that may synchronize the device.  This entry point keeps
that scratch in a fixed array inside the library instead.  The test calls it
through the C ABI twice in a row, with different queries, and checks each
result against pa_decode with a caller workspace, within the bf16 tolerance
the other decode tests use.  It lives in its own file so that pytest collects
it last.
"""

import numpy as np
import pytest
import torch

from tests._cases import as_f64, make_decode_case, to_dev
from tests._lib_fixture import ensure_built
from workloads import Workload, normal

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    ensure_built()
    import paged_kv_cache_216_gb300 as pa

    return pa


def _within_tolerance(got, ref):
    g, r = as_f64(got), as_f64(ref)
    err = np.abs(g - r)
    assert np.all(err <= 2e-2 + 1e-2 * np.abs(r)), f"max abs difference {err.max():.3g}"


def test_static_workspace_matches_pa_decode_on_two_calls(pa):
    w = Workload(name="noalloc", dtype="bf16", num_seqs=16, num_heads=32, num_kv_heads=8, head_dim=128,
                 block_size=16, seed=61, ctx_lo=300, ctx_hi=3000)
    case = make_decode_case(w)
    p = pa.decode_partition_size(w.num_seqs, w.num_kv_heads, case.max_ctx, 0)
    need = pa.decode_workspace_bytes(w.num_seqs, w.num_heads, w.head_dim, case.max_ctx, p)
    assert 0 < need <= pa._lib.PA_STATIC_WORKSPACE_BYTES  # the split path really uses the array
    queries = [case.q_d, to_dev(normal((w.num_seqs, w.num_heads, w.head_dim), 1.0, "bf16", w.seed, 99))]
    out = torch.empty_like(case.q_d)
    for q in queries:  # two calls in a row share the array
        ref = pa.paged_decode(q, case.k_cache, case.v_cache, case.tables_d, case.ctx_d, case.max_ctx, w.scale)
        pa.paged_decode_static_workspace(q, case.k_cache, case.v_cache, case.tables_d, case.ctx_d, case.max_ctx,
                                         w.scale, out)
        torch.cuda.synchronize()
        _within_tolerance(out, ref)
    assert pa.get_status() == 0


def test_static_workspace_rejects_sizes_beyond_the_array(pa):
    import ctypes

    fake = ctypes.c_void_p(0x100000)
    L = pa.lib()
    # 8 sequences of up to 131072 tokens, 64 heads, 512-token partitions: about 68 MB of partials
    rc = L.pa_decode_static_workspace(fake, fake, fake, fake, 4096, fake, 131072, 0.1, fake, 8, 64, 8, 128, 32,
                                      30000, 512, 1, None)
    assert rc == -1
    assert b"fixed" in L.pa_last_error()
