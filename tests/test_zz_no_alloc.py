"""pa_decode_static_workspace: paged decode for callers that cannot allocate.

Some callers cannot call cudaMalloc to give pa_decode its split-K workspace:
their device memory is reserved up front by another allocator, or their loop
must not make calls that may synchronize the device.  This entry point keeps
that scratch in a fixed array inside the library instead.  The test calls it
through the C ABI twice in a row, with different queries, on a batch whose
contexts span several partitions (so the partials and the merge really go
through the array), and checks each result element by element against the
CPU oracle within the bf16 tolerance of the other decode tests, and bit for
bit against pa_decode with a caller workspace (the same kernels and
partition size).  It lives in its own file so that pytest collects it last.
"""

import pytest
import torch

from tests._cases import assert_close, make_decode_case, to_dev
from tests._lib_fixture import ensure_built
from oracle.attention import paged_decode as oracle_decode
from workloads import Workload, normal

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    ensure_built()
    import paged_kv_cache_216_gb300 as pa

    return pa


def test_static_workspace_matches_oracle_and_pa_decode_on_two_calls(pa):
    w = Workload(name="noalloc", dtype="bf16", num_seqs=16, num_heads=32, num_kv_heads=8, head_dim=128,
                 block_size=16, seed=61, ctx_lo=300, ctx_hi=3000)
    case = make_decode_case(w)
    p = pa.decode_partition_size(w.num_seqs, w.num_kv_heads, case.max_ctx, 0)
    assert -(-case.max_ctx // p) > 1, "the batch must split, so that partials go through the array"
    need = pa.decode_workspace_bytes(w.num_seqs, w.num_heads, w.head_dim, case.max_ctx, p)
    assert need <= pa._lib.PA_STATIC_WORKSPACE_BYTES
    q2 = normal((w.num_seqs, w.num_heads, w.head_dim), 1.0, "bf16", w.seed, 99)
    out = torch.empty_like(case.q_d)
    for q_h in (case.q, q2):  # two calls in a row share the array
        q = to_dev(q_h)
        ref = oracle_decode(q_h, case.k_pool, case.v_pool, case.tables, case.ctx, w.scale, w.dtype)
        mine = pa.paged_decode(q, case.k_cache, case.v_cache, case.tables_d, case.ctx_d, case.max_ctx, w.scale)
        out.fill_(float("nan"))
        pa.paged_decode_static_workspace(q, case.k_cache, case.v_cache, case.tables_d, case.ctx_d, case.max_ctx,
                                         w.scale, out)
        torch.cuda.synchronize()
        assert_close(out, ref, "bf16", "static-workspace decode vs oracle")
        assert torch.equal(out, mine), "static-workspace decode differs from pa_decode"
    assert pa.get_status() == 0


def test_static_workspace_rejects_sizes_beyond_the_array(pa):
    L = pa.lib()
    # 8 sequences of up to 131072 tokens, 64 heads, 512-token partitions:
    # about 68 MB of partials.  The size check comes before any pointer is
    # looked at, so every pointer is null: were it ever skipped, the call
    # would stop at the null-pointer check instead of launching.
    rc = L.pa_decode_static_workspace(None, None, None, None, 4096, None, 131072, 0.1, None, 8, 64, 8, 128, 32,
                                      30000, 512, 1, None)
    assert rc == -1
    assert b"fixed" in L.pa_last_error()
