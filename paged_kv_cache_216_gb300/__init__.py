"""Paged KV cache decode for GB300 (sm_103a): KV append, paged decode
attention with split-K and log-sum-exp merge, copy-on-write block copy, and
a host block allocator, behind the C ABI of ``include/pa.h`` (libpa.so).

Build the library with :func:`paged_kv_cache_216_gb300.build.build`.
"""

from ._lib import PAError, OutOfBlocks, lib  # noqa: F401
from .allocator import BlockAllocator  # noqa: F401
from .ops import (  # noqa: F401
    cache_append,
    cache_append_fp8,
    copy_blocks,
    decode_partition_size,
    decode_workspace,
    decode_workspace_bytes,
    get_status,
    paged_decode,
    paged_decode_fp8,
    paged_decode_shared_prefix,
    paged_decode_static_workspace,
    prefill,
)
from .serving import ServingEngine  # noqa: F401
