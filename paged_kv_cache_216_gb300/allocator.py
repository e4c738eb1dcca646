"""Python handle on the C++ block allocator (pa_alloc_* / pa_seq_*)."""

from __future__ import annotations

import ctypes

import numpy as np

from . import _lib as _libmod
from ._lib import check, lib


def _np_ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


class BlockAllocator:
    """Free list + ref-counted sharing + copy-on-write over ``num_blocks``
    blocks of ``block_size`` tokens.  ``free_order`` (a permutation) is the
    hand-out order of a fresh pool; None means ascending."""

    def __init__(self, num_blocks: int, block_size: int, free_order=None):
        self._h = ctypes.c_void_p(0)
        self.num_blocks = num_blocks
        self.block_size = block_size
        order = None
        if free_order is not None:
            order = np.ascontiguousarray(free_order, dtype=np.int32)
            if order.shape != (num_blocks,):
                raise ValueError("free_order must have num_blocks entries")
        check(lib().pa_alloc_create(num_blocks, block_size, _np_ptr(order) if order is not None else None,
                                    ctypes.byref(self._h)))
        self._keep = order

    def __del__(self):
        h = getattr(self, "_h", None)
        try:
            if h and h.value and _libmod._lib is not None:
                _libmod._lib.pa_alloc_destroy(h)
                self._h = ctypes.c_void_p(0)
        except Exception:  # interpreter shutdown: the process frees everything anyway
            pass

    def num_free(self) -> int:
        return check(lib().pa_alloc_num_free(self._h))

    def add(self, seq_id: int, num_tokens: int) -> None:
        check(lib().pa_seq_add(self._h, seq_id, num_tokens))

    def fork(self, parent_id: int, child_id: int) -> None:
        check(lib().pa_seq_fork(self._h, parent_id, child_id))

    def append_slot(self, seq_id: int):
        slot = ctypes.c_int64()
        src = ctypes.c_int32()
        dst = ctypes.c_int32()
        check(lib().pa_seq_append_slot(self._h, seq_id, ctypes.byref(slot), ctypes.byref(src), ctypes.byref(dst)))
        return slot.value, src.value, dst.value

    def free(self, seq_id: int) -> None:
        check(lib().pa_seq_free(self._h, seq_id))

    def num_tokens(self, seq_id: int) -> int:
        return check(lib().pa_seq_num_tokens(self._h, seq_id))

    def refcount(self, block_id: int) -> int:
        return check(lib().pa_block_refcount(self._h, block_id))

    def block_table(self, seq_id: int) -> list:
        n = ctypes.c_int(0)
        rc = lib().pa_seq_block_table(self._h, seq_id, None, 0, ctypes.byref(n))
        if rc < 0 and n.value == 0:
            check(rc)
        out = np.empty(max(n.value, 1), dtype=np.int32)
        check(lib().pa_seq_block_table(self._h, seq_id, _np_ptr(out), out.shape[0], ctypes.byref(n)))
        return out[: n.value].tolist()

    def append_slots(self, seq_ids: np.ndarray, slot_mapping: np.ndarray, cow_pairs: np.ndarray,
                     block_tables: np.ndarray | None = None, context_lens: np.ndarray | None = None) -> int:
        """Batched append of one token to each of ``seq_ids`` (int64).
        Writes ``slot_mapping`` (int64 [n]) and ``cow_pairs`` (int32 [n, 2]);
        updates ``block_tables`` (int32 [n, width]) rows in place and
        ``context_lens`` (int32 [n]) when given.  Returns the number of
        copy-on-write pairs."""
        n = seq_ids.shape[0]
        nc = ctypes.c_int(0)
        width = block_tables.shape[1] if block_tables is not None else 0
        check(lib().pa_seqs_append_slots(self._h, _np_ptr(seq_ids), n, _np_ptr(slot_mapping), _np_ptr(cow_pairs),
                                         ctypes.byref(nc),
                                         _np_ptr(block_tables) if block_tables is not None else None, width,
                                         _np_ptr(context_lens) if context_lens is not None else None))
        return nc.value

    def block_tables(self, seq_ids: np.ndarray, block_tables: np.ndarray,
                     context_lens: np.ndarray | None = None) -> None:
        """Fill ``block_tables`` (int32 [n, width], -1 padded) and
        ``context_lens`` for ``seq_ids`` (int64)."""
        check(lib().pa_seqs_block_tables(self._h, _np_ptr(seq_ids), seq_ids.shape[0], _np_ptr(block_tables),
                                         block_tables.shape[1],
                                         _np_ptr(context_lens) if context_lens is not None else None))

