"""ctypes binding of libpa.so (include/pa.h).

Argument marshalling only: torch tensors are turned into device pointers and
sizes, the current CUDA stream is passed along, and a non-zero return code is
raised as :class:`PAError`.  Every step of the computation runs in the
library's kernels (or its C++ allocator); there is no fallback.
"""

from __future__ import annotations

import ctypes
import os

from .build import LIB

PA_F32 = 0
PA_BF16 = 1
PA_FP8_E4M3 = 2

PA_STATUS_BAD_SLOT = 1
PA_STATUS_BAD_BLOCK = 2
PA_STATUS_BAD_CONTEXT = 4
PA_STATUS_TIMEOUT = 8

# Size of the library's fixed decode scratch array (pa_decode_static_workspace).
PA_STATIC_WORKSPACE_BYTES = 16 << 20

# Most prefix groups one shared-prefix decode call takes.
PA_MAX_PREFIX_GROUPS = 64

_c_int, _c_i64, _c_sz, _c_f = ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
_vp = ctypes.c_void_p
_pi32 = ctypes.POINTER(ctypes.c_int32)
_pi64 = ctypes.POINTER(ctypes.c_int64)

# name -> (restype, argtypes)
SIGNATURES = {
    "pa_last_error": (ctypes.c_char_p, []),
    "pa_version": (_c_int, []),
    "pa_get_status": (_c_int, [_vp, ctypes.POINTER(ctypes.c_uint32)]),
    "pa_cache_append": (_c_int, [_vp, _vp, _vp, _c_int, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int, _vp]),
    "pa_copy_blocks": (_c_int, [_vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _vp]),
    "pa_decode_partition_size": (_c_int, [_c_int, _c_int, _c_int, _c_int]),
    "pa_decode_partition_size_shared_prefix": (_c_int, [_c_int, _c_int, _c_int, _c_int, _vp, _c_int]),
    "pa_decode_workspace_bytes": (_c_sz, [_c_int, _c_int, _c_int, _c_int, _c_int]),
    "pa_decode": (_c_int, [_vp, _vp, _vp, _vp, _c_int, _vp, _c_int, _c_f, _vp, _c_int, _c_int, _c_int, _c_int,
                           _c_int, _c_int, _c_int, _vp, _c_sz, _c_int, _vp]),
    "pa_prefill_test_items_per_launch": (_c_int, [_c_int]),
    "pa_prefill_test_withhold": (_c_int, [_c_int]),
    "pa_decode_test_withhold": (_c_int, [_vp, _vp, _vp, _vp, _c_int, _vp, _c_int, _c_f, _vp, _c_int, _c_int,
                                         _c_int, _c_int, _c_int, _c_int, _c_int, _vp, _c_sz, _c_int, _c_int, _vp]),
    "pa_decode_plan_bytes": (_c_sz, [_c_int, _c_int, _c_int]),
    "pa_decode_plan_host": (_c_int, [_vp, _c_int, _c_int, _c_int, _vp]),
    "pa_decode_planned": (_c_int, [_vp, _vp, _vp, _vp, _c_int, _vp, _c_int, _c_f, _vp, _c_int, _c_int, _c_int, _c_int,
                                   _c_int, _c_int, _c_int, _vp, _vp, _c_sz, _c_int, _vp]),
    "pa_decode_static_workspace": (_c_int, [_vp, _vp, _vp, _vp, _c_int, _vp, _c_int, _c_f, _vp, _c_int, _c_int,
                                            _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _vp]),
    "pa_cache_append_fp8": (_c_int, [_vp, _vp, _vp, _c_int, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_f, _c_f,
                                     _vp]),
    "pa_prefill": (_c_int, [_vp, _vp, _vp, _vp, _c_int, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_f, _vp, _vp, _vp,
                            _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _vp]),
    "pa_decode_fp8": (_c_int, [_vp, _vp, _vp, _vp, _c_int, _vp, _c_int, _c_f, _c_f, _c_f, _vp, _c_int, _c_int,
                               _c_int, _c_int, _c_int, _c_int, _c_int, _vp, _vp, _c_sz, _vp]),
    "pa_decode_shared_prefix": (_c_int, [_vp, _vp, _vp, _vp, _c_int, _vp, _c_int, _c_f, _vp, _c_int, _c_int,
                                         _c_int, _c_int, _c_int, _c_int, _c_int, _vp, _c_int, _vp, _c_sz, _c_int,
                                         _vp]),
    "pa_decode_plan_host_shared_prefix": (_c_int, [_vp, _c_int, _c_int, _c_int, _c_int, _c_int, _vp, _c_int, _vp]),
    "pa_decode_planned_shared_prefix": (_c_int, [_vp, _vp, _vp, _vp, _c_int, _vp, _c_int, _c_f, _vp, _c_int,
                                                 _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _vp, _c_int, _vp,
                                                 _vp, _c_sz, _c_int, _vp]),
    "pa_alloc_create": (_c_int, [_c_int, _c_int, _vp, ctypes.POINTER(_vp)]),
    "pa_alloc_destroy": (None, [_vp]),
    "pa_alloc_num_free": (_c_int, [_vp]),
    "pa_seq_add": (_c_int, [_vp, _c_i64, _c_int]),
    "pa_seq_fork": (_c_int, [_vp, _c_i64, _c_i64]),
    "pa_seq_append_slot": (_c_int, [_vp, _c_i64, _pi64, _pi32, _pi32]),
    "pa_seq_free": (_c_int, [_vp, _c_i64]),
    "pa_seq_num_tokens": (_c_int, [_vp, _c_i64]),
    "pa_seq_block_table": (_c_int, [_vp, _c_i64, _vp, _c_int, ctypes.POINTER(_c_int)]),
    "pa_block_refcount": (_c_int, [_vp, _c_int]),
    "pa_seqs_append_slots": (_c_int, [_vp, _vp, _c_int, _vp, _vp, ctypes.POINTER(_c_int), _vp, _c_int, _vp]),
    "pa_seqs_block_tables": (_c_int, [_vp, _vp, _c_int, _vp, _c_int, _vp]),
    "pa_stepper_layout": (_c_int, [_c_int, _c_int, _c_int, _c_int, ctypes.POINTER(_c_sz), ctypes.POINTER(_c_sz)]),
    "pa_stepper_create": (_c_int, [_vp, _vp, _c_int, _c_int, _c_int, _c_int, _vp, _vp, _vp, _c_sz,
                                   ctypes.POINTER(_vp)]),
    "pa_stepper_destroy": (None, [_vp]),
    "pa_stepper_prepare": (_c_int, [_vp, _vp, _vp, ctypes.POINTER(_c_int), ctypes.POINTER(_c_int)]),
    "pa_stepper_finish": (_c_int, [_vp, _vp]),
    "pa_stepper_set_prefix_groups": (_c_int, [_vp, _vp, _c_int, _c_int, _c_int]),
}

ERRORS = {-1: "PA_ERR_INVALID", -2: "PA_ERR_UNSUPPORTED", -3: "PA_ERR_OOM", -4: "PA_ERR_STATE", -5: "PA_ERR_CUDA"}


class PAError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{ERRORS.get(code, code)}: {msg}")
        self.code = code


class OutOfBlocks(PAError):
    pass


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library.  Raises if it has not been built: there is no
    other implementation to fall back on."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise RuntimeError(
                f"{LIB} is missing; build it with paged_kv_cache_216_gb300.build.build() (needs nvcc)")
        h = ctypes.CDLL(LIB)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(h, name)
            fn.restype = res
            fn.argtypes = args
        _lib = h
    return _lib


def check(rc: int) -> int:
    if rc < 0:
        msg = lib().pa_last_error().decode(errors="replace")
        raise (OutOfBlocks if rc == -3 else PAError)(rc, msg)
    return rc
