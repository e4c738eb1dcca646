"""The C ABI library loads, exports every symbol its header declares, and
rejects bad host-side arguments before touching the GPU (no GPU needed).

The refusal cases pass made-up device addresses for the pointers they do not
test.  They run in a child process that sees no GPU (tests/_abi_child.py):
should a host-side check ever stop refusing one of them, the call fails with
a CUDA "no device" error there instead of launching a kernel on the bogus
address on whatever GPU this suite runs on."""

import ctypes
import json
import os
import re
import subprocess
import sys

import numpy as np
import pytest

from tests._lib_fixture import ensure_built

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FAKE = {"ptr": 0x100000}  # a made-up device address (only ever used where no GPU is visible)


def run_without_gpu(calls):
    """[(function, args)] -> [(rc, message)], made in a process with
    CUDA_VISIBLE_DEVICES="" ."""
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "_abi_child.py")],
                       input=json.dumps([[f, a] for f, a in calls]), capture_output=True, text=True, env=env,
                       cwd=ROOT, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    return [tuple(x) for x in json.loads(r.stdout.strip().splitlines()[-1])]


@pytest.fixture(scope="module")
def L():
    ensure_built()
    from paged_kv_cache_216_gb300._lib import lib

    return lib()


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if not fn.endswith(".h"):
            continue
        with open(os.path.join(ROOT, "include", fn)) as f:
            src = f.read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        for m in re.finditer(r"\b(pa_[a-z0-9_]+)\s*\(", src):
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("pa_cache_append", "pa_decode", "pa_copy_blocks", "pa_alloc_create", "pa_seq_fork",
                     "pa_seq_append_slot", "pa_decode_workspace_bytes"):
        assert required in names


def test_library_exports_every_declared_symbol(L):
    from paged_kv_cache_216_gb300._lib import SIGNATURES

    for name in declared_functions():
        assert hasattr(L, name), name
        assert name in SIGNATURES, f"binding lacks {name}"


def test_version(L):
    assert L.pa_version() == 1


def _decode_args(**over):
    a = dict(q=FAKE, k=FAKE, v=FAKE, bt=FAKE, mb=8, ctx=FAKE, maxctx=100, scale=0.1, out=FAKE, S=2, H=8, Hkv=2,
             D=128, B=16, N=10, P=0, ws=FAKE, wsb=1 << 30, dtype=1, stream=None)
    a.update(over)
    return [a[k] for k in ("q", "k", "v", "bt", "mb", "ctx", "maxctx", "scale", "out", "S", "H", "Hkv", "D", "B",
                           "N", "P", "ws", "wsb", "dtype", "stream")]


DECODE_CASES = [
    (dict(H=12, Hkv=4), -2),              # g = 3
    (dict(H=32, Hkv=2), -2),              # g = 16
    (dict(H=8, Hkv=3), -1),               # not a multiple
    (dict(D=96), -2),
    (dict(B=24), -2),
    (dict(dtype=7), -2),
    (dict(maxctx=0), -1),
    (dict(mb=6), -1),                     # 6 blocks of 16 < 100 tokens
    (dict(P=48), -1),                     # not a multiple of 32
    (dict(q=None), -1),
    (dict(q={"ptr": 0x100004}), -1),      # misaligned
    (dict(wsb=16), -1),                   # workspace too small
    (dict(scale=float("nan")), -1),
]


def _prefill_args(**over):
    a = dict(q=FAKE, k=FAKE, v=FAKE, slots=FAKE, T=64, qs=FAKE, ctx=FAKE, bt=FAKE, mb=8, mql=64, maxctx=128,
             scale=0.1, kc=FAKE, vc=FAKE, out=FAKE, S=1, H=8, Hkv=2, D=128, B=16, N=16, dtype=1, stream=None)
    a.update(over)
    return [a[k] for k in ("q", "k", "v", "slots", "T", "qs", "ctx", "bt", "mb", "mql", "maxctx", "scale", "kc",
                           "vc", "out", "S", "H", "Hkv", "D", "B", "N", "dtype", "stream")]


PREFILL_CASES = [
    (dict(H=12, Hkv=4), -2),              # g = 3
    (dict(H=32, Hkv=2), -2),              # g = 16
    (dict(D=96), -2),
    (dict(dtype=2), -2),                  # FP8 caches are decode-only
    (dict(dtype=0), -2),                  # fp16
    (dict(mql=200), -1),                  # longer than the context
    (dict(mb=4), -1),                     # 4 blocks of 16 < 128 tokens
    (dict(S=70000), -2),
    # 8 heads per KV head x 1.1M prompt tokens = 68750 query tiles of 128 rows
    (dict(H=16, Hkv=2, mql=1_100_000, maxctx=1_100_000, mb=70_000), -2),
    (dict(q=None), -1),
    (dict(q={"ptr": 0x100004}), -1),      # misaligned
]

f = FAKE
OTHER_CASES = [
    ("pa_cache_append", [f, f, f, 4, f, f, 10, 2, 96, 16, 1, None], -2),
    ("pa_cache_append", [f, f, f, -1, f, f, 10, 2, 128, 16, 1, None], -1),
    ("pa_cache_append", [None, f, f, 4, f, f, 10, 2, 128, 16, 1, None], -1),
    ("pa_cache_append", [f, f, f, 0, f, f, 10, 2, 128, 16, 1, None], 0),  # nothing to do
    ("pa_copy_blocks", [f, f, f, 3, 10, 2, 128, 12, 1, None], -2),
    ("pa_copy_blocks", [f, f, None, 3, 10, 2, 128, 16, 1, None], -1),
    ("pa_copy_blocks", [f, f, f, 0, 10, 2, 128, 16, 1, None], 0),
]
del f


@pytest.fixture(scope="module")
def refusals(L):
    calls = ([("pa_decode", _decode_args(**o)) for o, _ in DECODE_CASES] +
             [("pa_prefill", _prefill_args(**o)) for o, _ in PREFILL_CASES] +
             [(fn, a) for fn, a, _ in OTHER_CASES])
    res = run_without_gpu(calls)
    nd, npf = len(DECODE_CASES), len(PREFILL_CASES)
    return res[:nd], res[nd:nd + npf], res[nd + npf:]


@pytest.mark.parametrize("i", range(len(DECODE_CASES)))
def test_decode_rejects_bad_arguments_without_a_launch(refusals, i):
    rc, msg = refusals[0][i]
    assert rc == DECODE_CASES[i][1], msg
    assert msg


@pytest.mark.parametrize("i", range(len(PREFILL_CASES)))
def test_prefill_rejects_bad_arguments_without_a_launch(refusals, i):
    rc, msg = refusals[1][i]
    assert rc == PREFILL_CASES[i][1], msg
    assert msg


def test_append_and_copy_reject_bad_arguments(refusals):
    for (fn, args, code), (rc, msg) in zip(OTHER_CASES, refusals[2]):
        assert rc == code, (fn, args, msg)


def test_partition_and_workspace_sizing(L):
    # explicit partition sizes pass through; auto sizing is a multiple of 32
    assert L.pa_decode_partition_size(8, 8, 131072, 512) == 512
    # a wide batch: one partition per context up to 4096 tokens, else 4096
    assert L.pa_decode_partition_size(256, 8, 4116, 0) == 4096
    assert L.pa_decode_partition_size(32, 32, 2068, 0) == 2080
    # a narrow one keeps 512-token partitions (or smaller, for enough items)
    assert L.pa_decode_partition_size(64, 8, 8200, 0) == 512
    p = L.pa_decode_partition_size(1, 1, 5000, 0)
    assert p % 32 == 0 and 64 <= p < 512
    assert L.pa_decode_partition_size(1, 1, 100, 33) == -1
    # with prefix groups: doubled up to 1024 while every prefix holds a
    # whole partition; explicit sizes and wide batches unchanged
    def shared(S, hkv, mx, P, groups):
        g = np.ascontiguousarray(np.asarray(groups, dtype=np.int32).reshape(-1, 3))
        return L.pa_decode_partition_size_shared_prefix(S, hkv, mx, P, ctypes.c_void_p(g.ctypes.data), g.shape[0])
    assert shared(64, 8, 8200, 0, [(0, 32, 1024)]) == 1024
    assert shared(64, 8, 8200, 0, [(0, 32, 1024), (40, 4, 600)]) == 512
    assert shared(64, 8, 8200, 0, [(0, 32, 5000)]) == 1024
    assert shared(64, 8, 8200, 256, [(0, 32, 1024)]) == 256
    assert shared(9, 8, 2600, 0, [(0, 6, 1024)]) == 1024  # from 128
    assert shared(9, 8, 2600, 0, [(0, 6, 100)]) == L.pa_decode_partition_size(9, 8, 2600, 0)
    assert shared(256, 8, 4116, 0, [(0, 32, 1024)]) == 4096
    assert L.pa_decode_partition_size_shared_prefix(64, 8, 8200, 0, None, 0) == 512
    assert L.pa_decode_partition_size_shared_prefix(64, 8, 8200, 0, None, 1) < 0
    # one partition: header + work list only
    assert L.pa_decode_workspace_bytes(4, 8, 128, 512, 512) == 256 + 256
    # header, work list (8 B per sequence x partition, 256-aligned), then
    # S * parts * H rows of D fp32 (256-aligned) and a float2 per row
    pairs, rows = 8 * 256, 8 * 256 * 64
    assert L.pa_decode_workspace_bytes(8, 64, 128, 131072, 512) == 256 + pairs * 8 + rows * 128 * 4 + rows * 8
    pairs, rows = 3 * 2, 3 * 2 * 5
    assert L.pa_decode_workspace_bytes(3, 5, 64, 600, 512) == 256 + 256 + ((rows * 64 * 4 + 255) // 256) * 256 + rows * 8
    assert L.pa_decode_workspace_bytes(0, 5, 64, 600, 512) == 0
