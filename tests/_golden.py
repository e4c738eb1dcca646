"""Parsers for the hand-derived fixtures in tests/golden/."""

from __future__ import annotations

import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for raw in f:
            line = raw.split("#", 1)[0].strip()
            if line:
                yield line


def allocator_trace():
    """Returns ``(init, steps)``: init = (num_blocks, block_size, free_order);
    steps = list of ("op", op, args, result) and ("expect", dict)."""
    init = None
    steps = []
    for line in _lines("allocator_trace.txt"):
        if line.startswith("init "):
            _, n, b, order = line.split()
            init = (int(n), int(b), [int(x) for x in order.split(",")])
        elif line.startswith("expect "):
            kv = {}
            for tok in line.split()[1:]:
                k, v = tok.split("=")
                kv[k] = [int(x) for x in v.split(",")] if k.startswith("table.") else int(v)
            steps.append(("expect", kv))
        else:
            lhs, rhs = [x.strip() for x in line.split("=>")]
            parts = lhs.split()
            op, args = parts[0], [int(x) for x in parts[1:]]
            if rhs in ("ok", "oom"):
                res = rhs
            else:
                slot_tok, cow_tok = rhs.split()
                src, dst = cow_tok.split("=")[1].split(",")
                res = (int(slot_tok.split("=")[1]), int(src), int(dst))
            steps.append(("op", op, args, res))
    return init, steps


def append_layout():
    d = {}
    for line in _lines("append_layout.txt"):
        key, *vals = line.split()
        d[key] = vals
    shape = tuple(int(x) for x in d["shape"])
    n, hkv, b, dim = shape
    slots = np.array([int(x) for x in d["slots"]], dtype=np.int64)
    t = len(slots)
    k = np.array([float(x) for x in d["k"]], dtype=np.float32).reshape(t, hkv, dim)
    v = np.array([float(x) for x in d["v"]], dtype=np.float32).reshape(t, hkv, dim)

    def nz(key):
        out = np.zeros(int(np.prod(shape)), dtype=np.float32)
        for tok in d[key]:
            i, val = tok.split(":")
            out[int(i)] = float(val)
        return out.reshape(shape)

    return shape, slots, k, v, nz("k_nonzero"), nz("v_nonzero")
