"""The oracle's pins catch planted mistakes.  Each case replaces one oracle
function by a plausibly wrong variant (on the CPU, in this process only) and
checks that at least one pin of tests/test_oracle_attention.py fails."""

import numpy as np
import pytest

import oracle.attention as att
import tests.test_oracle_attention as pins


def _wrong_gqa(q, k_cache, v_cache, block_tables, context_lens, scale, dtype, seqs=None):
    """KV head h % Hkv instead of h // g."""
    s_all, h, d = q.shape
    hkv = k_cache.shape[1]
    seqs = range(s_all) if seqs is None else list(seqs)
    out = np.empty((len(seqs), h, d))
    for i, s in enumerate(seqs):
        n = int(context_lens[s])
        for hh in range(h):
            kv = hh % hkv
            k = att.to_f64(att.gather_sequence(k_cache, block_tables[s], n, kv), dtype)
            v = att.to_f64(att.gather_sequence(v_cache, block_tables[s], n, kv), dtype)
            out[i, hh] = att.decode_one(att.to_f64(q[s, hh:hh + 1], dtype), k, v, scale)[0]
    return out


def _no_scale(q_heads, k_rows, v_rows, scale):
    return _orig_decode_one(q_heads, k_rows, v_rows, 1.0)


def _swap_kv(q_heads, k_rows, v_rows, scale):
    return _orig_decode_one(q_heads, v_rows, k_rows, scale)


def _no_max(q_heads, k_rows, v_rows, scale):
    z = scale * (q_heads @ k_rows.T)
    with np.errstate(over="ignore", invalid="ignore"):
        p = np.exp(z)
        p = p / p.sum(axis=1, keepdims=True)
    return p @ v_rows


def _off_by_one_gather(cache, table_row, ctx, kv_head):
    return _orig_gather(cache, table_row, ctx + 1, kv_head)[1:]


_orig_decode_one = att.decode_one
_orig_gather = att.gather_sequence
PIN_TESTS = [getattr(pins, n) for n in dir(pins) if n.startswith("test_") and "bf16_inputs" not in n]


@pytest.mark.parametrize("target,wrong", [
    ("paged_decode", _wrong_gqa),
    ("decode_one", _no_scale),
    ("decode_one", _swap_kv),
    ("decode_one", _no_max),
    ("gather_sequence", _off_by_one_gather),
])
def test_a_planted_mistake_fails_some_pin(monkeypatch, target, wrong):
    monkeypatch.setattr(att, target, wrong)
    monkeypatch.setattr(pins, "paged_decode", att.paged_decode)
    failed = []
    for t in PIN_TESTS:
        args = [] if t.__code__.co_argcount == 0 else None
        if args is None:
            continue
        try:
            t()
        except Exception:  # noqa: BLE001 - any failure counts
            failed.append(t.__name__)
    assert failed, f"no pin caught the planted mistake in {target}"
