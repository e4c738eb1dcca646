"""Builds libpa.so once per test session if it is missing or stale."""

from __future__ import annotations

import threading

_lock = threading.Lock()
_done = False


def ensure_built():
    global _done
    with _lock:
        if not _done:
            from paged_kv_cache_216_gb300 import build

            build.build()
            _done = True
