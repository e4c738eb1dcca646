"""Child process for the C-ABI refusal tests: makes the calls it reads from
standard input and prints, for each, the return code and pa_last_error().

The parent starts it with CUDA_VISIBLE_DEVICES set to the empty string, so
this process sees no GPU.  The calls pass made-up device addresses for the
pointers a case does not test (they must get past the null-pointer checks to
reach the check under test); should a host-side check ever stop refusing
such a call, the library's first CUDA call fails with "no device" and the
case returns PA_ERR_CUDA instead of launching a kernel on a bogus address.

Input: a JSON list of [function name, [argument, ...]], an argument being a
number, null, or {"ptr": address}.  Output: one JSON list of [rc, message].
"""

import ctypes
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def main():
    if os.environ.get("CUDA_VISIBLE_DEVICES", None) != "":
        raise SystemExit("refusing to run: CUDA_VISIBLE_DEVICES must be set to the empty string")
    from paged_kv_cache_216_gb300._lib import lib

    L = lib()
    calls = json.loads(sys.stdin.read())
    out = []
    for name, args in calls:
        conv = [ctypes.c_void_p(a["ptr"]) if isinstance(a, dict) else a for a in args]
        rc = getattr(L, name)(*conv)
        out.append([rc, L.pa_last_error().decode(errors="replace")])
    print(json.dumps(out))


if __name__ == "__main__":
    main()
