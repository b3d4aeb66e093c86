"""Philox4x32-10 words from triton's own implementation, run by triton's CPU interpreter.

Used by the oracle pin tests as an independent reference for the oracle's
Philox.  Run as a subprocess (the interpreter must be enabled before triton
is imported): reads {"c": [[c0...], [c1...], [c2...], [c3...]], "keys": [[k0, k1], ...]}
as JSON on stdin, prints [[[w0, w1, w2, w3], ...] per key] as JSON.
"""
import json
import os
import sys

os.environ["TRITON_INTERPRET"] = "1"

import numpy as np  # noqa: E402
import torch  # noqa: E402
import triton  # noqa: E402
import triton.language as tl  # noqa: E402


@triton.jit
def _kern(out_ptr, key_ptr, c0_ptr, c1_ptr, c2_ptr, c3_ptr, N: tl.constexpr):
    i = tl.arange(0, N)
    a0 = tl.load(c0_ptr + i)
    a1 = tl.load(c1_ptr + i)
    a2 = tl.load(c2_ptr + i)
    a3 = tl.load(c3_ptr + i)
    k0 = tl.load(key_ptr + i * 0)
    k1 = tl.load(key_ptr + 1 + i * 0)
    r0, r1, r2, r3 = tl.philox_impl(a0, a1, a2, a3, k0, k1, 10)
    tl.store(out_ptr + 4 * i + 0, r0)
    tl.store(out_ptr + 4 * i + 1, r1)
    tl.store(out_ptr + 4 * i + 2, r2)
    tl.store(out_ptr + 4 * i + 3, r3)


def main():
    req = json.load(sys.stdin)
    cs = [torch.tensor(np.array(c, dtype=np.uint64).astype(np.uint32)) for c in req["c"]]
    n = cs[0].numel()
    res = []
    for k0, k1 in req["keys"]:
        key = torch.tensor(np.array([k0, k1], dtype=np.uint64).astype(np.uint32))
        out = torch.zeros(4 * n, dtype=torch.uint32)
        _kern[(1,)](out, key, *cs, N=n)
        res.append(out.numpy().astype(np.uint64).reshape(n, 4).tolist())
    json.dump(res, sys.stdout)


if __name__ == "__main__":
    main()
