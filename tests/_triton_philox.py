"""Runs Triton's Philox4x32 (its CPU interpreter, numpy underneath) as a black
box: reads JSON [[seed, c0, c1, c2, c3], ...] on stdin, prints the four output
words of each.  Test helper, run in a subprocess so that the interpreter
setting stays out of the test process; not collected by pytest."""

import json
import os
import sys

os.environ["TRITON_INTERPRET"] = "1"

import torch  # noqa: E402
import triton  # noqa: E402
import triton.language as tl  # noqa: E402


@triton.jit
def _philox_kernel(seed_ptr, c_ptr, out_ptr, n: tl.constexpr):
    i = tl.arange(0, n)
    seed = tl.load(seed_ptr + i)
    c0 = tl.load(c_ptr + 4 * i + 0)
    c1 = tl.load(c_ptr + 4 * i + 1)
    c2 = tl.load(c_ptr + 4 * i + 2)
    c3 = tl.load(c_ptr + 4 * i + 3)
    a, b, c, d = tl.philox(seed, c0, c1, c2, c3, 10)
    tl.store(out_ptr + 4 * i + 0, a)
    tl.store(out_ptr + 4 * i + 1, b)
    tl.store(out_ptr + 4 * i + 2, c)
    tl.store(out_ptr + 4 * i + 3, d)


def main():
    cases = json.loads(sys.stdin.read())
    n = 1
    while n < len(cases):
        n *= 2
    seeds = torch.zeros(n, dtype=torch.int64)
    ctr = torch.zeros(4 * n, dtype=torch.int64)
    for i, (s, *c) in enumerate(cases):
        seeds[i] = s - (1 << 64) if s >= (1 << 63) else s
        for j in range(4):
            ctr[4 * i + j] = c[j]
    # 32-bit words as two's-complement int32 (same bits)
    ctr = (ctr - (ctr >= (1 << 31)).to(torch.int64) * (1 << 32)).to(torch.int32)
    out = torch.zeros(4 * n, dtype=torch.int32)
    _philox_kernel[(1,)](seeds, ctr, out, n=n)
    res = [[int(x) & 0xFFFFFFFF for x in out[4 * i:4 * i + 4].tolist()]
           for i in range(len(cases))]
    print(json.dumps(res))


if __name__ == "__main__":
    main()
