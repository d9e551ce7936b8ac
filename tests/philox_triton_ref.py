"""Philox4x32-10 words from triton's own Philox, run on the CPU interpreter.

Run as a script with TRITON_INTERPRET=1 in the environment. Reads a JSON
list of [c0, c1, c2, c3, k0, k1] on stdin and prints a JSON list of the four
output words for each. It serves the oracle's Philox pin only: an
implementation of the same published generator that this repository did
not write.
"""
import json
import sys

import torch
import triton
import triton.language as tl


@triton.jit
def _philox_kernel(c_ptr, k_ptr, o_ptr, n, BLOCK: tl.constexpr):
    offs = tl.program_id(0) * BLOCK + tl.arange(0, BLOCK)
    m = offs < n
    c0 = tl.load(c_ptr + offs * 4 + 0, mask=m).to(tl.uint32)
    c1 = tl.load(c_ptr + offs * 4 + 1, mask=m).to(tl.uint32)
    c2 = tl.load(c_ptr + offs * 4 + 2, mask=m).to(tl.uint32)
    c3 = tl.load(c_ptr + offs * 4 + 3, mask=m).to(tl.uint32)
    k0 = tl.load(k_ptr + offs * 2 + 0, mask=m).to(tl.uint32)
    k1 = tl.load(k_ptr + offs * 2 + 1, mask=m).to(tl.uint32)
    r0, r1, r2, r3 = tl.random.philox_impl(c0, c1, c2, c3, k0, k1, 10)
    tl.store(o_ptr + offs * 4 + 0, r0.to(tl.int64), mask=m)
    tl.store(o_ptr + offs * 4 + 1, r1.to(tl.int64), mask=m)
    tl.store(o_ptr + offs * 4 + 2, r2.to(tl.int64), mask=m)
    tl.store(o_ptr + offs * 4 + 3, r3.to(tl.int64), mask=m)


def main():
    rows = json.load(sys.stdin)
    n = len(rows)
    c = torch.tensor([r[:4] for r in rows], dtype=torch.int64)
    k = torch.tensor([r[4:] for r in rows], dtype=torch.int64)
    o = torch.zeros(n, 4, dtype=torch.int64)
    block = 64
    _philox_kernel[(triton.cdiv(n, block),)](c, k, o, n, BLOCK=block)
    json.dump(o.tolist(), sys.stdout)


if __name__ == "__main__":
    main()
