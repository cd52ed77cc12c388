"""Pins for the oracle's Philox4x32-10 and its 24-bit uniforms.

The pages only ask for independent Bernoulli draws ("Verify Before You Fetch", summary page,
Methodology, PoissonComp); the generator is our reading.  The oracle's Philox is pinned to an
independent implementation of the same published generator: Triton's `tl.philox`, executed on the
CPU by Triton's interpreter (a library routine, not code of this repository).
"""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

import oracle as O

_TRITON_SCRIPT = r"""
import json, os, sys
os.environ["TRITON_INTERPRET"] = "1"
import numpy as np
import torch
import triton
import triton.language as tl

@triton.jit
def _k(c_ptr, out_ptr, seed, N: tl.constexpr):
    o = tl.arange(0, N)
    c0 = tl.load(c_ptr + 4 * o + 0)
    c1 = tl.load(c_ptr + 4 * o + 1)
    c2 = tl.load(c_ptr + 4 * o + 2)
    c3 = tl.load(c_ptr + 4 * o + 3)
    a, b, c, d = tl.philox(seed, c0, c1, c2, c3)
    tl.store(out_ptr + 4 * o + 0, a)
    tl.store(out_ptr + 4 * o + 1, b)
    tl.store(out_ptr + 4 * o + 2, c)
    tl.store(out_ptr + 4 * o + 3, d)

cases = json.loads(sys.stdin.read())
res = []
for seed, ctrs in cases:
    c = torch.tensor(np.array(ctrs, dtype=np.uint32).view(np.int32).reshape(-1))
    out = torch.zeros_like(c)
    _k[(1,)](c, out, seed, N=len(ctrs))
    res.append((out.numpy().view(np.uint32).reshape(-1, 4)).tolist())
print(json.dumps(res))
"""


def _triton_philox(cases):
    pytest.importorskip("triton")
    env = dict(os.environ, TRITON_INTERPRET="1")
    p = subprocess.run([sys.executable, "-c", _TRITON_SCRIPT], input=json.dumps(cases),
                       capture_output=True, text=True, env=env, timeout=300)
    if p.returncode != 0:
        pytest.skip(f"triton interpreter unavailable: {p.stderr[-400:]}")
    return json.loads(p.stdout)


def test_philox_matches_triton_interpreter():
    rng = np.random.default_rng(7)
    seeds = [0, 1, 0xFFFFFFFF, 0x123456789ABCDEF0, (1 << 64) - 1, 42]
    cases = []
    for s in seeds:
        ctrs = rng.integers(0, 1 << 32, size=(32, 4), dtype=np.uint64).astype(np.uint32)
        ctrs[0] = [0, 0, 0, 0]
        ctrs[1] = [0xFFFFFFFF] * 4
        ctrs[2] = [5, 3, 2, 1]
        cases.append((s if s < (1 << 63) else s - (1 << 64), ctrs.tolist()))
    ref = _triton_philox(cases)
    for (s, ctrs), outs in zip(cases, ref):
        su = s & ((1 << 64) - 1)
        key = [su & 0xFFFFFFFF, su >> 32]
        for c, want in zip(ctrs, outs):
            got = O.philox4x32_10(c, key)
            assert got.tolist() == want, (hex(su), c)


def test_uniform24_layout_and_range():
    # u_i is word (i mod 4) of the block at counter (i // 4, head, layer, seq), top 24 bits.
    seed, seq, layer, head = 0x0123456789ABCDEF, 3, 5, 7
    key = [seed & 0xFFFFFFFF, seed >> 32]
    for i in [0, 1, 2, 3, 4, 5, 1023, 4097, (1 << 20) + 3]:
        block = O.philox4x32_10([i // 4, head, layer, seq], key)
        want = float(block[i % 4] >> 8) / float(1 << 24)
        assert O.uniform24(seed, seq, layer, head, i) == want
        assert 0.0 <= want < 1.0


def test_uniform24_chi_square():
    # 2^16 draws into 64 equal bins: chi^2 with 63 dof stays well below its 1e-4 tail (~112).
    M, bins = 1 << 16, 64
    u = np.array([O.uniform24(99, 0, 1, 2, i) for i in range(M)])
    counts = np.bincount((u * bins).astype(int), minlength=bins)
    exp = M / bins
    chi2 = ((counts - exp) ** 2 / exp).sum()
    assert chi2 < 112.0, chi2
    # Serial pairs (u_i, u_{i+1}) on an 8x8 grid: also uniform.
    pairs = (u[:-1:2] * 8).astype(int) * 8 + (u[1::2] * 8).astype(int)
    c2 = np.bincount(pairs, minlength=64)
    e2 = len(pairs) / 64
    assert ((c2 - e2) ** 2 / e2).sum() < 112.0
