"""The C ABI library builds, loads without a GPU and exports every function include/verkv.h
declares; shape validation and status names need no GPU either."""
import ctypes
import os
import re

import pytest

from verified_kv_cache_poissoncomp_gb300 import binding as B
from verified_kv_cache_poissoncomp_gb300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return B.lib()


def declared_functions():
    with open(os.path.join(ROOT, "include", "verkv.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(verkv_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 12
    for name in names:
        assert hasattr(lib, name), name
    assert sorted(B.EXPORTED) == names


def test_workspace_size_and_shape_validation(lib):
    good = B.verkv_shape(1, 1, 8, 4, 128, 32768, 2600)
    ws = B.verkv_workspace_size(good)
    # scores 32*32768*4 + staging 8*32768*512 dominate
    assert ws >= 32 * 32768 * 4 + 8 * 32768 * 512
    bad = [B.verkv_shape(1, 1, 8, 3, 128, 32768, 2600),     # G not a power of two
           B.verkv_shape(1, 1, 8, 4, 96, 32768, 2600),      # d
           B.verkv_shape(1, 1, 8, 4, 128, 200000, 2600),    # n too large
           B.verkv_shape(1, 1, 8, 4, 128, 1000, 2000),      # cap > n
           B.verkv_shape(0, 1, 8, 4, 128, 1000, 100)]       # batch
    for s in bad:
        assert B.verkv_workspace_size(s) == 0
    # verkv_create rejects a bad shape or workspace before touching CUDA.
    ctx = ctypes.c_void_p()
    assert lib.verkv_create(ctypes.byref(ctx), 0, None, ctypes.byref(bad[0]), 256, 1 << 30) == \
        B.VERKV_EINVAL
    assert lib.verkv_create(ctypes.byref(ctx), 0, None, ctypes.byref(good), 0, ws) == B.VERKV_EINVAL
    assert lib.verkv_create(ctypes.byref(ctx), 0, None, ctypes.byref(good), 256, ws - 1) == \
        B.VERKV_EINVAL
    assert lib.verkv_create(ctypes.byref(ctx), 0, None, ctypes.byref(good), 257, ws) == \
        B.VERKV_EINVAL


def test_null_context_and_status_names(lib):
    assert lib.verkv_sync(None) == B.VERKV_EINVAL
    assert lib.verkv_fetch_refine(None, None, None, None, None, None, None) == B.VERKV_EINVAL
    assert lib.verkv_last_error(None) == b""
    for st, name in [(0, "VERKV_OK"), (2, "VERKV_EBUDGET"), (8, "VERKV_ESTATE"),
                     (9, "VERKV_ETOOLARGE")]:
        assert B.verkv_status_string(st) == name


def test_noalloc_argument_checks_need_no_gpu(lib):
    # The allocation-free certificate rejects an oversized or malformed call before touching CUDA
    # (dummy pointers: never dereferenced).
    c = lib.verkv_certify_noalloc
    args = [0, None, 8, 4, 128, 32768, 16, 16, 16, 0.05, 0.05, 16, 16, 16]
    big = list(args)
    big[5] = 131072  # 8 x 4 x 131072 = 2^22 logits: at the limit, so one more KV head is over
    big[2] = 9
    assert c(*big) == B.VERKV_ETOOLARGE
    for i, v in [(3, 3), (4, 96), (5, 0), (5, 131073), (2, 0), (6, None), (13, None), (9, 0.0),
                 (10, 1.0)]:
        bad = list(args)
        bad[i] = v
        assert c(*bad) == B.VERKV_EINVAL, (i, v)
    # Misaligned pointers: q and the sketch need 16 bytes (vector loads, bulk copies), the other
    # arrays 4; each is refused before any launch.
    for i, v in [(6, 24), (6, 18), (7, 40), (7, 17), (8, 18), (11, 21), (12, 22), (13, 19)]:
        bad = list(args)
        bad[i] = v
        assert c(*bad) == B.VERKV_EINVAL, (i, v)


def test_kernel_ids_and_names_match_the_header(lib):
    with open(os.path.join(ROOT, "include", "verkv.h")) as f:
        text = f.read()
    body = text[text.index("VERKV_K_PC_SOLVE = 0"):text.index("VERKV_K_COUNT")]
    ids = re.findall(r"\b(VERKV_K_[A-Z_]+)", body)
    assert [getattr(B, k) for k in ids] == list(range(len(ids)))
    assert B.VERKV_K_COUNT == len(ids)
    assert B.verkv_kernel_name(B.VERKV_K_CERTIFY) == "k_certify"
    assert B.verkv_kernel_name(B.VERKV_K_COUNT) == ""


def test_sketch_bytes(lib):
    s = B.verkv_shape(2, 3, 8, 4, 128, 32768, 2600)
    rows = 2 * 3 * 8 * 32768
    assert B.verkv_sketch_bytes(s, B.VERKV_SKETCH_EXACT) == rows * 256
    assert B.verkv_sketch_bytes(s, B.VERKV_SKETCH_Q2) == rows * 48
    s64 = B.verkv_shape(1, 1, 1, 4, 64, 1000, 100)
    assert B.verkv_sketch_bytes(s64, B.VERKV_SKETCH_Q2) == 1000 * 32
    assert B.verkv_sketch_bytes(s, 7) == 0


def test_default_capacity():
    # eta n plus 8 standard deviations of the Poisson sample size plus 64, rounded up to a
    # multiple of 16 so that the MEMCPY path can bulk-copy each pivotal item's id and r lists,
    # and never more than n.
    import math

    from verified_kv_cache_poissoncomp_gb300.engine import default_cap
    for n in (1000, 3000, 8192, 20000, 32768, 50001, 131072):
        for eta in (1 / 32, 1 / 16, 1 / 8, 1 / 4, 1.0):
            m = eta * n
            need = m + 8.0 * math.sqrt(m) + 64
            c = default_cap(n, eta)
            assert c <= n
            if c < n:
                assert c % 16 == 0 and need <= c < need + 17, (n, eta, c)
