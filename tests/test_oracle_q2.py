"""Pins of the oracle's 2-bit sketch: the binary16 directed rounding against numpy's float16 (an
independent library conversion), the byte layout by decoding, and the quantiser by the bounds a
nearest-level 4-level code must meet (every k-hat within half a step of its key, the levels
covering the group's range)."""
import numpy as np

import oracle as O
from verified_kv_cache_poissoncomp_gb300.inputs import f32_to_bf16


def _f16_neighbours(x):
    h = np.float16(x)  # round to nearest even: one of the two neighbours
    lo = h if float(h) <= x else np.nextafter(h, np.float16(-np.inf))
    hi = h if float(h) >= x else np.nextafter(h, np.float16(np.inf))
    return float(lo), float(hi)


def test_f16_directed_rounding_matches_float16_neighbours():
    rng = np.random.default_rng(5)
    xs = np.concatenate([np.clip(rng.standard_normal(2000) * 10 ** rng.uniform(-9, 4.7, 2000),
                                 -65000.0, 65000.0),
                         [0.0, 1.0, -1.0, 65504.0, -65504.0, 2.0 ** -24, 2.0 ** -14,
                          2.0 ** -14 - 2.0 ** -30, 1.0 + 2.0 ** -11, 3.0e-8, -7.1e-6]])
    for x in xs:
        lo, hi = _f16_neighbours(x)
        assert O.f16_round(x, -1) == lo, x
        assert O.f16_round(x, +1) == hi, x
    # signed zero and the smallest subnormal
    assert O.f16_bits(-0.0) == 0x8000 and O.f16_bits(0.0) == 0
    assert O.f16_round(-1e-12, -1) == -2.0 ** -24 and O.f16_round(1e-12, -1) == 0.0
    # beyond the finite range: clamped
    assert O.f16_round(1e6, +1) == 65504.0 and O.f16_round(-1e6, -1) == -65504.0


def test_f16_bits_match_float16_encoding():
    rng = np.random.default_rng(6)
    vals = np.float16(rng.standard_normal(3000) * 10 ** rng.uniform(-7, 4.5, 3000))
    vals = np.concatenate([vals, np.float16([0.0, 6e-8, -6e-8, 65504.0, 2.0 ** -14])])
    for v in vals:
        if not np.isfinite(v):
            continue
        b = O.f16_bits(float(v))
        assert b == int(np.array(v, dtype=np.float16).view(np.uint16)), float(v)
        assert O.f16_value(b) == float(v)


def _decode(rows, d):
    n = rows.shape[0]
    codes = np.zeros((n, d), dtype=np.int64)
    for c in range(d):
        codes[:, c] = (rows[:, c // 4] >> (2 * (c % 4))) & 3
    ng = d // 32
    par = rows[:, d // 4:d // 4 + 4 * ng].copy().view(np.uint16).reshape(n, ng, 2)
    lo = par[..., 0].view(np.float16).astype(np.float64)
    step = par[..., 1].view(np.float16).astype(np.float64)
    return codes, lo, step


def test_q2_sketch_layout_and_quantisation_bounds():
    rng = np.random.default_rng(7)
    for d in (64, 128):
        n = 300
        x = rng.standard_normal((n, d)).astype(np.float32) * np.where(rng.random(d) < 0.1, 8, 1)
        x[0, :32] = 1.5  # a constant group: step 0
        kb = f32_to_bf16(x)
        rows, khat = O.q2_sketch(kb)
        assert rows.shape == (n, O.q2_row_bytes(d)) and rows.shape[1] % 16 == 0
        assert not rows[:, d // 4 + 4 * (d // 32):].any()  # padding is zero
        codes, lo, step = _decode(rows, d)
        xf = O.bf16_to_f64(kb).reshape(n, d // 32, 32)
        # the exact dequantised keys follow from the bytes alone
        rebuilt = lo[..., None] + codes.reshape(n, d // 32, 32) * step[..., None]
        assert np.array_equal(rebuilt.reshape(n, d), khat)
        # lo is at or below the group minimum and the top level reaches the maximum
        assert np.all(lo <= xf.min(-1))
        assert np.all(lo + 3 * step >= xf.max(-1) * (1 - 1e-7) - 1e-30)
        # every key lies within half a step of its level (float32 arithmetic in the rule)
        err = np.abs(khat.reshape(n, d // 32, 32) - xf)
        assert np.all(err <= 0.5 * step[..., None] * (1 + 1e-6) + 1e-12)
        assert codes[0, :32].max() == 0 and step[0, 0] == 0.0 and khat[0, 0] == lo[0, 0]
