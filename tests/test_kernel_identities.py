"""The integer and algebraic rewrites the CUDA kernels rely on, checked on the CPU against the
quantities they stand for (the kernels themselves are checked against the oracle by the GPU tests).

* PoissonComp sums tau exactly as floor(tau 2^46), built from the float's bits: with tau =
  m 2^(e - 150) (m the significand with its implicit bit, e the biased exponent),
  floor(tau 2^46) = (m 2^23) >> (127 - e).
* Its budget check sums r as floor(r 2^24) = m >> (126 - e) below 1, and 2^24 at 1.
* The estimator weighs a sampled, unfetched token by lambda / r with lambda = clip(beta r /
  (w-hat (1 - r)), r, 1) (summary page, Definition 2); the kernel takes the quotient directly as
  clip(beta / (w-hat (1 - r)), 1, 1 / r), and 1 / r when w-hat underflows (lambda = 1).
"""
import numpy as np


def _bits_sample(rng, k=2_000_000):
    """float32 bit patterns of (0, 1]: uniform over the patterns, plus the edge cases."""
    b = rng.integers(1, 0x3F800001, size=k, dtype=np.int64).astype(np.uint32)
    edges = np.array([1, 2, 0x007FFFFF, 0x00800000, 0x00800001, 0x2B7FFFFF, 0x2B800000,
                      0x33800000, 0x3F000000, 0x3F7FFFFF, 0x3F800000], dtype=np.uint32)
    return np.concatenate([b, edges])


def _fixed46(b):
    e = (b >> np.uint32(23)).astype(np.int64)
    m = ((b & np.uint32(0x7FFFFF)) | np.where(e > 0, np.uint32(0x800000), np.uint32(0))).astype(np.uint64)
    rs = 127 - e
    return np.where(rs < 64, (m << np.uint64(23)) >> np.minimum(rs, 63).astype(np.uint64), np.uint64(0))


def _fixed24(b):
    e = (b >> np.uint32(23)).astype(np.int64)
    m = ((b & np.uint32(0x7FFFFF)) | np.where(e > 0, np.uint32(0x800000), np.uint32(0))).astype(np.uint64)
    rs = 126 - e
    shifted = m >> np.clip(rs, 0, 31).astype(np.uint64)
    return np.where(e >= 127, np.uint64(1 << 24), np.where(rs < 32, shifted, np.uint64(0)))


def test_tau_fixed_point_from_bits():
    b = _bits_sample(np.random.default_rng(46))
    x = b.view(np.float32).astype(np.float64)
    # x 2^46 is exact in float64 (24 significant bits), so floor() is the exact integer part
    want = np.floor(x * 2.0 ** 46).astype(np.uint64)
    assert np.array_equal(_fixed46(b), want)


def test_r_fixed_point_from_bits():
    b = _bits_sample(np.random.default_rng(24))
    r = b.view(np.float32).astype(np.float64)
    want = np.floor(r * 2.0 ** 24).astype(np.uint64)
    assert np.array_equal(_fixed24(b), want)


def test_lambda_over_r_rewrite():
    rng = np.random.default_rng(5)
    k = 200_000
    r = np.concatenate([rng.uniform(1e-6, 1 - 1e-6, k), [1e-6, 0.5, 1 - 1e-9]])
    wh = np.concatenate([np.exp(rng.uniform(-60.0, 0.0, k)), [1e-30, 1.0, 0.25]])
    beta = np.concatenate([np.exp(rng.uniform(-40.0, 5.0, k)), [0.0, 3.0, 1e-12]])
    lam = np.clip(beta * r / (wh * (1.0 - r)), r, 1.0)
    direct = np.minimum(1.0 / r, np.maximum(1.0, beta / (wh * (1.0 - r))))
    np.testing.assert_allclose(direct, lam / r, rtol=1e-12)
