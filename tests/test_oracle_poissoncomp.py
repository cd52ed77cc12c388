"""Pins for the oracle's PoissonComp ("Verify Before You Fetch", summary page, Methodology,
POISSONCOMP, Eq. (3), the H / L partition and the Poisson sample S)."""
import numpy as np
import pytest
from scipy.optimize import brentq

import oracle as O


def _lognormal_tau(rng, n):
    x = rng.lognormal(0.0, 1.5, n)
    return (x / x.max()).astype(np.float32)


def _forced(n, n_sink, n_local):
    i = np.arange(n)
    return (i < n_sink) | (i >= n - n_local)


@pytest.mark.parametrize("n,eta", [(1024, 1 / 8), (4096, 1 / 16), (32768, 1 / 16),
                                   (32768, 1 / 32), (32768, 1 / 8), (5000, 0.3)])
def test_budget_sum_equals_eta_n(n, eta):
    # Eq. (3): c is chosen so that sum_i min(1, c tau_i) = eta n (forced H counted as 1).
    rng = np.random.default_rng(n + int(1 / eta))
    tau = _lognormal_tau(rng, n)
    nl = 512 if eta * n > 600 else 64
    pc = O.poissoncomp(tau, eta, 4, nl, seed=0)
    assert abs(float(pc["r32"].astype(np.float64).sum()) - eta * n) < 1e-6 * n
    # The exact (fp64) c meets the equation to rounding.
    f = _forced(n, 4, nl)
    exact = f.sum() + np.minimum(1.0, pc["c_exact"] * tau[~f].astype(np.float64)).sum()
    assert abs(exact - eta * n) < 1e-9 * n


def test_c_matches_independent_root_finder():
    # Brent's method on the piecewise-linear budget function finds the same root.
    rng = np.random.default_rng(3)
    for trial in range(20):
        n = int(rng.integers(20, 300))
        tau = _lognormal_tau(rng, n) if trial % 2 else rng.uniform(0.01, 1, n).astype(np.float32)
        n_sink, n_local = int(rng.integers(0, 4)), int(rng.integers(0, 8))
        f = _forced(n, n_sink, n_local)
        eta = float(rng.uniform((f.sum() + 1) / n, 0.9))
        pc = O.poissoncomp(tau, eta, n_sink, n_local, seed=trial)
        t = tau[~f].astype(np.float64)
        b = eta * n - f.sum()
        if b >= len(t):
            assert np.isinf(pc["c_exact"])
            continue
        root = brentq(lambda c: np.minimum(1.0, c * t).sum() - b, 0.0, 1.0 / t.min(),
                      xtol=1e-300, rtol=1e-15, maxiter=500)
        assert abs(pc["c_exact"] - root) <= 1e-12 * root


def test_no_saturation_closed_form():
    # When no token saturates, c = (eta n - |H_forced|) / sum(tau) exactly.
    rng = np.random.default_rng(5)
    n = 2000
    tau = rng.uniform(0.5, 1.0, n).astype(np.float32)
    pc = O.poissoncomp(tau, 0.1, 2, 10, seed=1)
    t = tau[2:n - 10].astype(np.float64)
    assert pc["c_exact"] == pytest.approx((0.1 * n - 12) / t.sum(), rel=1e-14)


def test_r_definition_H_and_L():
    rng = np.random.default_rng(11)
    n = 16384
    tau = _lognormal_tau(rng, n)
    pc = O.poissoncomp(tau, 1 / 16, 4, 512, seed=0)
    f = _forced(n, 4, 512)
    r = pc["r32"]
    assert np.all(r[f] == 1.0)
    # r is published as the float32 product fminf(1, float(c) * tau) (the decision precision).
    want = np.minimum(np.float32(1.0), (pc["c32"] * tau).astype(np.float32))
    assert np.array_equal(r[~f], want[~f])
    assert pc["c32"] == np.float32(pc["c_exact"])
    # H (r = 1) is always resident; L = 0 < r < 1.
    assert np.all(pc["resident"][r == 1.0])
    assert np.all(r > 0)
    # Some non-forced tokens saturate at this budget (lognormal tail), and they are in H.
    assert np.count_nonzero((r == 1.0) & ~f) > 0


def test_eta_one_keeps_everything():
    rng = np.random.default_rng(2)
    tau = _lognormal_tau(rng, 3000)
    pc = O.poissoncomp(tau, 1.0, 4, 64, seed=9)
    assert np.all(pc["r32"] == 1.0) and np.all(pc["resident"]) and pc["count"] == 3000


def test_sample_rule_matches_uniforms():
    # Z_i = [u_i < r_i] with u_i the 24-bit Philox uniform of (seed, seq, layer, head, i).
    rng = np.random.default_rng(12)
    n = 700
    tau = rng.uniform(0.001, 1, n).astype(np.float32)
    pc = O.poissoncomp(tau, 0.2, 3, 7, seed=77, seq=2, layer=4, head=6)
    u = np.array([O.uniform24(77, 2, 4, 6, i) for i in range(n)])
    assert np.array_equal(pc["resident"], u < pc["r32"].astype(np.float64))
    assert pc["count"] == int(pc["resident"].sum())


def test_inclusion_frequencies_and_sample_size():
    # Over many seeds each token's inclusion frequency matches r_i, and |S| has mean sum_L r and
    # variance sum_L r (1 - r) (independent Bernoulli draws).
    rng = np.random.default_rng(4)
    n = 200
    tau = rng.uniform(0.02, 1, n).astype(np.float32)
    M = 3000
    hits = np.zeros(n)
    sizes = []
    for s in range(M):
        pc = O.poissoncomp(tau, 0.25, 2, 4, seed=1000 + s)
        hits += pc["resident"]
        sizes.append(pc["count"])
    r = pc["r32"].astype(np.float64)
    sd = np.sqrt(r * (1 - r) / M)
    assert np.all(np.abs(hits / M - r) <= 5 * sd + 1e-12)
    Lm = r < 1
    mean, var = r[Lm].sum(), (r[Lm] * (1 - r[Lm])).sum()
    sizes = np.array(sizes) - (~Lm).sum()
    assert abs(sizes.mean() - mean) < 5 * np.sqrt(var / M)
    assert 0.85 * var < sizes.var() < 1.15 * var


def test_invalid_inputs():
    tau = np.full(100, 0.5, dtype=np.float32)
    bad = tau.copy()
    bad[50] = 0.0
    with pytest.raises(O.OracleError):
        O.poissoncomp(bad, 0.5, 2, 2, 0)
    bad[50] = 1.5
    with pytest.raises(O.OracleError):
        O.poissoncomp(bad, 0.5, 2, 2, 0)
    bad[50] = np.nan
    with pytest.raises(O.OracleError):
        O.poissoncomp(bad, 0.5, 2, 2, 0)
    # tau of forced tokens is ignored.
    ok = tau.copy()
    ok[0] = 0.0
    O.poissoncomp(ok, 0.5, 2, 2, 0)
    # Budget at or below the forced set.
    with pytest.raises(O.OracleError):
        O.poissoncomp(tau, 0.04, 2, 2, 0)
    with pytest.raises(O.OracleError):
        O.poissoncomp(tau, 0.03, 2, 2, 0)
