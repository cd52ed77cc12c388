"""Pins of the oracle's shortlist variant (only tokens of a per-KV-head shortlist may be fetched):
with every token a candidate it is the unrestricted certificate exactly; with a partial mask the
restricted order of Eq. (10) and eps-hat of every remaining set are recomputed set by set in
50-digit arithmetic; the shortlist itself is checked against its definition by brute force."""
import mpmath
import numpy as np
import pytest

import oracle as O
from tests.test_oracle_estimator import _eps_hat_mp, _small_problem


def test_all_candidates_is_the_plain_certificate():
    rng = np.random.default_rng(11)
    for _ in range(5):
        s, r, res = _small_problem(rng, n=200, n_h=8, spread=rng.uniform(0.5, 3))
        eps = float(rng.uniform(0.01, 0.2))
        a = O.certify(s, r, res, eps, 0.05)
        b = O.certify_cand(s, r, res, eps, 0.05, np.ones(200, bool))
        for k in ("certified", "k_star", "eps_L", "eps_final", "beta", "V", "b", "n_fetch"):
            assert a[k] == b[k], k
        assert np.array_equal(a["F"], b["F"]) and np.array_equal(a["order"], b["order"])
        assert np.array_equal(a["eps_k"], b["eps_k"]) and not b["exhausted"]


def test_restricted_order_brute_force():
    rng = np.random.default_rng(12)
    seen_exhausted = seen_met = False
    for trial in range(12):
        n = 40
        s, r, res = _small_problem(rng, n=n, n_h=5, spread=rng.uniform(1.0, 3.5))
        eps, delta = float(rng.uniform(0.005, 0.2)), 0.05
        Lset = [i for i in range(n) if r[i] < 1]
        cand = np.zeros(n, bool)
        cand[rng.choice(Lset, size=int(rng.integers(1, len(Lset))), replace=False)] = True
        c = O.certify_cand(s, r, res, eps, delta, cand)
        plain = O.certify(s, r, res, eps, delta)
        # the per-token terms do not depend on the mask
        assert np.array_equal(c["lam"], plain["lam"]) and np.array_equal(c["g"], plain["g"])
        w = np.exp(s - c["m"])
        l = mpmath.log(mpmath.mpf(2) / mpmath.mpf(delta))
        order = list(c["order"])
        assert sorted(order) == [i for i in Lset if cand[i]]
        gs = [c["g"][i] for i in order]
        assert all(x > y or (x == y and i < j)
                   for x, y, i, j in zip(gs, gs[1:], order, order[1:]))
        others = [i for i in Lset if not cand[i]]
        for k in range(len(order) + 1):
            ek = _eps_hat_mp(order[k:] + others, w, r, c["lam"], l, c["D"])
            assert float(ek) == pytest.approx(c["eps_k"][k], rel=1e-12, abs=1e-300)
        ek = c["eps_k"]
        if ek[0] < eps:
            want, exh = 0, False
        else:
            hit = [k for k in range(1, len(ek)) if ek[k] < eps]
            want, exh = (hit[0], False) if hit else (len(order), True)
        assert c["k_star"] == want and c["exhausted"] == exh
        F = np.zeros(n, bool)
        F[order[:want]] = True
        assert np.array_equal(c["F"], F) and not (F & ~cand).any()
        seen_exhausted |= exh
        seen_met |= (want > 0 and not exh)
    assert seen_exhausted and seen_met


def test_shortlist_definition():
    rng = np.random.default_rng(13)
    G, n = 4, 300
    s = rng.normal(0, 2, (G, n))
    s[1, 17] = s[0, 18] = s.max() + 1.0   # a tie in the key: the lower id comes first
    r = rng.uniform(0.1, 0.9, n).astype(np.float32)
    r[:10] = 1.0                            # H tokens are never shortlisted
    for size in (1, 2, 16, 128, 1000):
        m = O.shortlist(s, r, size)
        key = s.max(0)
        L = [i for i in range(n) if r[i] < 1]
        best = sorted(L, key=lambda i: (-key[i], i))[:size]
        assert set(np.nonzero(m)[0]) == set(best)
    assert O.shortlist(s, r, 1)[17] and not O.shortlist(s, r, 1)[18]
