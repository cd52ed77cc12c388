"""Pins for the oracle's estimator, certificate and selection ("Verify Before You Fetch", summary
page: Definition 2 / Eq. (5), Theorem 1 / Eq. (6), Lemma 1 / Eq. (7), KVFETCH Eqs. (9)-(10),
Theorem 2) and for its dense SDPA."""
import itertools

import mpmath
import numpy as np
import pytest
import torch
from scipy.optimize import minimize

import oracle as O
from verified_kv_cache_poissoncomp_gb300 import inputs as I


def _small_problem(rng, n=24, n_h=4, spread=2.0):
    s = rng.normal(0.0, spread, n)
    r = rng.uniform(0.05, 0.95, n).astype(np.float32)
    r[:n_h] = 1.0
    res = np.zeros(n, dtype=np.uint8)
    res[:n_h] = 1
    return s, r, res


# ------------------------------------------------------------------------------------------------
def test_dense_matches_torch_sdpa_fp64():
    rng = np.random.default_rng(0)
    n, d = 300, 64
    q = rng.standard_normal(d)
    K = rng.standard_normal((n, d)) * 1.5
    V = rng.standard_normal((n, d))
    dn = O.dense(O.logits(q, K), V)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.tensor(q)[None, None, None], torch.tensor(K)[None, None], torch.tensor(V)[None, None])
    np.testing.assert_allclose(dn["o"], ref[0, 0, 0].numpy(), rtol=1e-12, atol=1e-13)
    # Brute force by the definition, with logsumexp from mpmath.
    s = [mpmath.fdot(map(mpmath.mpf, q), map(mpmath.mpf, K[i])) / mpmath.sqrt(d)
         for i in range(n)]
    lse = mpmath.log(mpmath.fsum(mpmath.exp(x) for x in s))
    assert float(lse) == pytest.approx(dn["m"] + np.log(dn["D"]), rel=1e-13)


# ------------------------------------------------------------------------------------------------
def test_beta_is_the_fixed_point():
    # Definition 2: beta = sum_L w_i (1 - lambda_i) with lambda_i = clip(beta r / (w (1-r)), r, 1).
    rng = np.random.default_rng(1)
    for trial in range(30):
        s, r, res = _small_problem(rng, n=int(rng.integers(5, 200)), spread=rng.uniform(0.1, 6))
        c = O.certify(s, r, res, 0.05, 0.05)
        w = np.exp(s - s.max())
        L = r < 1
        r = r.astype(np.float64)
        lam_want = np.clip(c["beta"] * r[L] / (w[L] * (1 - r[L])), r[L], 1.0)
        np.testing.assert_allclose(c["lam"][L], lam_want, rtol=1e-9, atol=1e-14)
        assert c["beta"] == pytest.approx((w[L] * (1 - c["lam"][L])).sum(), rel=1e-10, abs=1e-300)


def test_theorem1_lambda_minimises_mse():
    # Theorem 1 / Eq. (6): the estimator's lambda is the unique minimiser over [r, 1]^L of
    # (sum_L w (1 - lambda))^2 + sum_L lambda^2 w^2 (1 - r) / r.  Solve that box QP by brute force.
    rng = np.random.default_rng(2)
    for trial in range(15):
        n = int(rng.integers(3, 20))
        s, r, res = _small_problem(rng, n=n + 2, n_h=2, spread=rng.uniform(0.2, 3))
        c = O.certify(s, r, res, 0.05, 0.05)
        w = np.exp(s - s.max())
        L = r < 1
        wl, rl = w[L], r[L].astype(np.float64)

        def mse(lam):
            bias = (wl * (1 - lam)).sum()
            return bias * bias + (lam * lam * wl * wl * (1 - rl) / rl).sum()

        def grad(lam):
            bias = (wl * (1 - lam)).sum()
            return -2 * bias * wl + 2 * lam * wl * wl * (1 - rl) / rl

        best = None
        for start in [rl.copy(), np.ones_like(rl), 0.5 * (rl + 1)]:
            opt = minimize(mse, start, jac=grad, method="L-BFGS-B",
                           bounds=list(zip(rl, np.ones_like(rl))),
                           options=dict(ftol=1e-16, gtol=1e-14, maxiter=10000))
            if best is None or opt.fun < best.fun:
                best = opt
        assert mse(c["lam"][L]) <= best.fun * (1 + 1e-9) + 1e-300
        np.testing.assert_allclose(c["lam"][L], best.x, atol=2e-5)


def test_estimator_exact_mean_and_variance_by_enumeration():
    # Eq. (5) with independent Z_i ~ Bernoulli(r_i): enumerate every outcome of Z on a small L;
    # E[D-hat] = D - beta(L) and Var[D-hat] = V(L) exactly (the quantities of Eq. (7)).
    rng = np.random.default_rng(3)
    n, d = 14, 3
    s, r, _ = _small_problem(rng, n=n, n_h=3, spread=1.5)
    values = rng.standard_normal((n, d))
    none = np.zeros(n, dtype=np.uint8)
    c = O.certify(s, r, np.ones(n, np.uint8), 0.05, 0.05)
    w = np.exp(s - c["m"])
    Lidx = np.nonzero(r < 1)[0]
    mean = var2 = 0.0
    meanN = np.zeros(d)
    for bits in itertools.product([0, 1], repeat=len(Lidx)):
        res = np.ones(n, dtype=np.uint8)
        res[Lidx] = bits
        p = np.prod([float(r[i]) if z else 1.0 - float(r[i]) for i, z in zip(Lidx, bits)])
        est = O.refine(s, values, r, res, none, c["lam"], c["m"])
        mean += p * est["D_hat"]
        var2 += p * est["D_hat"] ** 2
        meanN += p * est["N_hat"]
    D = w.sum()
    assert mean == pytest.approx(D - c["beta"], rel=1e-12)
    assert var2 - mean ** 2 == pytest.approx(c["V"], rel=1e-8)
    # N-hat applies the same weights to w_i v_i.
    lam = c["lam"]
    np.testing.assert_allclose(meanN, (lam[:, None] * w[:, None] * values).sum(0), rtol=1e-10)


def test_lemma1_b_is_the_largest_summand_deviation():
    # Lemma 1 / Eq. (7) applies Bernstein's inequality to D-hat = sum_H w + sum_L X_i with
    # independent summands X_i = Z_i lambda_i w_i / r_i; b(L) must be the bound on every summand's
    # deviation from its mean, max_i max_{Z_i in {0, 1}} |X_i - E X_i|.  Each X_i is read off the
    # oracle's own estimator by enumerating Z_i for one token at a time (the others unsampled), so
    # b is pinned to what D-hat computes, not to a second copy of its formula.  The draws put r on
    # both sides of 1/2, where the larger deviation switches between Z_i = 0 and Z_i = 1.
    rng = np.random.default_rng(11)
    for trial in range(12):
        n, d = int(rng.integers(6, 40)), 2
        s, r, res_h = _small_problem(rng, n=n, n_h=3, spread=rng.uniform(0.3, 4.0))
        values = rng.standard_normal((n, d))
        c = O.certify(s, r, res_h, 0.05, 0.05)
        none = np.zeros(n, dtype=np.uint8)
        base = O.refine(s, values, r, res_h, none, c["lam"], c["m"])["D_hat"]
        b = 0.0
        for i in np.nonzero(r < 1)[0]:
            res = res_h.copy()
            res[i] = 1
            x1 = O.refine(s, values, r, res, none, c["lam"], c["m"])["D_hat"] - base  # Z_i = 1
            mean = float(r[i]) * x1                                                  # E X_i
            b = max(b, abs(x1 - mean), abs(0.0 - mean))
        assert (r[r < 1] > 0.5).any() and (r[r < 1] < 0.5).any()
        assert c["b"] == pytest.approx(b, rel=1e-10, abs=1e-300)


def _eps_hat_mp(idx, w, r, lam, l, D):
    """eps_hat of the subset idx of L from Eq. (7) with lambda held fixed, in 50-digit arithmetic."""
    w = [float(x) for x in w]
    r = [float(x) for x in r]
    lam = [float(x) for x in lam]
    with mpmath.workdps(50):
        beta = mpmath.fsum(mpmath.mpf(w[i]) * (1 - mpmath.mpf(lam[i])) for i in idx)
        V = mpmath.fsum(mpmath.mpf(lam[i]) ** 2 * mpmath.mpf(w[i]) ** 2 * (1 - mpmath.mpf(r[i]))
                        / mpmath.mpf(r[i]) for i in idx)
        b = max([mpmath.mpf(lam[i]) * mpmath.mpf(w[i]) / mpmath.mpf(r[i]) *
                 max(mpmath.mpf(r[i]), 1 - mpmath.mpf(r[i])) for i in idx] or [mpmath.mpf(0)])
        a = b * l / 3
        return (beta + a + mpmath.sqrt(a * a + 2 * V * l)) / mpmath.mpf(D)


def test_certificate_g_and_kstar_brute_force():
    # Lemma 1 / Eq. (7), Eq. (9) and Eq. (10) recomputed set by set in 50-digit arithmetic.
    rng = np.random.default_rng(4)
    for trial in range(6):
        n = 40
        s, r, res = _small_problem(rng, n=n, n_h=5, spread=rng.uniform(0.5, 3))
        eps, delta = float(rng.uniform(0.02, 0.3)), 0.05
        c = O.certify(s, r, res, eps, delta)
        w = np.exp(s - c["m"])
        l = mpmath.log(mpmath.mpf(2) / mpmath.mpf(delta))
        Lset = [i for i in range(n) if r[i] < 1]
        full = _eps_hat_mp(Lset, w, r, c["lam"], l, c["D"])
        assert float(full) == pytest.approx(c["eps_L"], rel=1e-12)
        for i in Lset:
            gi = full - _eps_hat_mp([j for j in Lset if j != i], w, r, c["lam"], l, c["D"])
            assert float(gi) == pytest.approx(c["g"][i], rel=1e-9, abs=1e-15)
        order = list(c["order"])
        assert sorted(order) == Lset
        gs = [c["g"][i] for i in order]
        assert all(a >= b for a, b in zip(gs, gs[1:]))
        for k in range(len(order) + 1):
            ek = _eps_hat_mp(order[k:], w, r, c["lam"], l, c["D"])
            assert float(ek) == pytest.approx(c["eps_k"][k], rel=1e-12, abs=1e-300)
        ek = c["eps_k"]
        assert np.all(np.diff(ek) <= 1e-15)
        assert ek[-1] == 0.0
        want = 0 if ek[0] < eps else next(k for k in range(1, len(ek)) if ek[k] < eps)
        assert c["k_star"] == want
        assert c["certified"] == (want == 0)
        F = np.zeros(n, bool)
        F[order[:want]] = True
        assert np.array_equal(c["F"], F)


def test_shift_invariance_and_tie_break():
    rng = np.random.default_rng(5)
    s, r, res = _small_problem(rng, n=60, n_h=4, spread=2.5)
    a = O.certify(s, r, res, 0.03, 0.05)
    b = O.certify(s + 7.25, r, res, 0.03, 0.05)
    np.testing.assert_allclose(a["lam"], b["lam"], rtol=1e-12)
    assert a["eps_L"] == pytest.approx(b["eps_L"], rel=1e-12)
    assert np.array_equal(a["F"], b["F"]) and a["k_star"] == b["k_star"]
    # Duplicate tokens (same logit and r) tie in g; the lower id comes first.
    s2 = np.concatenate([s, s[10:12]])
    r2 = np.concatenate([r, r[10:12]])
    res2 = np.concatenate([res, res[10:12]])
    c = O.certify(s2, r2, res2, 0.03, 0.05)
    pos = {int(t): k for k, t in enumerate(c["order"])}
    assert pos[10] < pos[60] and pos[11] < pos[61]


def test_eta_one_and_fetch_all_are_exact():
    rng = np.random.default_rng(6)
    n, d = 500, 16
    s = rng.normal(0, 2, n)
    V = rng.standard_normal((n, d))
    dn = O.dense(s, V)
    # eta = 1: every token in H -> L empty, eps_hat = 0, D-hat = D and N-hat = N exactly.
    r1 = np.ones(n, np.float32)
    c = O.certify(s, r1, np.ones(n, np.uint8), 0.05, 0.05)
    assert c["certified"] and c["eps_L"] == 0.0 and c["n_L"] == 0
    est = O.refine(s, V, r1, np.ones(n, np.uint8), c["F"], c["lam"], c["m"])
    assert est["D_hat"] == pytest.approx(dn["D"], rel=1e-14)
    np.testing.assert_allclose(est["N_hat"], dn["N"], rtol=1e-12, atol=1e-12)
    # A tolerance below every nonzero eps_hat(k) fetches all of L: again exact.
    r = rng.uniform(0.01, 0.9, n).astype(np.float32)
    res = (rng.uniform(size=n) < r).astype(np.uint8)
    c = O.certify(s, r, res, 1e-300, 0.05)
    assert c["k_star"] == c["n_L"] == n and c["F"].all()
    est = O.refine(s, V, r, res, c["F"], c["lam"], c["m"])
    assert est["D_hat"] == pytest.approx(dn["D"], rel=1e-13)
    np.testing.assert_allclose(est["o"], dn["o"], rtol=1e-11, atol=1e-12)


@pytest.mark.slow
def test_theorem2_monte_carlo_and_unbiasedness():
    # Theorem 2 (exact sketch, fixed query, Poisson sampling): the returned estimator's relative
    # error on D exceeds eps with probability at most delta.  Also: the MC mean of D-hat is
    # D - beta(L') and the MC mean of M2 is V(L') for the remaining set L'.
    w_ = I.tiny()
    K = O.bf16_to_f64(w_.kv[0, 0, 0, :, 0, :])
    V = O.bf16_to_f64(w_.kv[0, 0, 0, :, 1, :])
    pc0 = O.poissoncomp(w_.tau[0, 0, 0], w_.eta, w_.n_sink, w_.n_local, 0)
    M = 2000
    seeds_res = [O.poissoncomp(w_.tau[0, 0, 0], w_.eta, w_.n_sink, w_.n_local, 5000 + k)["resident"]
                 for k in range(M)]
    fail_total = trials = 0
    for qi in [0, 1, 2, 3]:
        q = O.bf16_to_f64(w_.queries[qi, 0, 0])
        s = O.logits(q, K)
        dn = O.dense(s, V)
        c = O.certify(s, pc0["r32"], pc0["resident"], w_.eps, w_.delta)
        w = np.exp(s - c["m"])
        Lp = (pc0["r32"] < 1) & ~c["F"]
        r = pc0["r32"].astype(np.float64)
        bias = (w[Lp] * (1 - c["lam"][Lp])).sum()
        var = (c["lam"][Lp] ** 2 * w[Lp] ** 2 * (1 - r[Lp]) / r[Lp]).sum()
        Dh = np.empty(M)
        M2 = np.empty(M)
        for k in range(M):
            est = O.refine(s, V, pc0["r32"], seeds_res[k], c["F"], c["lam"], c["m"])
            Dh[k] = est["D_hat"]
            M2[k] = est["M2"]
        D = dn["D"] / np.exp(c["m"] - dn["m"])
        assert abs(Dh.mean() - (D - bias)) < 4.5 * np.sqrt(var / M) + 1e-12 * D
        if var > 0:
            assert abs(M2.mean() - var) < 6 * M2.std() / np.sqrt(M) + 1e-12
        fail_total += int((np.abs(Dh - D) / D > w_.eps).sum())
        trials += M
    p = fail_total / trials
    assert p <= w_.delta + 3 * np.sqrt(w_.delta * (1 - w_.delta) / trials)
