"""GPU-vs-oracle parity harness: runs a seeded workload through libverkv (via the engine, i.e. the
C ABI) and through the fp64 oracle, and compares them element by element.

Tolerances (float32 logits carry up to ~1.5e-5 relative error into w-hat -- bf16 products are
exact in fp32, twelve roundings per dot product -- and g inherits about twice that):
  * PoissonComp: c32, r, the resident bitmap, pivotal ids / r / rows -- bit-exact.
  * Certificate decision: may differ only when the oracle's eps-hat(L) lies within EPS_TIE = 1e-5
    relative of eps (the stated bar).
  * k*: must lie in the oracle's acceptable set {k : eps_o(k) < eps (1 + EPS_TIE) and
    (k = 0 or eps_o(k-1) >= eps (1 - EPS_TIE))} along the oracle's order.
  * F: equal to the oracle's top-k* set, except for swaps among tokens whose oracle g lies within
    G_TIE = 1e-5 relative of g at the cut, the same window as the decision's.  (float32 logits
    carry up to ~1.5e-5 relative error into w-hat in the worst case, but over the whole GPU suite
    -- 1440 query heads at 1K to 128K tokens -- no swap occurred at all: the run reports
    tie_F = 0 and max_g_gap = 0 in its parity summary line.)
  * D-hat, N-hat, o: error <= 1e-3 (bf16 storage, fp32 accumulation) -- |lse - lse_o| for D-hat,
    and max_c |x_c - x_o,c| / max_c |x_o,c| element by element for N-hat and o -- on every head:
    against the oracle's estimator when the GPU's F equals the oracle's, else against the oracle's
    refine() for the GPU's F (a near-tie swap changes which estimator is returned, not whether it
    is computed right).
"""
import numpy as np
import torch

import oracle as O
from verified_kv_cache_poissoncomp_gb300 import binding as B
from verified_kv_cache_poissoncomp_gb300.engine import VerKV, default_cap, stats_to_dict

EPS_TIE = 1e-5
G_TIE = 1e-5
EST_TOL = 1e-3


def bits_to_bool(words, n):
    w = np.ascontiguousarray(words).view(np.uint32)
    bits = ((w[..., None] >> np.arange(32, dtype=np.uint32)) & 1).astype(bool)
    return bits.reshape(*w.shape[:-1], -1)[..., :n]


# ------------------------------------------------------------------------------------------------
def make_engine(w, cap=None, fetch_mode=B.VERKV_FETCH_ZEROCOPY, sketch_format=B.VERKV_SKETCH_EXACT):
    cap = cap or default_cap(w.n, w.eta)
    eng = VerKV(w.B, w.L, w.h_kv, w.G, w.d, w.n, cap, fetch_mode=fetch_mode,
                sketch_format=sketch_format)
    eng.load(w.tau.reshape(-1, w.n), w.kv.reshape(-1, w.n, 2, w.d))
    return eng


def oracle_poissoncomp(w):
    out = {}
    for b in range(w.B):
        for l in range(w.L):
            for h in range(w.h_kv):
                out[(b, l, h)] = O.poissoncomp(w.tau[b, l, h], w.eta, w.n_sink, w.n_local,
                                               w.seed, b, l, h)
    return out


def check_poissoncomp(eng, w, pcs):
    """Bit-exact comparison of the pivotal set against the oracle."""
    torch.cuda.synchronize()
    r = eng.r_full.cpu().numpy()
    res = bits_to_bool(eng.p_res.cpu().numpy(), w.n)
    ids = eng.p_ids.cpu().numpy()
    pr = eng.p_r.cpu().numpy()
    cnt = eng.p_count.cpu().numpy()
    c = eng.p_c.cpu().numpy()
    pkv = eng.p_kv.cpu().numpy().view(np.uint16)
    u = 0
    for b in range(w.B):
        for l in range(w.L):
            for h in range(w.h_kv):
                o = pcs[(b, l, h)]
                assert np.float32(c[u]) == o["c32"], (u, c[u], o["c32"])
                assert np.array_equal(r[u], o["r32"]), u
                assert np.array_equal(res[u], o["resident"]), u
                want = np.nonzero(o["resident"])[0]
                assert cnt[u] == len(want) == o["count"], (u, cnt[u], len(want))
                assert np.array_equal(ids[u, :cnt[u]], want), u
                assert np.array_equal(pr[u, :cnt[u]], o["r32"][want]), u
                assert np.array_equal(pkv[u, :cnt[u]], w.kv[b, l, h][want]), u
                u += 1


# ------------------------------------------------------------------------------------------------
def gpu_query(eng, w, t, eps=None, delta=None):
    eps = w.eps if eps is None else eps
    delta = w.delta if delta is None else delta
    q = torch.as_tensor(w.queries[t].view(np.int16)).to(eng.dev)
    eng.attend(int(w.query_layer[t]), q, eps, delta)
    F = eng.selection_bitmap()
    o, lse, stats = eng.fetch_refine()
    eng.sync()
    return dict(o=o.cpu().numpy().copy(), lse=lse.cpu().numpy().copy(),
                stats=stats_to_dict(stats), F=bits_to_bool(F.cpu().numpy(), w.n),
                ids=eng.fetch_ids.cpu().numpy().copy(), counts=eng.fetch_counts.cpu().numpy().copy())


def oracle_query(w, t, pcs, eps=None, delta=None, sketches=None, cands=None):
    """sketches: None for the exact sketch, else {(b, l, h): dequantised sketch keys}.
    cands: None, or {(b, h): bool mask} of fetch candidates (the shortlist variant)."""
    eps = w.eps if eps is None else eps
    delta = w.delta if delta is None else delta
    l = int(w.query_layer[t])
    units = []
    for b in range(w.B):
        for h in range(w.h_kv):
            pc = pcs[(b, l, h)]
            K = O.bf16_to_f64(w.kv[b, l, h, :, 0, :])
            V = O.bf16_to_f64(w.kv[b, l, h, :, 1, :])
            Ks = K if sketches is None else sketches[(b, l, h)]
            qs = O.bf16_to_f64(w.queries[t, b, h * w.G:(h + 1) * w.G])
            cm = None if cands is None else cands[(b, h)]
            units.append(O.attend_unit(qs, Ks, K, V, pc["r32"], pc["resident"], eps, delta,
                                       cand=cm))
    return units


def oracle_q2_sketches(w):
    """The oracle's 2-bit sketch of every unit: {(b, l, h): (rows uint8, dequantised keys)}."""
    return {(b, l, h): O.q2_sketch(w.kv[b, l, h, :, 0, :])
            for b in range(w.B) for l in range(w.L) for h in range(w.h_kv)}


def _check_estimator(g, qh, st, est, rep):
    """D-hat (through lse), N-hat and o of query head qh against one oracle refine() result:
    |lse - lse_o| <= EST_TOL, and for o and N-hat the largest element error relative to the
    largest element, max_c |x_c - x_o,c| / max_c |x_o,c| <= EST_TOL."""
    dl = abs(float(g["lse"][qh]) - est["lse"])
    rep["max_lse"] = max(rep["max_lse"], dl)
    assert dl <= EST_TOL, (qh, float(g["lse"][qh]), est["lse"])
    o_g = np.asarray(g["o"][qh], dtype=np.float64)
    oe = np.max(np.abs(o_g - est["o"])) / max(np.max(np.abs(est["o"])), 1e-300)
    rep["max_o"] = max(rep["max_o"], oe)
    assert oe <= EST_TOL, (qh, oe)
    # N-hat with the oracle's shift: D-hat_gpu exp(m_gpu - m_o) o_gpu = exp(lse_gpu - m_o) o_gpu
    n_g = np.exp(float(g["lse"][qh]) - est["m"]) * o_g
    ne = np.max(np.abs(n_g - est["N_hat"])) / max(np.max(np.abs(est["N_hat"])), 1e-300)
    rep["max_N"] = max(rep["max_N"], ne)
    assert ne <= EST_TOL, (qh, ne)
    rep["est_checked"] += 1


def new_report():
    return dict(heads=0, exact_F=0, tie_F=0, tie_decision=0, est_checked=0, max_lse=0.0,
                max_o=0.0, max_N=0.0, max_eps_rel=0.0, max_beta_rel=0.0, max_g_gap=0.0,
                max_decision_gap=0.0)


# Counters over every compare_query call of the process (printed at the end of a pytest run).
SUITE = new_report()


def _add_to_suite(rep_before, rep):
    for k, v in rep.items():
        if k.startswith("max_"):
            SUITE[k] = max(SUITE[k], v)
        else:
            SUITE[k] += v - rep_before.get(k, 0)


def compare_query(g, units, w, eps=None, report=None):
    """Asserts the tie-aware parity bar for one query; returns counters.

    Every head's estimator is checked: against the oracle's own result when the GPU's F equals
    the oracle's, else against the oracle's refine() re-run with the GPU's F (and the oracle's
    lambda), so a tie-swapped F or a decision inside the tie window still gets D-hat, N-hat and o
    held to EST_TOL.  max_g_gap records the largest relative g gap between a swapped token and
    the cut, max_decision_gap the largest |eps-hat(L) - eps| / eps of a decision that differs."""
    eps = w.eps if eps is None else eps
    rep = report if report is not None else new_report()
    for k, v in new_report().items():
        rep.setdefault(k, v)
    before = dict(rep)
    st = g["stats"]
    for ul, unit in enumerate(units):
        unit_exact = True
        tie_tokens = set()
        res = np.asarray(unit["resident"], dtype=bool)
        for gi, hd in enumerate(unit["heads"]):
            qh = ul * w.G + gi
            cert, est = hd["cert"], hd["est"]
            rep["heads"] += 1
            gcert = bool(st["certified"][qh])
            Fg = g["F"][qh]
            # eps-hat and beta
            e_rel = abs(float(st["eps_hat"][qh]) - cert["eps_L"]) / max(cert["eps_L"], 1e-30)
            rep["max_eps_rel"] = max(rep["max_eps_rel"], e_rel)
            if cert["beta"] > 0:
                b_rel = abs(float(st["beta"][qh]) * np.exp(float(st["m"][qh]) - cert["m"]) -
                            cert["beta"]) / cert["beta"]
                rep["max_beta_rel"] = max(rep["max_beta_rel"], b_rel)
            assert st["n_L"][qh] == cert["n_L"], (qh, st["n_L"][qh], cert["n_L"])
            if gcert != cert["certified"]:
                gap = abs(cert["eps_L"] - eps) / eps
                rep["max_decision_gap"] = max(rep["max_decision_gap"], gap)
                assert gap <= EPS_TIE, (qh, gcert, cert["eps_L"], float(st["eps_hat"][qh]))
                rep["tie_decision"] += 1
                unit_exact = False
                tie_tokens |= set(np.nonzero(Fg | cert["F"])[0].tolist())
            else:
                k = int(st["k_star"][qh])
                assert int(Fg.sum()) == k, (qh, int(Fg.sum()), k)
                ek = cert["eps_k"]
                gexh = bool(st["flags"][qh] & 4)
                if not gcert and (gexh or cert.get("exhausted")):
                    # shortlist variant: the whole shortlist taken without meeting eps on one side
                    # is allowed only within the tie window on the other
                    nc = len(cert["order"])
                    if gexh:
                        assert k == nc and ek[nc] >= eps * (1 - EPS_TIE), (qh, k, nc, ek[nc])
                    else:
                        assert k >= 1 and ek[k] < eps * (1 + EPS_TIE), (qh, k, ek[k])
                elif not gcert:
                    assert k >= 1 and ek[k] < eps * (1 + EPS_TIE) and \
                        ek[k - 1] >= eps * (1 - EPS_TIE), \
                        (qh, k, cert["k_star"], ek[max(k - 1, 0)], ek[k])
                else:
                    assert k == 0 and not Fg.any()
                if not np.array_equal(Fg, cert["F"]):
                    rep["tie_F"] += 1
                    unit_exact = False
                    order = cert["order"]
                    gv = cert["g"]
                    top = np.zeros(w.n, dtype=bool)
                    top[order[:k]] = True
                    diff = np.nonzero(Fg ^ top)[0]
                    gb = gv[order[k - 1]] if k >= 1 else gv[order[0]]
                    for tok in diff:
                        gap = abs(gv[tok] - gb) / gb
                        rep["max_g_gap"] = max(rep["max_g_gap"], gap)
                        assert gap <= G_TIE, (qh, int(tok), gv[tok], gb)
                    # k* may differ from the oracle's inside the acceptable set: the boundary
                    # tokens then differ too, and may change the per-KV-head union.
                    tie_tokens |= set(np.nonzero(Fg ^ cert["F"])[0].tolist())
            # The estimator the GPU returned, for the F it chose.
            if np.array_equal(Fg, cert["F"]):
                rep["exact_F"] += int(gcert == cert["certified"])
                assert st["n_fetch"][qh] == cert["n_fetch"]
                _check_estimator(g, qh, st, dict(est, m=cert["m"]), rep)
            else:
                assert st["n_fetch"][qh] == int(np.count_nonzero(Fg & ~res)), qh
                est_g = O.refine(hd["s"], unit["values"], unit["r32"], res, Fg, cert["lam"],
                                 cert["m"])
                _check_estimator(g, qh, st, dict(est_g, m=cert["m"]), rep)
        got = set(g["ids"][ul, :g["counts"][ul]].tolist())
        want = set(unit["fetch_ids"].tolist())
        assert list(g["ids"][ul, :g["counts"][ul]]) == sorted(got)
        if unit_exact:
            assert got == want, (ul, len(got), len(want))
        else:
            assert (got ^ want) <= tie_tokens, (ul, sorted(got ^ want)[:10])
    _add_to_suite(before, rep)
    return rep
