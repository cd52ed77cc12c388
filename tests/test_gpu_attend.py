"""GPU KVFetch (certificate, selection, estimator, fetch and refine) against the fp64 oracle
under the tie-aware parity bar of tests/parity.py."""
import numpy as np
import pytest
import torch

from tests import parity as P
from verified_kv_cache_poissoncomp_gb300 import binding as B
from verified_kv_cache_poissoncomp_gb300 import inputs as I
from verified_kv_cache_poissoncomp_gb300.engine import default_cap

pytestmark = pytest.mark.gpu


def _run_all(w, queries=None, eps=None, fetch_mode=B.VERKV_FETCH_ZEROCOPY, cap=None):
    eng = P.make_engine(w, cap=cap, fetch_mode=fetch_mode)
    eng.compress(w.eta, w.n_sink, w.n_local, w.seed)
    eng.sync()
    pcs = P.oracle_poissoncomp(w)
    P.check_poissoncomp(eng, w, pcs)
    rep = None
    outs = []
    for t in (range(w.queries.shape[0]) if queries is None else queries):
        g = P.gpu_query(eng, w, t, eps=eps)
        units = P.oracle_query(w, t, pcs, eps=eps)
        rep = P.compare_query(g, units, w, eps=eps, report=rep)
        outs.append(g)
    print(rep)
    return rep, outs


def test_tiny_all_queries():
    rep, _ = _run_all(I.tiny())
    assert rep["exact_F"] >= 0.9 * rep["heads"]


def test_multi_cta_ragged():
    # n = 20000: three-CTA certify cluster, ragged last CTA; batch 2, two layers, 2 KV heads.
    w = I.make_workload("mid", B=2, L=2, h_kv=2, G=4, d=128, n=20000, n_queries=6, n_local=512)
    rep, _ = _run_all(w)
    assert rep["exact_F"] >= 0.9 * rep["heads"]


@pytest.mark.parametrize("G,d", [(1, 64), (2, 64), (8, 64), (2, 128), (8, 128)])
def test_gqa_and_head_dims(G, d):
    w = I.make_workload("gqa", B=1, L=1, h_kv=2, G=G, d=d, n=3000, eta=1 / 8, n_local=64,
                        n_queries=4, plant_every=2)
    rep, _ = _run_all(w)
    assert rep["exact_F"] >= 0.9 * rep["heads"]


def test_single_layer_32k_sampled_queries():
    # The benchmark's layer shape at full size: 8 KV heads x 4 query heads, d = 128, n = 32768,
    # eta = 1/16; plain and planted queries.
    w = I.single_layer_32k(layers=1, n_queries=8)
    rep, _ = _run_all(w, queries=[0, 1, 2, 3, 7])
    assert rep["exact_F"] >= 0.9 * rep["heads"]


def test_128k_context():
    w = I.make_workload("128k", B=1, L=1, h_kv=1, G=4, d=128, n=131072, eta=1 / 32,
                        n_queries=4, plant_every=2)
    rep, _ = _run_all(w)
    assert rep["exact_F"] >= 0.9 * rep["heads"]


def test_128k_needle_sets_stress_the_fetch():
    # The long-context workload's generator at reduced width: 128K tokens, eta = 1/32, a needle
    # set of 2-25 % of the context per KV head; the certificate must fetch much of it.
    w = I.long_context_128k(B=1, h_kv=2, n_queries=2)
    rep, outs = _run_all(w)
    assert rep["exact_F"] >= 0.9 * rep["heads"]
    fetched = np.array([o["counts"] for o in outs], dtype=np.float64) / w.n
    assert fetched.mean() > 0.01, fetched


def test_memcpy_mode_matches_zerocopy():
    w = I.make_workload("modes", B=1, L=1, h_kv=2, G=4, d=128, n=8192, eta=1 / 8, n_queries=4,
                        plant_every=2)
    _, a = _run_all(w)
    _, b = _run_all(w, fetch_mode=B.VERKV_FETCH_MEMCPY)
    for x, y in zip(a, b):
        assert np.array_equal(x["o"], y["o"]) and np.array_equal(x["F"], y["F"])
        assert np.array_equal(x["counts"], y["counts"])
        for ul, c in enumerate(x["counts"]):
            assert np.array_equal(x["ids"][ul, :c], y["ids"][ul, :c])


@pytest.mark.parametrize("G,d", [(4, 128), (8, 64)])
def test_staged_pivotal_sums_match_unstaged(G, d):
    # In MEMCPY mode the pivotal sums run in a kernel that bulk-copies each item's rows, ids and r
    # into shared memory when the capacity is a multiple of 4 (the default capacity is), else in
    # one that reads them from global memory; both must give the same bits and match the oracle.
    w = I.make_workload("staged", B=2, L=1, h_kv=2, G=G, d=d, n=8192, eta=1 / 8, n_queries=3,
                        plant_every=2)
    cap = default_cap(w.n, w.eta)
    assert cap % 4 == 0
    _, a = _run_all(w, fetch_mode=B.VERKV_FETCH_MEMCPY, cap=cap)
    _, b = _run_all(w, fetch_mode=B.VERKV_FETCH_MEMCPY, cap=cap + 1)
    for x, y in zip(a, b):
        assert np.array_equal(x["o"], y["o"]) and np.array_equal(x["lse"], y["lse"])


def test_fetching_keys_too_matches_values_only():
    # With the exact sketch the fetch moves only V rows by default; moving full K|V rows must give
    # bitwise the same results, in both fetch modes.
    w = I.make_workload("keys", B=1, L=2, h_kv=2, G=4, d=128, n=8192, eta=1 / 8, n_queries=4,
                        plant_every=2)
    _, a = _run_all(w)
    _, b = _run_all(w, fetch_mode=B.VERKV_FETCH_ZEROCOPY | B.VERKV_FETCH_KEYS)
    _, c = _run_all(w, fetch_mode=B.VERKV_FETCH_MEMCPY | B.VERKV_FETCH_KEYS)
    for x, y, z in zip(a, b, c):
        assert np.array_equal(x["o"], y["o"]) and np.array_equal(x["o"], z["o"])
        assert np.array_equal(x["lse"], y["lse"]) and np.array_equal(x["lse"], z["lse"])


def test_eta_one_is_dense_attention():
    import oracle as O
    w = I.make_workload("dense", B=1, L=1, h_kv=2, G=4, d=128, n=2048, eta=1.0, n_local=64,
                        n_queries=2)
    eng = P.make_engine(w, cap=2048)
    eng.compress(w.eta, w.n_sink, w.n_local, w.seed)
    for t in range(2):
        g = P.gpu_query(eng, w, t)
        assert np.all(g["stats"]["certified"] == 1) and np.all(g["stats"]["n_L"] == 0)
        for h in range(w.h_kv):
            K = O.bf16_to_f64(w.kv[0, 0, h, :, 0, :])
            V = O.bf16_to_f64(w.kv[0, 0, h, :, 1, :])
            for gi in range(w.G):
                q = O.bf16_to_f64(w.queries[t, 0, h * w.G + gi])
                dn = O.dense(O.logits(q, K), V)
                qh = h * w.G + gi
                assert np.linalg.norm(g["o"][qh] - dn["o"]) <= 1e-4 * np.linalg.norm(dn["o"])
                assert abs(g["lse"][qh] - (dn["m"] + np.log(dn["D"]))) <= 1e-4


def test_tiny_tolerance_fetches_all_of_L():
    import oracle as O
    w = I.tiny()
    eng = P.make_engine(w)
    eng.compress(w.eta, w.n_sink, w.n_local, w.seed)
    K = O.bf16_to_f64(w.kv[0, 0, 0, :, 0, :])
    V = O.bf16_to_f64(w.kv[0, 0, 0, :, 1, :])
    g = P.gpu_query(eng, w, 0, eps=1e-30)
    for gi in range(w.G):
        dn = O.dense(O.logits(O.bf16_to_f64(w.queries[0, 0, gi]), K), V)
        assert np.linalg.norm(g["o"][gi] - dn["o"]) <= 1e-4 * np.linalg.norm(dn["o"])


def test_without_fetch_outputs_matches_with_them():
    # A caller that asks for neither fetch ids nor counts gets no fetch list from the certify
    # kernel; the refine reads the selection bitmaps either way, so o, lse and the per-head
    # statistics (n_fetch included) must be the same bits as with the outputs requested.
    w = I.make_workload("nolist", B=2, L=2, h_kv=2, G=4, d=128, n=20000, eta=1 / 8, n_queries=4,
                        plant_every=2)
    eng = P.make_engine(w)
    eng.compress(w.eta, w.n_sink, w.n_local, w.seed)
    eng.sync()
    uncertified = 0
    for t in range(w.queries.shape[0]):
        q = torch.as_tensor(w.queries[t].view(np.int16)).to(eng.dev)
        out = []
        for with_ids in (True, False):
            eng.attend(int(w.query_layer[t]), q, w.eps, w.delta, with_ids=with_ids)
            o, lse, st = eng.fetch_refine()
            eng.sync()
            out.append((o.cpu().numpy().copy(), lse.cpu().numpy().copy(), st.cpu().numpy().copy()))
        (o1, l1, s1), (o2, l2, s2) = out
        assert np.array_equal(o1, o2) and np.array_equal(l1, l2) and np.array_equal(s1, s2), t
        uncertified += int((s1[:, 10] == 0).sum())
    assert uncertified > 0  # the selection and the fetch ran
    eng.close()


@pytest.mark.parametrize("n,G,d", [(40, 4, 128), (64, 4, 128), (65, 4, 128), (200, 4, 128),
                                   (1000, 4, 128), (40, 8, 64), (65, 8, 64)])
def test_short_and_ragged_contexts(n, G, d):
    # Contexts shorter than one 64-row scoring stage or a stage and a row: the scoring kernel's
    # tensor copies read past the unit's last row (zero fill, not stored), the certificate runs in
    # one CTA with a partly filled last warp, and the refine's single token range is ragged.
    w = I.make_workload("short", B=1, L=1, h_kv=2, G=G, d=d, n=n, eta=1 / 2, n_local=8,
                        n_queries=4, plant_every=2)
    rep, outs = _run_all(w)
    assert rep["exact_F"] >= 0.9 * rep["heads"]
    assert all(np.isfinite(o["o"]).all() and np.isfinite(o["lse"]).all() for o in outs)
