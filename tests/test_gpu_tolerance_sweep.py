"""Tolerance sweep on the GPU: eps-hat(L) and the g order do not depend on eps, so raising eps can
only certify more query heads and shrink k* (Eq. (10) takes the first k with eps-hat < eps)."""
import numpy as np
import pytest
import torch

from tests import parity as P
from verified_kv_cache_poissoncomp_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def test_kstar_and_fetches_are_monotone_in_eps():
    w = I.make_workload("sweep", B=1, L=1, h_kv=2, G=4, d=128, n=8192, eta=1 / 16, n_queries=6,
                        plant_every=2, n_local=256)
    eng = P.make_engine(w)
    eng.compress(w.eta, w.n_sink, w.n_local, w.seed)
    eng.sync()
    pcs = P.oracle_poissoncomp(w)
    prev = None
    for eps in [0.01, 0.03, 0.1, 0.3, 1.0]:
        ks, cert, counts = [], [], []
        for t in range(w.queries.shape[0]):
            g = P.gpu_query(eng, w, t, eps=eps)
            ks.append(g["stats"]["k_star"])
            cert.append(g["stats"]["certified"])
            counts.append(g["counts"])
        ks, cert, counts = np.array(ks), np.array(cert), np.array(counts)
        if prev is not None:
            pk, pc, pn = prev
            assert np.all(ks <= pk), eps
            assert np.all(cert >= pc), eps
            assert np.all(counts <= pn), eps
        prev = (ks, cert, counts)
    # the extremes differ: the sweep actually moves the decisions
    assert prev[1].sum() > 0
    # one point of the sweep against the oracle under the parity bar
    for t in range(w.queries.shape[0]):
        P.compare_query(P.gpu_query(eng, w, t, eps=0.1), P.oracle_query(w, t, pcs, eps=0.1), w,
                        eps=0.1)
    eng.close()
