"""GPU PoissonComp against the fp64 oracle: bit-exact c (float32), r, resident bitmap, pivotal ids,
r and rows ("Verify Before You Fetch", summary page, POISSONCOMP, Eq. (3) and the sample S)."""
import numpy as np
import pytest
import torch

from tests import parity as P
from verified_kv_cache_poissoncomp_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def _run(w, cap=None):
    eng = P.make_engine(w, cap=cap)
    eng.compress(w.eta, w.n_sink, w.n_local, w.seed)
    eng.sync()
    P.check_poissoncomp(eng, w, P.oracle_poissoncomp(w))
    return eng


def test_tiny():
    _run(I.tiny())


@pytest.mark.parametrize("n,eta,n_sink,n_local,seed", [
    (1000, 1 / 8, 4, 64, 0),          # ragged tail (n not a multiple of 32), one CTA
    (4096, 1 / 4, 0, 0, 7),           # no forced H
    (32768, 1 / 16, 4, 512, 0),       # the single-layer 32K budget
    (32768, 1 / 32, 4, 512, 123456789),
    (32768, 1 / 8, 4, 512, 2 ** 40 + 5),
    (50001, 1 / 16, 4, 512, 3),       # two-CTA cluster, ragged
    (131072, 1 / 32, 4, 512, 1),      # four-CTA cluster, 128K
])
def test_shapes_and_budgets(n, eta, n_sink, n_local, seed):
    w = I.make_workload("pc", B=2, L=2, h_kv=2, G=1, d=64, n=n, eta=eta, n_sink=n_sink,
                        n_local=n_local, n_queries=1, philox_seed=seed,
                        data_seed=n + int(1 / eta))
    _run(w)


def test_eta_one_keeps_every_token():
    w = I.make_workload("eta1", B=1, L=1, h_kv=2, G=1, d=64, n=3000, eta=1.0, n_queries=1,
                        n_local=64)
    eng = _run(w, cap=3000)
    assert np.all(eng.r_full.cpu().numpy() == 1.0)
    assert np.all(eng.p_count.cpu().numpy() == 3000)


def test_deterministic_across_calls():
    w = I.make_workload("det", B=1, L=1, h_kv=4, G=1, d=128, n=20000, n_queries=1)
    eng = P.make_engine(w)
    eng.compress(w.eta, w.n_sink, w.n_local, w.seed)
    eng.sync()
    a = [t.clone() for t in (eng.r_full, eng.p_ids, eng.p_kv, eng.p_res)]
    eng.compress(w.eta, w.n_sink, w.n_local, w.seed)
    eng.sync()
    for x, y in zip(a, (eng.r_full, eng.p_ids, eng.p_kv, eng.p_res)):
        assert torch.equal(x, y)
