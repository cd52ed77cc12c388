"""The 2-bit sketch on the GPU: its bytes against the oracle's quantiser (bit-exact), and the
whole decode path scored from it -- certificate, selection and the refined estimator (fetching
K and V rows) -- against the oracle run on the exact dequantised sketch keys, under the same
tie-aware parity bar as the exact sketch."""
import numpy as np
import pytest
import torch

from tests import parity as P
from verified_kv_cache_poissoncomp_gb300 import binding as B
from verified_kv_cache_poissoncomp_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def _run(w, queries):
    eng = P.make_engine(w, sketch_format=B.VERKV_SKETCH_Q2)
    eng.compress(w.eta, w.n_sink, w.n_local, w.seed)
    eng.sync()
    sk = P.oracle_q2_sketches(w)
    got = eng.sketch.cpu().numpy()
    u = 0
    for b in range(w.B):
        for l in range(w.L):
            for h in range(w.h_kv):
                rows, _ = sk[(b, l, h)]
                assert np.array_equal(got[u], rows), (b, l, h)
                u += 1
    pcs = P.oracle_poissoncomp(w)
    khat = {k: v[1] for k, v in sk.items()}
    rep = None
    for t in queries:
        g = P.gpu_query(eng, w, t)
        rep = P.compare_query(g, P.oracle_query(w, t, pcs, sketches=khat), w, report=rep)
    eng.close()
    print(rep)
    return rep


def test_q2_tiny():
    rep = _run(I.tiny(), range(16))
    assert rep["exact_F"] >= 0.9 * rep["heads"]


def test_q2_ragged_gqa_and_head_dims():
    w = I.make_workload("q2mid", B=2, L=1, h_kv=2, G=4, d=128, n=20000, n_queries=4,
                        plant_every=2, n_local=512)
    rep = _run(w, range(4))
    assert rep["exact_F"] >= 0.9 * rep["heads"]
    for G, d in [(8, 64), (2, 128)]:
        w = I.make_workload("q2shape", B=1, L=1, h_kv=2, G=G, d=d, n=3000, eta=1 / 8,
                            n_local=64, n_queries=2, plant_every=2)
        _run(w, range(2))
