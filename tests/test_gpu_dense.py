"""The offloaded-dense baseline (every K|V row read from page-locked host memory) against the
oracle's dense attention: o and log-sum-exp within the estimator tolerance (fp32 accumulation
of bf16 inputs)."""
import numpy as np
import pytest
import torch

import oracle as O
from tests import parity as P
from verified_kv_cache_poissoncomp_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def _check(w, queries):
    eng = P.make_engine(w)
    worst_o = worst_l = 0.0
    for t in queries:
        l = int(w.query_layer[t])
        q = torch.as_tensor(w.queries[t].view(np.int16)).to(eng.dev)
        o, lse = eng.attend_dense_host(l, q)
        torch.cuda.synchronize()
        o, lse = o.cpu().numpy(), lse.cpu().numpy()
        for b in range(w.B):
            for h in range(w.h_kv):
                K = O.bf16_to_f64(w.kv[b, l, h, :, 0, :])
                V = O.bf16_to_f64(w.kv[b, l, h, :, 1, :])
                for g in range(w.G):
                    qh = (b * w.h_kv + h) * w.G + g
                    qv = O.bf16_to_f64(w.queries[t, b, h * w.G + g])
                    ref = O.dense(O.logits(qv, K), V)
                    eo = np.linalg.norm(o[qh] - ref["o"]) / np.linalg.norm(ref["o"])
                    el = abs(float(lse[qh]) - (ref["m"] + np.log(ref["D"])))
                    worst_o, worst_l = max(worst_o, eo), max(worst_l, el)
                    assert eo <= P.EST_TOL and el <= P.EST_TOL, (t, qh, eo, el)
    eng.close()
    print("worst o", worst_o, "worst lse", worst_l)


def test_dense_tiny():
    _check(I.tiny(), range(4))


def test_dense_ragged_batched():
    # n = 20000 (last chunk ragged), two sequences, two layers, GQA 4
    w = I.make_workload("dense", B=2, L=2, h_kv=2, G=4, d=128, n=20000, n_queries=3,
                        plant_every=2, n_local=512)
    _check(w, range(3))


@pytest.mark.parametrize("G,d", [(1, 64), (8, 128)])
def test_dense_head_shapes(G, d):
    w = I.make_workload("dshape", B=1, L=1, h_kv=2, G=G, d=d, n=3000, eta=1 / 8, n_local=64,
                        n_queries=2, plant_every=2)
    _check(w, range(2))
