"""The shortlist variant on the GPU (only a per-KV-head shortlist of S tokens may be fetched):
the GPU's shortlist against its definition on the oracle's fp64 logits (swaps only among
near-equal keys at the boundary), then -- given the GPU's shortlist -- certificate, restricted
selection, exhaustion flag, fetch list and estimator against the oracle under the tie-aware
parity bar."""
import numpy as np
import pytest

import oracle as O
from tests import parity as P
from verified_kv_cache_poissoncomp_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def _run(w, size, queries, eps=None):
    eps = w.eps if eps is None else eps
    eng = P.make_engine(w)
    eng.compress(w.eta, w.n_sink, w.n_local, w.seed)
    eng.sync()
    eng.set_shortlist(size)
    pcs = P.oracle_poissoncomp(w)
    seen = dict(exhausted=0, met=0)
    for t in queries:
        g = P.gpu_query(eng, w, t, eps=eps)
        slb = P.bits_to_bool(eng.shortlist_bitmap().cpu().numpy(), w.n)
        l = int(w.query_layer[t])
        cands = {}
        for b in range(w.B):
            for h in range(w.h_kv):
                ul = b * w.h_kv + h
                r32 = pcs[(b, l, h)]["r32"]
                K = O.bf16_to_f64(w.kv[b, l, h, :, 0, :])
                qs = O.bf16_to_f64(w.queries[t, b, h * w.G:(h + 1) * w.G])
                s_hats = [O.logits(q, K) for q in qs]
                om = O.shortlist(s_hats, r32, size)
                gm = slb[ul]
                assert gm.sum() == om.sum() == min(size, int((r32 < 1).sum()))
                if not np.array_equal(gm, om):
                    key = np.max(s_hats, axis=0)
                    cut = np.min(key[om])
                    for tok in np.nonzero(gm ^ om)[0]:
                        assert abs(key[tok] - cut) <= 1e-5 * (abs(cut) + 1.0), (t, ul, tok)
                cands[(b, h)] = gm
                for g_ in range(w.G):
                    qh = ul * w.G + g_
                    assert not (g["F"][qh] & ~gm).any()
                    flags = int(g["stats"]["flags"][qh])
                    if not g["stats"]["certified"][qh]:
                        seen["exhausted" if flags & 4 else "met"] += 1
                assert g["counts"][ul] <= size
        units = P.oracle_query(w, t, pcs, eps=eps, cands=cands)
        P.compare_query(g, units, w, eps=eps)
    eng.close()
    return seen


def test_shortlist_tiny_and_mid():
    seen = _run(I.tiny(), 16, range(16))
    w = I.make_workload("slmid", B=2, L=1, h_kv=2, G=4, d=128, n=20000, n_queries=6,
                        plant_every=2, n_local=512)
    s2 = _run(w, 128, range(6))
    assert seen["exhausted"] + s2["exhausted"] > 0
    assert seen["met"] + s2["met"] > 0


def test_shortlist_covering_L_is_the_plain_path():
    # A shortlist larger than L lets every token of L be fetched: the plain certificate's result.
    w = I.make_workload("slall", B=1, L=1, h_kv=2, G=4, d=64, n=300, eta=1 / 4, n_local=16,
                        n_sink=4, n_queries=4, plant_every=2)
    eng = P.make_engine(w)
    eng.compress(w.eta, w.n_sink, w.n_local, w.seed)
    eng.sync()
    pcs = P.oracle_poissoncomp(w)
    eng.set_shortlist(256)
    for t in range(4):
        g = P.gpu_query(eng, w, t)
        P.compare_query(g, P.oracle_query(w, t, pcs), w)
        assert not (g["stats"]["flags"] & 4).any()
    eng.close()
