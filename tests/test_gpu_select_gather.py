"""The selection's gathered finish against its histogram passes, bit for bit.

With clusters of 1 and 4 CTAs the certificate kernel may end the selection of Eq. (10) ("Verify
Before You Fetch", summary page, KVFETCH steps 3-4) by gathering the tokens of the cut bin into
one CTA and ranking them there, once at most 512 remain.  It takes k* from the same exact
fixed-point sums and the same eps-hat expression as the finer histogram passes, so the two must
give the same bits: F, k*, eps-hat and, downstream, o and lse.  Here the same queries run with the
gathered finish allowed (the default) and with the histogram passes forced to the end, and every
output is compared bitwise (the stats flag 8, which records the gathered finish, aside).  The
oracle comparison of both runs is in the other parity tests; this one pins their equality.
"""
import numpy as np
import pytest

from tests import parity as P
from verified_kv_cache_poissoncomp_gb300 import binding as B
from verified_kv_cache_poissoncomp_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def _outputs(w, gather):
    eng = P.make_engine(w)
    eng.compress(w.eta, w.n_sink, w.n_local, w.seed)
    eng.sync()
    B.verkv_test_inject(eng.ctx, B.VERKV_INJECT_SELECT_GATHER, 1 if gather else 0)
    outs = [P.gpu_query(eng, w, t) for t in range(w.queries.shape[0])]
    eng.close()
    return outs


# Clusters of 4 (n = 20000: a ragged last CTA) and of 1 (n = 8192).
@pytest.mark.parametrize("n,h_kv,eta,n_local", [(20000, 8, 1 / 16, 512), (8192, 2, 1 / 8, 256)])
def test_gathered_select_matches_histogram_passes(n, h_kv, eta, n_local):
    w = I.make_workload("gather", B=1, L=2, h_kv=h_kv, G=4, d=128, n=n, eta=eta, n_local=n_local,
                        n_queries=8, plant_every=2)
    a = _outputs(w, gather=True)
    b = _outputs(w, gather=False)
    gathered = 0
    for x, y in zip(a, b):
        for k in ("o", "lse", "F", "counts"):
            assert np.array_equal(np.asarray(x[k]).view(np.uint8), np.asarray(y[k]).view(np.uint8)), k
        for ul, c in enumerate(x["counts"]):  # the list's entries past each count are not written
            assert np.array_equal(x["ids"][ul, :c], y["ids"][ul, :c])
        for k, v in x["stats"].items():
            u = y["stats"][k]
            if k == "flags":
                assert np.array_equal(v & ~8, u), k
                assert not (u & 8).any()
                gathered += int((v & 8).astype(bool).sum())
            else:
                assert np.array_equal(np.asarray(v).view(np.uint8), np.asarray(u).view(np.uint8)), k
        fetching = int((x["stats"]["certified"] == 0).sum())
        assert int((x["stats"]["flags"] & 8).astype(bool).sum()) <= fetching
    assert gathered > 0  # the gathered finish ran on some heads
