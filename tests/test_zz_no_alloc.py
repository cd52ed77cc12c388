"""verkv_certify_noalloc, the allocation-free certificate, against verkv_attend_verified.

Callers that cannot allocate device memory (a runtime that has already reserved the GPU's memory
for its own pools, or a plugin interface that hands an operator only its inputs and outputs)
cannot give a context its workspace.  verkv_certify_noalloc computes the same per-query-head
certificate, k* and fetch set F for them with its logits in a fixed array owned by the library.
Here it is called through the C ABI several times in a row -- so every call after the first
finds the previous call's logits in that array -- and each result must equal what the context
path computes for the same query, within the parity tolerances of tests/parity.py.

This file is collected last on purpose: a run that stops at the first failure has run every
other test before it.
"""
import numpy as np
import pytest
import torch

from tests import parity as P
from verified_kv_cache_poissoncomp_gb300 import binding as B
from verified_kv_cache_poissoncomp_gb300 import inputs as I
from verified_kv_cache_poissoncomp_gb300.engine import stats_to_dict

pytestmark = pytest.mark.gpu

CERT_FLOATS = ["m", "D", "beta", "V", "b", "eps_hat", "eps_final"]
CERT_INTS = ["certified", "k_star", "n_L", "iters", "flags"]


def _noalloc(eng, w, layer, q, eps, delta):
    """One verkv_certify_noalloc call over the KV heads of `layer` (batch 1: they are consecutive
    units).  The outputs are pre-filled with garbage so that every word must be written."""
    units, qh = w.h_kv, w.h_kv * w.G
    u0 = layer * w.h_kv
    stats = torch.full((qh, 16), 0x7F7F7F7F, dtype=torch.int32, device=eng.dev)
    F = torch.full((qh, eng.W), -1, dtype=torch.int32, device=eng.dev)
    err = torch.full((1,), -1, dtype=torch.int32, device=eng.dev)
    B.verkv_certify_noalloc(eng.dev.index, torch.cuda.current_stream(eng.dev).cuda_stream,
                            units, w.G, w.d, w.n, q.data_ptr(), eng.sketch[u0].data_ptr(),
                            eng.r_full[u0].data_ptr(), eps, delta, stats.data_ptr(),
                            F.data_ptr(), err.data_ptr())
    torch.cuda.synchronize(eng.dev)
    return stats_to_dict(stats), F.cpu().numpy(), int(err.item())


def _context_path(eng, layer, q, eps, delta):
    eng.attend(layer, q, eps, delta)
    F = eng.selection_bitmap()
    _, _, stats = eng.fetch_refine()
    eng.sync()
    return stats_to_dict(stats), F.cpu().numpy()


def test_noalloc_certificate_matches_context_path_on_consecutive_calls():
    w = I.make_workload("noalloc", B=1, L=2, h_kv=2, G=4, d=128, n=20000, n_queries=4,
                        plant_every=2, n_local=512)
    eng = P.make_engine(w)
    eng.compress(w.eta, w.n_sink, w.n_local, w.seed)
    eng.sync()
    uncertified = 0
    for t in (1, 0, 3):  # planted (layer 1), plain (layer 0), planted (layer 1)
        layer = int(w.query_layer[t])
        q = torch.as_tensor(w.queries[t].view(np.int16)).to(eng.dev)
        got, Fg, err = _noalloc(eng, w, layer, q, w.eps, w.delta)
        want, Fw = _context_path(eng, layer, q, w.eps, w.delta)
        assert err == 0, (t, err)
        for k in CERT_INTS:
            assert np.array_equal(got[k], want[k]), (t, k, got[k], want[k])
        for k in CERT_FLOATS:
            np.testing.assert_allclose(got[k], want[k], rtol=P.EPS_TIE, atol=0, err_msg=f"{t} {k}")
        for k in ["D_hat", "M2", "lse", "n_fetch"]:
            assert not np.any(got[k]), (t, k)
        assert np.array_equal(Fg, Fw), t
        uncertified += int((got["certified"] == 0).sum())
    # the planted queries make some certificates fail, so the selection ran too
    assert uncertified > 0
    eng.close()


def test_noalloc_rejects_more_logits_than_its_scratch_holds():
    # 8 KV heads x 8 query heads x 65537 tokens = 4194368 > 2^22 logits; rejected before any
    # launch (the pointers are never dereferenced).
    with pytest.raises(B.VerkvError) as e:
        B.verkv_certify_noalloc(0, None, 8, 8, 128, 65537, 16, 16, 16, 0.05, 0.05, 16, 16, 16)
    assert e.value.status == B.VERKV_ETOOLARGE
    assert 8 * 8 * 65536 <= B.VERKV_NOALLOC_MAX_LOGITS < 8 * 8 * 65537
