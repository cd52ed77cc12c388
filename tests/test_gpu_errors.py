"""Failure paths, all made on the host or by invalid inputs the library checks: no GPU fault."""
import numpy as np
import pytest
import torch

from tests import parity as P
from verified_kv_cache_poissoncomp_gb300 import binding as B
from verified_kv_cache_poissoncomp_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def test_budget_below_forced_set_is_rejected_on_host():
    w = I.tiny()
    eng = P.make_engine(w)
    with pytest.raises(B.VerkvError) as e:
        eng.compress(60 / 1024, w.n_sink, w.n_local, 0)   # eta n = 60 < 68 forced
    assert e.value.status == B.VERKV_EBUDGET


def test_capacity_overflow_is_reported():
    w = I.tiny()
    eng = P.make_engine(w, cap=64)   # |H| alone is 68
    eng.compress(w.eta, w.n_sink, w.n_local, w.seed)
    assert B.verkv_sync_status(eng.ctx) == B.VERKV_ECAPACITY
    assert eng.p_count.cpu().numpy()[0] == 64
    assert B.verkv_sync_status(eng.ctx) == B.VERKV_OK   # cleared


@pytest.mark.parametrize("bad", [0.0, -0.5, 1.5, float("nan"), float("inf")])
def test_invalid_tau_is_reported(bad):
    w = I.tiny()
    tau = w.tau.copy()
    tau[0, 0, 0, 500] = bad
    eng = P.make_engine(w)
    eng.load(tau.reshape(-1, w.n), w.kv.reshape(-1, w.n, 2, w.d))
    eng.compress(w.eta, w.n_sink, w.n_local, w.seed)
    assert B.verkv_sync_status(eng.ctx) == B.VERKV_EINVAL


def test_call_order_and_arguments():
    w = I.tiny()
    eng = P.make_engine(w)
    eng.compress(w.eta, w.n_sink, w.n_local, w.seed)
    o = torch.empty_like(eng.o)
    st = B.lib().verkv_fetch_refine(eng.ctx, None, None, eng.host_kv.data_ptr(), o.data_ptr(),
                                    None, None)
    assert st == B.VERKV_ESTATE
    q = torch.as_tensor(w.queries[0].view(np.int16)).cuda()
    with pytest.raises(B.VerkvError):
        eng.attend(1, q, w.eps, w.delta)             # layer out of range
    with pytest.raises(B.VerkvError):
        eng.attend(0, q, w.eps, 1.5)                 # delta outside (0, 1)
    eng.attend(0, q, w.eps, w.delta)
    # fetch_refine needs page-locked host memory
    dev_kv = eng.kv
    st = B.lib().verkv_fetch_refine(eng.ctx, eng._ids, eng._cnt, dev_kv.data_ptr(), o.data_ptr(),
                                    None, None)
    assert st == B.VERKV_EINVAL
    eng.fetch_refine()
    eng.sync()
