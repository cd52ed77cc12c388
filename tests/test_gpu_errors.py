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


def test_misaligned_pointers_are_rejected_before_launch():
    # Every call checks the alignment its kernels rely on (16 bytes for bf16 rows and queries,
    # 4 for the other arrays) and returns VERKV_EINVAL before launching anything: the offset
    # pointers below are never dereferenced.
    w = I.tiny()
    eng = P.make_engine(w)
    eng.compress(w.eta, w.n_sink, w.n_local, w.seed)
    eng.sync()
    lib = B.lib()
    q = torch.as_tensor(w.queries[0].view(np.int16)).to(eng.dev)
    launches = B.verkv_launch_counts(eng.ctx)

    def attend(qp=q.data_ptr(), sketch=eng.sketch.data_ptr(), r=eng.r_full.data_ptr(), ids=None):
        sk = B.verkv_sketch(B.VERKV_SKETCH_EXACT, sketch)
        return lib.verkv_attend_verified(eng.ctx, 0, qp, eng.pivotal, r, sk, w.eps, w.delta,
                                         ids, None)

    assert attend(qp=q.data_ptr() + 8) == B.VERKV_EINVAL
    assert attend(sketch=eng.sketch.data_ptr() + 2) == B.VERKV_EINVAL
    assert attend(r=eng.r_full.data_ptr() + 2) == B.VERKV_EINVAL
    assert attend(ids=eng.fetch_ids.data_ptr() + 1) == B.VERKV_EINVAL
    pv = B.verkv_pivotal(eng.p_ids.data_ptr(), eng.p_r.data_ptr(), eng.p_kv.data_ptr() + 4,
                         eng.p_count.data_ptr(), eng.p_res.data_ptr(), eng.p_c.data_ptr())
    sk = B.verkv_sketch(B.VERKV_SKETCH_EXACT, eng.sketch.data_ptr())
    assert lib.verkv_attend_verified(eng.ctx, 0, q.data_ptr(), pv, eng.r_full.data_ptr(), sk,
                                     w.eps, w.delta, None, None) == B.VERKV_EINVAL
    assert lib.verkv_sketch_build(eng.ctx, eng.kv.data_ptr() + 2, B.VERKV_SKETCH_EXACT,
                                  eng.sketch.data_ptr()) == B.VERKV_EINVAL
    assert lib.verkv_poissoncomp(eng.ctx, eng.tau.data_ptr(), w.eta, B.verkv_hset(4, 64), 0,
                                 eng.kv.data_ptr() + 8, eng.r_full.data_ptr(),
                                 eng.pivotal) == B.VERKV_EINVAL
    o = torch.empty_like(eng.o)
    assert lib.verkv_attend_dense_host(eng.ctx, 0, q.data_ptr(), eng.host_kv.data_ptr() + 2,
                                       o.data_ptr(), None) == B.VERKV_EINVAL
    assert B.verkv_launch_counts(eng.ctx) == launches  # nothing was launched
    eng.attend(0, q, w.eps, w.delta)
    assert lib.verkv_fetch_refine(eng.ctx, eng._ids, eng._cnt, eng.host_kv.data_ptr() + 4,
                                  o.data_ptr(), None, None) == B.VERKV_EINVAL
    assert lib.verkv_fetch_refine(eng.ctx, eng._ids, eng._cnt, eng.host_kv.data_ptr(),
                                  o.data_ptr() + 2, None, None) == B.VERKV_EINVAL
    eng.fetch_refine()
    eng.sync()
    eng.close()


def _query_ok(eng, w, t, pcs):
    """One query through the context, checked against the oracle: the context is usable."""
    g = P.gpu_query(eng, w, t)
    P.compare_query(g, P.oracle_query(w, t, pcs), w)


def test_fetch_copy_failure_is_reported_and_the_context_recovers():
    # A host-side failure of the MEMCPY fetch's copy (injected before it reaches CUDA) comes back
    # as VERKV_ECOPY from verkv_fetch_refine; the next decode call on the context succeeds.
    w = I.tiny()
    eng = P.make_engine(w, fetch_mode=B.VERKV_FETCH_MEMCPY)
    eng.compress(w.eta, w.n_sink, w.n_local, w.seed)
    eng.sync()
    pcs = P.oracle_poissoncomp(w)
    t = int(np.nonzero(w.planted)[0][0])  # a planted query: its certificate fails, rows move
    B.verkv_test_inject(eng.ctx, B.VERKV_INJECT_COPY_FAIL, 1)
    q = torch.as_tensor(w.queries[t].view(np.int16)).to(eng.dev)
    eng.attend(int(w.query_layer[t]), q, w.eps, w.delta)
    with pytest.raises(B.VerkvError) as e:
        eng.fetch_refine()
    assert e.value.status == B.VERKV_ECOPY
    assert B.verkv_sync_status(eng.ctx) == B.VERKV_OK
    _query_ok(eng, w, t, pcs)
    eng.close()


def test_beta_iteration_cap_is_reported_and_can_be_lifted():
    # With the beta solve capped at one pass, heads that need more are flagged (stats flags & 1)
    # and verkv_sync returns VERKV_ENOCONVERGE; the default cap gives results at the parity bar.
    w = I.tiny()
    eng = P.make_engine(w)
    eng.compress(w.eta, w.n_sink, w.n_local, w.seed)
    eng.sync()
    pcs = P.oracle_poissoncomp(w)
    B.verkv_test_inject(eng.ctx, B.VERKV_INJECT_BETA_MAXIT, 1)
    flagged = 0
    for t in range(w.queries.shape[0]):
        q = torch.as_tensor(w.queries[t].view(np.int16)).to(eng.dev)
        eng.attend(int(w.query_layer[t]), q, w.eps, w.delta)
        _, _, st = eng.fetch_refine()
        status = B.verkv_sync_status(eng.ctx)
        f = int((st.cpu().numpy()[:, 15] & 1).sum())
        assert status == (B.VERKV_ENOCONVERGE if f else B.VERKV_OK), (t, status, f)
        flagged += f
    assert flagged > 0
    B.verkv_test_inject(eng.ctx, B.VERKV_INJECT_BETA_MAXIT, 0)
    for t in range(4):
        _query_ok(eng, w, t, pcs)
    eng.close()


def test_bounded_copy_wait_expiry_is_reported_and_the_context_recovers():
    # The scoring kernel's first CTA arms a copy barrier for a copy it never issues; its bounded
    # wait gives up after 2 ms, the kernel latches VERKV_ETIMEOUT and returns (no trap, no fault),
    # verkv_sync reports it, and the next call on the same context meets the parity bar.
    w = I.tiny()
    eng = P.make_engine(w)
    eng.compress(w.eta, w.n_sink, w.n_local, w.seed)
    eng.sync()
    pcs = P.oracle_poissoncomp(w)
    B.verkv_test_inject(eng.ctx, B.VERKV_INJECT_SCORE_STALL, 2_000_000)
    q = torch.as_tensor(w.queries[0].view(np.int16)).to(eng.dev)
    eng.attend(0, q, w.eps, w.delta)
    eng.fetch_refine()
    assert B.verkv_sync_status(eng.ctx) == B.VERKV_ETIMEOUT
    assert B.verkv_sync_status(eng.ctx) == B.VERKV_OK  # cleared
    for t in range(4):
        _query_ok(eng, w, t, pcs)
    eng.close()


def test_injection_arguments_are_checked():
    w = I.tiny()
    eng = P.make_engine(w)
    for what, value in [(0, 1), (B.VERKV_INJECT_COPY_FAIL, -1), (B.VERKV_INJECT_BETA_MAXIT, 65),
                        (B.VERKV_INJECT_SCORE_STALL, 10), (B.VERKV_INJECT_SELECT_GATHER, 2)]:
        with pytest.raises(B.VerkvError) as e:
            B.verkv_test_inject(eng.ctx, what, value)
        assert e.value.status == B.VERKV_EINVAL
    with pytest.raises(B.VerkvError) as e:  # a sequence offset below zero
        B.verkv_set_sequence_offset(eng.ctx, -1)
    assert e.value.status == B.VERKV_EINVAL
    eng.close()


def test_sketch_stream_measurement_call():
    # The measurement call streams a layer's exact sketch through the scoring kernel's copy ring;
    # it checks its arguments on the host and leaves no error behind.
    w = I.tiny()
    eng = P.make_engine(w)
    eng.compress(w.eta, w.n_sink, w.n_local, w.seed)
    eng.sync()
    launches = B.verkv_launch_counts(eng.ctx)
    B.verkv_measure_sketch_stream(eng.ctx, 0, eng.sketch_desc)
    assert B.verkv_sync_status(eng.ctx) == B.VERKV_OK
    assert B.verkv_launch_counts(eng.ctx) == launches  # not a decode kernel: not counted
    lib = B.lib()
    bad = [(w.L, eng.sketch_desc),
           (0, B.verkv_sketch(B.VERKV_SKETCH_Q2, eng.sketch.data_ptr())),
           (0, B.verkv_sketch(B.VERKV_SKETCH_EXACT, eng.sketch.data_ptr() + 8))]
    for layer, sk in bad:
        assert lib.verkv_measure_sketch_stream(eng.ctx, layer, sk) == B.VERKV_EINVAL
    eng.close()
