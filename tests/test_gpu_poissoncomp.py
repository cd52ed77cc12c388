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


@pytest.mark.parametrize("n,eta", [(32768, 1 / 16), (131072, 1 / 32)])
def test_full_cache_sampled_heads(n, eta):
    """The PoissonComp throughput configuration at full size -- 36 layers x 8 KV heads in one
    call, as bench.py --pc-sweep times it -- with three sampled heads checked against the oracle
    bit for bit (c, r, the sample, ids and the gathered rows)."""
    import oracle as O
    from verified_kv_cache_poissoncomp_gb300 import binding as B
    from verified_kv_cache_poissoncomp_gb300.engine import default_cap

    layers, kvh, d = 36, 8, 128
    units = layers * kvh
    dev = torch.device("cuda", torch.cuda.current_device())
    tau_np = I.pc_sweep_tau(units, n)
    tau = torch.from_numpy(tau_np).to(dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(7)
    kv = torch.empty((units, n, 2, d), dtype=torch.int16, device=dev)
    kv.random_(-32768, 32767, generator=gen)
    cap = default_cap(n, eta)
    shape = B.verkv_shape(1, layers, kvh, 4, d, n, cap)
    ws_bytes = B.verkv_workspace_size(shape)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    r_full = torch.empty((units, n), dtype=torch.float32, device=dev)
    ids = torch.empty((units, cap), dtype=torch.int32, device=dev)
    pr = torch.empty((units, cap), dtype=torch.float32, device=dev)
    pkv = torch.empty((units, cap, 2, d), dtype=torch.int16, device=dev)
    cnt = torch.empty((units,), dtype=torch.int32, device=dev)
    res = torch.empty((units, (n + 31) // 32), dtype=torch.int32, device=dev)
    c = torch.empty((units,), dtype=torch.float32, device=dev)
    piv = B.verkv_pivotal(ids.data_ptr(), pr.data_ptr(), pkv.data_ptr(), cnt.data_ptr(),
                          res.data_ptr(), c.data_ptr())
    stream = torch.cuda.current_stream(dev)
    ctx = B.verkv_create(dev.index, stream.cuda_stream, shape, ws.data_ptr(), ws_bytes)
    seed = 2 ** 33 + 11
    B.verkv_poissoncomp(ctx, tau.data_ptr(), eta, B.verkv_hset(4, 512), seed, kv.data_ptr(),
                        r_full.data_ptr(), piv)
    B.verkv_sync(ctx)
    for u in (0, 137, units - 1):
        l, h = u // kvh, u % kvh
        o = O.poissoncomp(tau_np[u], eta, 4, 512, seed, 0, l, h)
        assert np.float32(c[u].item()) == o["c32"], u
        assert np.array_equal(r_full[u].cpu().numpy(), o["r32"]), u
        k = int(cnt[u].item())
        want = np.nonzero(o["resident"])[0]
        assert k == len(want) == o["count"], (u, k, len(want))
        assert np.array_equal(ids[u, :k].cpu().numpy(), want), u
        assert np.array_equal(P.bits_to_bool(res[u].cpu().numpy(), n), o["resident"]), u
        idx = torch.as_tensor(want, device=dev, dtype=torch.long)
        assert torch.equal(pkv[u, :k], kv[u].index_select(0, idx)), u
    B.verkv_destroy(ctx)
