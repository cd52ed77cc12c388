"""The full-decode-step shapes against the fp64 oracle on sampled units: batch 8 x 8 KV heads x 4
query heads, d = 128, n = 32768, eta in {1/8, 1/32}.

One layer call at batch 8 covers 64 KV heads and 256 query heads, so the certify grid is 1024 CTAs
in 256 clusters (several waves), the score kernel splits each head into a few long spans, and the
fetch moves thousands of rows per KV head.  The cache comes from the decode-step workload's
device-side generator with two layers (the full step has 36; that only changes the host cache's
size).  Each call is followed by a synchronisation.  On the sampled units, the PoissonComp output is
compared bit-exact, and the certificate, the selection, the fetch list and the estimator are held to
the parity bar of tests/parity.py.
"""
import types

import numpy as np
import pytest
import torch

import oracle as O
from tests import parity as P
from verified_kv_cache_poissoncomp_gb300 import binding as B
from verified_kv_cache_poissoncomp_gb300 import inputs as I
from verified_kv_cache_poissoncomp_gb300.engine import VerKV, default_cap, stats_to_dict

pytestmark = pytest.mark.gpu

LAYERS, BATCH, KVH, G, D, N = 2, 8, 8, 4, 128, 32768
SAMPLED = [0, 13, 38, 63]  # layer-local units u' = b * KVH + h: (0,0), (1,5), (4,6), (7,7)


@pytest.fixture(scope="module")
def cache():
    dev = torch.device("cuda", 0)
    units = BATCH * LAYERS * KVH
    tau, kv, queries, planted = I.decode_step_cache_torch(units, N, D, G, LAYERS, BATCH, KVH, dev)
    assert planted.any()
    host_kv = torch.empty(kv.shape, dtype=torch.int16, pin_memory=True)
    host_kv.copy_(kv)
    torch.cuda.synchronize()
    return dict(dev=dev, tau=tau, kv=kv, queries=queries, host_kv=host_kv,
                tau_np=tau.cpu().numpy(), q_np=queries.cpu().numpy().view(np.uint16))


def _unit(b, l, h):
    return (b * LAYERS + l) * KVH + h


def _subset(g, uls):
    """The GPU results of the units `uls`, renumbered 0..len(uls)-1 as compare_query expects."""
    rows = np.concatenate([np.arange(u * G, (u + 1) * G) for u in uls])
    return dict(o=g["o"][rows], lse=g["lse"][rows], F=g["F"][rows],
                stats={k: v[rows] for k, v in g["stats"].items()},
                ids=g["ids"][uls], counts=g["counts"][uls])


@pytest.mark.parametrize("eta", [1 / 8, 1 / 32])
def test_decode_step_sampled_units(cache, eta):
    c = cache
    eps = delta = 0.05
    eng = VerKV(BATCH, LAYERS, KVH, G, D, N, default_cap(N, eta))
    eng.load_device(c["tau"], c["kv"], c["host_kv"])
    eng.compress(eta, 4, 512, 0)
    eng.sync()
    p_ids, p_cnt = eng.p_ids.cpu().numpy(), eng.p_count.cpu().numpy()
    p_kv = eng.p_kv.cpu().numpy().view(np.uint16)
    r_full = eng.r_full.cpu().numpy()
    w = types.SimpleNamespace(G=G, n=N)
    rep = None
    uncertified = 0
    for l in range(LAYERS):
        q = c["queries"][l]
        eng.attend(l, q, eps, delta)
        eng.sync()
        F = eng.selection_bitmap()
        o, lse, stats = eng.fetch_refine()
        eng.sync()
        g = dict(o=o.cpu().numpy(), lse=lse.cpu().numpy(), stats=stats_to_dict(stats),
                 F=P.bits_to_bool(F.cpu().numpy(), N), ids=eng.fetch_ids.cpu().numpy(),
                 counts=eng.fetch_counts.cpu().numpy())
        units = []
        for ul in SAMPLED:
            b, h = divmod(ul, KVH)
            u = _unit(b, l, h)
            pc = O.poissoncomp(c["tau_np"][u], eta, 4, 512, 0, b, l, h)
            want = np.nonzero(pc["resident"])[0]
            assert np.array_equal(r_full[u], pc["r32"]), u
            assert p_cnt[u] == len(want) == pc["count"], (u, p_cnt[u], len(want))
            assert np.array_equal(p_ids[u, :p_cnt[u]], want), u
            kv_u = c["kv"][u].cpu().numpy().view(np.uint16)
            assert np.array_equal(p_kv[u, :p_cnt[u]], kv_u[want]), u
            K = O.bf16_to_f64(kv_u[:, 0, :])
            V = O.bf16_to_f64(kv_u[:, 1, :])
            qs = O.bf16_to_f64(c["q_np"][l, b, h * G:(h + 1) * G])
            units.append(O.attend_unit(qs, K, K, V, pc["r32"], pc["resident"], eps, delta))
        sub = _subset(g, SAMPLED)
        rep = P.compare_query(sub, units, w, eps=eps, report=rep)
        uncertified += int((sub["stats"]["certified"] == 0).sum())
    print(rep)
    assert uncertified > 0  # the selection and the fetch ran on sampled heads
    assert rep["exact_F"] >= 0.9 * rep["heads"]
    eng.close()


def test_memcpy_mode_matches_zerocopy_at_step_size(cache):
    # At these shapes every CTA of the MEMCPY path's staged pivotal kernel takes about ten items
    # (4,672 items over 456 CTAs), so its two-stage ring is refilled and its barrier phases flip;
    # the two fetch modes must still give the same bits.  Layer 1, to index the second layer.
    c = cache
    eta = 1 / 8
    res = []
    for mode in (B.VERKV_FETCH_ZEROCOPY, B.VERKV_FETCH_MEMCPY):
        eng = VerKV(BATCH, LAYERS, KVH, G, D, N, default_cap(N, eta), fetch_mode=mode)
        eng.load_device(c["tau"], c["kv"], c["host_kv"])
        eng.compress(eta, 4, 512, 0)
        eng.sync()
        eng.attend(1, c["queries"][1], 0.05, 0.05)
        o, lse, _ = eng.fetch_refine()
        eng.sync()
        res.append((o.cpu().numpy(), lse.cpu().numpy()))
        eng.close()
    assert np.isfinite(res[0][0]).all()
    assert np.array_equal(res[0][0], res[1][0]) and np.array_equal(res[0][1], res[1][1])
