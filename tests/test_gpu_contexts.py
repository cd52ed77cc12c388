"""Several contexts at once: a batch split over contexts on their own streams, run concurrently,
against one context for the whole batch.

A context owns its workspace, streams and counters, so contexts on different streams must not
interfere; and a context computes each (sequence, layer, KV head) unit as a larger one does (with
its sequence offset set, a sequence's Poisson draws are those of the whole-batch context; a logit
does not depend on the tile its row falls in; every refine item writes its own partial).  So the
outputs of the split run must equal, bit for bit, the matching slices of the whole-batch run: o,
lse, the head statistics and F.
"""
import numpy as np
import pytest
import torch

from verified_kv_cache_poissoncomp_gb300 import inputs as I
from verified_kv_cache_poissoncomp_gb300.engine import VerKV, default_cap, stats_to_dict

pytestmark = pytest.mark.gpu

BT, L, KVH, G, D, N = 4, 2, 2, 4, 128, 8192
ETA = 1 / 8


def _engines(w, groups, dev):
    bg = BT // groups
    ug = bg * L * KVH
    tau = torch.as_tensor(w.tau.reshape(-1, N)).to(dev)
    kv = torch.as_tensor(w.kv.reshape(-1, N, 2, D).view(np.int16)).to(dev)
    host = torch.empty(kv.shape, dtype=torch.int16, pin_memory=True)
    host.copy_(kv)
    streams = [torch.cuda.Stream(dev) for _ in range(groups)]
    engs = []
    for gi in range(groups):
        with torch.cuda.stream(streams[gi]):
            e = VerKV(bg, L, KVH, G, D, N, default_cap(N, ETA), seq0=gi * bg)
            e.load_device(tau[gi * ug:(gi + 1) * ug], kv[gi * ug:(gi + 1) * ug],
                          host[gi * ug:(gi + 1) * ug])
            e.compress(ETA, w.n_sink, w.n_local, w.seed)
        engs.append(e)
    torch.cuda.synchronize()
    return engs, streams, (tau, kv, host)


def _run(w, groups, dev):
    engs, streams, keep = _engines(w, groups, dev)
    bg = BT // groups
    hg = bg * KVH * G
    out = []
    for t in range(w.queries.shape[0]):
        layer = int(w.query_layer[t])
        q = torch.as_tensor(w.queries[t].view(np.int16)).to(dev)  # [BT][KVH * G][D]
        res = []
        for gi, e in enumerate(engs):  # every group enqueued before any is waited for
            with torch.cuda.stream(streams[gi]):
                e.attend(layer, q[gi * bg:(gi + 1) * bg], w.eps, w.delta, with_ids=False)
                F = e.selection_bitmap()
                o, lse, st = e.fetch_refine(torch.empty_like(e.o), torch.empty_like(e.lse),
                                            torch.empty_like(e.stats))
                res.append((F, o, lse, st))
        torch.cuda.synchronize()
        for e in engs:
            e.sync()
        F = torch.cat([r[0] for r in res]).cpu().numpy()
        o = torch.cat([r[1] for r in res]).cpu().numpy()
        lse = torch.cat([r[2] for r in res]).cpu().numpy()
        st = torch.cat([r[3] for r in res])
        assert o.shape[0] == BT * KVH * G and hg * groups == o.shape[0]
        out.append(dict(F=F, o=o, lse=lse, stats=stats_to_dict(st)))
    for e in engs:
        e.close()
    del keep
    return out


def test_concurrent_contexts_match_one_context():
    dev = torch.device("cuda", 0)
    w = I.make_workload("ctx", B=BT, L=L, h_kv=KVH, G=G, d=D, n=N, eta=ETA, n_queries=6,
                        plant_every=2)
    one = _run(w, 1, dev)
    split = _run(w, BT, dev)  # one sequence per context, all four streams in flight together
    fetching = 0
    for a, b in zip(one, split):
        for k in ("F", "o", "lse"):
            assert np.array_equal(a[k].view(np.uint8), b[k].view(np.uint8)), k
        for k, v in a["stats"].items():
            assert np.array_equal(np.asarray(v).view(np.uint8), np.asarray(b["stats"][k]).view(np.uint8)), k
        fetching += int((a["stats"]["certified"] == 0).sum())
    assert fetching > 0  # the fetch path ran
