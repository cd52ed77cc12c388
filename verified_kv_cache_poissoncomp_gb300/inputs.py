"""Seeded synthetic inputs shared by the CUDA path's tests/benchmark and the CPU oracle.

This module only synthesises data (importance scores, keys, values, queries) and converts float32
to bf16 bit patterns.  It holds none of VerKV's arithmetic: no inclusion probabilities, no
sampling, no estimator, no certificate.  The random draws that the method itself makes (the
Poisson sample) are not drawn here; both sides derive them from the Philox seed.

The pages evaluate on RULER and LOFT with BF16 Qwen3 / Ministral models ("Verify Before You
Fetch", summary page, Experimental Setup).  Neither the datasets nor the weights are used; these
generators stand in for them with the shapes of that setup (8 KV heads, 4 query heads per KV head,
d = 128, 32K / 128K contexts, 8-32x compression) and an attention model chosen so that the
certificate behaves like the pages' Table 2 (about a fifth to a quarter of decisions need no
fetch, a few percent of the context per fetching decision):

* importance scores tau: i.i.d. lognormal(0, 1.5) divided by their maximum (uniform in (0, 1) for
  the tiny case);
* keys: N(0, 1) per channel with outlier channels (4 channels x8 and 4 channels x4);
* queries: a shared per-head direction mu (on the outlier channels) times 4, plus N(0, 1);
* attention sinks: the first four keys get a component along mu so that they hold about half of
  the expected attention mass;
* planted queries: a quarter of the queries add a component along one planted key per KV head,
  scaled so that key holds about 20% of that head's attention mass; planted keys carry the
  smallest importance score of their head, so PoissonComp almost never keeps them.
"""
from dataclasses import dataclass, field

import numpy as np


def f32_to_bf16(x):
    """Round float32 to bf16 (round to nearest even), returned as uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_to_f32(u16):
    """Widen bf16 bit patterns to float32 (exact)."""
    return (np.asarray(u16, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclass
class Workload:
    """One synthetic workload.

    tau      float32 [B][L][h_kv][n]            importance scores
    kv       uint16  [B][L][h_kv][n][2][d]      bf16 K (index 0) and V (index 1) rows
    queries  uint16  [Q][B][h_kv*G][d]          bf16 decode queries; query head h*G+g uses KV head h
    query_layer int32 [Q]                       the layer each query attends
    planted  bool    [Q]                        query aimed at planted keys
    plant_pos int64  [B][L][h_kv][P]            planted token positions
    """
    name: str
    B: int
    L: int
    h_kv: int
    G: int
    d: int
    n: int
    eta: float
    n_sink: int
    n_local: int
    eps: float
    delta: float
    seed: int
    tau: np.ndarray
    kv: np.ndarray
    queries: np.ndarray
    query_layer: np.ndarray
    planted: np.ndarray
    plant_pos: np.ndarray
    meta: dict = field(default_factory=dict)

    @property
    def hq(self):
        return self.h_kv * self.G

    def kv_bytes(self):
        return self.kv.nbytes


def _channel_scales(d, outliers):
    s = np.ones(d, dtype=np.float32)
    if outliers:
        s[:4] = 8.0
        s[4:8] = 4.0
    return s


def _head_keys(rng, n, d, scales, mu, alpha, sink_frac, n_sinks=4):
    """Keys of one KV head with attention sinks along mu (see the module docstring)."""
    K = rng.standard_normal((n, d), dtype=np.float32) * scales
    if sink_frac > 0 and n_sinks > 0 and n > n_sinks:
        # Expected log-weight of a key under q = alpha*mu + N(0, I): alpha mu.k/sqrt(d) + |k|^2/(2d).
        base = alpha * (K @ mu) / np.sqrt(d) + (K * K).sum(1) / (2 * d)
        top = base.max()
        mass = np.exp(base - top).sum(dtype=np.float64)
        target = np.log(sink_frac / (1.0 - sink_frac) * mass / n_sinks) + top
        for i in range(n_sinks):
            K[i] += np.float32((target - base[i]) * np.sqrt(d) / alpha) * mu
    return K


def make_workload(name, *, B=1, L=1, h_kv=8, G=4, d=128, n=32768, eta=1.0 / 16, n_sink=4,
                  n_local=512, n_queries=256, plant_every=4, n_plants=8, eps=0.05, delta=0.05,
                  tau_kind="lognormal", outliers=True, alpha=4.0, sink_frac=0.5, plant_frac=0.2,
                  data_seed=1234, philox_seed=0):
    """Build a seeded workload.  Every fourth query (plant_every) is aimed at planted keys."""
    rng = np.random.default_rng(data_seed)
    scales = _channel_scales(d, outliers)
    tau = np.empty((B, L, h_kv, n), dtype=np.float32)
    kv = np.empty((B, L, h_kv, n, 2, d), dtype=np.uint16)
    mus = np.empty((B, L, h_kv, d), dtype=np.float32)
    n_plants = max(0, min(n_plants, n - n_sink - n_local))
    plant_pos = np.zeros((B, L, h_kv, n_plants), dtype=np.int64)
    lo, hi = n_sink, n - n_local
    for b in range(B):
        for l in range(L):
            for h in range(h_kv):
                mu = np.zeros(d, dtype=np.float32)
                k8 = min(8, d)
                mu[:k8] = rng.standard_normal(k8, dtype=np.float32)
                mu /= np.linalg.norm(mu)
                mus[b, l, h] = mu
                K = _head_keys(rng, n, d, scales, mu, alpha, sink_frac)
                V = rng.standard_normal((n, d), dtype=np.float32)
                if tau_kind == "lognormal":
                    x = rng.lognormal(0.0, 1.5, n)
                    t = (x / x.max()).astype(np.float32)
                else:  # uniform in (0, 1): (k + 1/2) / 2^24 with k uniform on 0..2^24-1
                    k = rng.integers(0, 1 << 24, n)
                    t = ((k.astype(np.float64) + 0.5) / float(1 << 24)).astype(np.float32)
                if n_plants > 0 and hi > lo:
                    pos = np.sort(rng.choice(np.arange(lo, hi), size=n_plants, replace=False))
                    plant_pos[b, l, h] = pos
                    others = np.ones(n, dtype=bool)
                    others[pos] = False
                    t[pos] = t[others].min()
                tau[b, l, h] = t
                kv[b, l, h, :, 0, :] = f32_to_bf16(K)
                kv[b, l, h, :, 1, :] = f32_to_bf16(V)

    Q = n_queries
    queries = np.empty((Q, B, h_kv * G, d), dtype=np.uint16)
    query_layer = (np.arange(Q) % L).astype(np.int32)
    planted = np.zeros(Q, dtype=bool)
    if plant_every > 0 and n_plants > 0:
        planted[plant_every - 1::plant_every] = True
    for t in range(Q):
        l = int(query_layer[t])
        for b in range(B):
            for h in range(h_kv):
                mu = mus[b, l, h]
                for g in range(G):
                    q = alpha * mu + rng.standard_normal(d, dtype=np.float32)
                    if planted[t]:
                        p = int(plant_pos[b, l, h, rng.integers(0, n_plants)])
                        Kh = bf16_to_f32(kv[b, l, h, :, 0, :])
                        s0 = (Kh @ q).astype(np.float64) / np.sqrt(d)
                        others = np.delete(s0, p)
                        top = others.max()
                        mass = np.exp(others - top).sum()
                        target = np.log(plant_frac / (1.0 - plant_frac) * mass) + top
                        kp = Kh[p]
                        knorm = float(np.linalg.norm(kp))
                        gamma = (target - s0[p]) * np.sqrt(d) / knorm
                        q = q + np.float32(gamma / knorm) * kp
                    queries[t, b, h * G + g] = f32_to_bf16(q)
    return Workload(name=name, B=B, L=L, h_kv=h_kv, G=G, d=d, n=n, eta=eta, n_sink=n_sink,
                    n_local=n_local, eps=eps, delta=delta, seed=philox_seed, tau=tau, kv=kv,
                    queries=queries, query_layer=query_layer, planted=planted,
                    plant_pos=plant_pos,
                    meta=dict(data_seed=data_seed, tau_kind=tau_kind, outliers=outliers,
                              alpha=alpha, sink_frac=sink_frac, plant_frac=plant_frac))


def tiny(data_seed=1234):
    """The oracle-in-seconds case: 1 layer, 1 KV head with 4 query heads, d = 64, n = 1024,
    tau uniform in (0, 1), H = 4 sinks + 64 local, eta = 1/8, 16 queries (half planted),
    eps = delta = 0.05, Philox seed 0."""
    return make_workload("tiny", B=1, L=1, h_kv=1, G=4, d=64, n=1024, eta=1.0 / 8, n_sink=4,
                         n_local=64, n_queries=16, plant_every=2, n_plants=8,
                         tau_kind="uniform", outliers=False, data_seed=data_seed)


def single_layer_32k(layers=4, n=32768, n_queries=256, data_seed=1235, **kw):
    """Single-layer 32K: n = 32768, 8 KV heads x 4 query heads, d = 128, eta = 1/16, H = 4 + 512,
    256 queries with a quarter planted, eps = delta = 0.05.  `layers` independent instances of
    the layer are generated so that a benchmark can rotate over more resident state than L2
    holds; each query attends one of them (query t -> layer t mod layers)."""
    return make_workload("single-layer-32k", B=1, L=layers, h_kv=8, G=4, d=128, n=n,
                         eta=1.0 / 16, n_sink=4, n_local=512, n_queries=n_queries,
                         plant_every=4, n_plants=8, data_seed=data_seed, **kw)


def pc_sweep_tau(units, n, data_seed=1239):
    """Importance scores for the PoissonComp throughput sweep: for each of `units` heads,
    i.i.d. lognormal(0, 1.5) divided by the head's maximum (float32 [units][n])."""
    rng = np.random.default_rng(data_seed)
    tau = np.empty((units, n), dtype=np.float32)
    for u in range(units):
        x = rng.lognormal(0.0, 1.5, n)
        tau[u] = (x / x.max()).astype(np.float32)
    return tau


def long_context_128k(B=4, L=1, h_kv=8, G=4, d=128, n=131072, eta=1.0 / 32, n_sink=4,
                      n_local=512, n_queries=8, eps=0.05, delta=0.05, boost=3.0,
                      p_range=(0.02, 0.25), alpha=4.0, data_seed=1237, philox_seed=0):
    """Long context with the fetch path stressed (128K tokens, batch 4, eta = 1/32).

    Keys, values, scores and sinks as in make_workload.  In addition every KV head gets a needle
    set: p n tokens (p ~ U[p_range] per head) at uniform positions outside the forced set, whose
    keys share a component a u along a random unit direction u of that head; every query adds
    the same a u, so a needle's logit rises by a^2 / sqrt(d) = boost.  With eta = 1/32 almost all
    needles are unsampled, so a certificate can only be met by fetching much of the needle set
    (the fraction actually fetched is measured, not set)."""
    rng = np.random.default_rng(data_seed)
    scales = _channel_scales(d, True)
    a = np.float32(np.sqrt(boost * np.sqrt(d)))
    tau = np.empty((B, L, h_kv, n), dtype=np.float32)
    kv = np.empty((B, L, h_kv, n, 2, d), dtype=np.uint16)
    mus = np.empty((B, L, h_kv, d), dtype=np.float32)
    us = np.empty((B, L, h_kv, d), dtype=np.float32)
    pfrac = np.empty((B, L, h_kv), dtype=np.float64)
    lo, hi = n_sink, n - n_local
    for b in range(B):
        for l in range(L):
            for h in range(h_kv):
                mu = np.zeros(d, dtype=np.float32)
                mu[:8] = rng.standard_normal(8, dtype=np.float32)
                mu /= np.linalg.norm(mu)
                mus[b, l, h] = mu
                K = _head_keys(rng, n, d, scales, mu, alpha, 0.5)
                V = rng.standard_normal((n, d), dtype=np.float32)
                x = rng.lognormal(0.0, 1.5, n)
                tau[b, l, h] = (x / x.max()).astype(np.float32)
                u = rng.standard_normal(d).astype(np.float32)
                u /= np.linalg.norm(u)
                us[b, l, h] = u
                p = rng.uniform(*p_range)
                pfrac[b, l, h] = p
                pos = rng.choice(np.arange(lo, hi), size=int(p * (hi - lo)), replace=False)
                K[pos] += a * u
                kv[b, l, h, :, 0, :] = f32_to_bf16(K)
                kv[b, l, h, :, 1, :] = f32_to_bf16(V)
    Q = n_queries
    queries = np.empty((Q, B, h_kv * G, d), dtype=np.uint16)
    query_layer = (np.arange(Q) % L).astype(np.int32)
    for t in range(Q):
        l = int(query_layer[t])
        for b in range(B):
            for h in range(h_kv):
                for g in range(G):
                    q = alpha * mus[b, l, h] + rng.standard_normal(d, dtype=np.float32) + a * us[b, l, h]
                    queries[t, b, h * G + g] = f32_to_bf16(q)
    return Workload(name="long-128k", B=B, L=L, h_kv=h_kv, G=G, d=d, n=n, eta=eta,
                    n_sink=n_sink, n_local=n_local, eps=eps, delta=delta, seed=philox_seed,
                    tau=tau, kv=kv, queries=queries, query_layer=query_layer,
                    planted=np.ones(Q, dtype=bool), plant_pos=np.zeros((B, L, h_kv, 0), np.int64),
                    meta=dict(data_seed=data_seed, boost=boost, needle_frac=pfrac))


def _sinks_torch(K, mu, alpha, n_sinks, sink_frac=0.5):
    """Attention sinks for a slice of units (torch, in place): the first n_sinks keys of each unit
    move along its direction mu until, for a query alpha mu + N(0, I), they hold about sink_frac
    of the expected attention mass -- the recipe of _head_keys.  K float32 [u][n][d], mu [u][d]."""
    import torch

    d = K.shape[-1]
    base = alpha * torch.einsum("und,ud->un", K, mu) / np.sqrt(d) + (K * K).sum(-1) / (2 * d)
    top = base.max(dim=1, keepdim=True).values
    mass = torch.exp(base - top).double().sum(dim=1, keepdim=True)
    target = torch.log(sink_frac / (1.0 - sink_frac) * mass / n_sinks).float() + top
    shift = (target - base[:, :n_sinks]) * (np.sqrt(d) / alpha)           # [u][n_sinks]
    K[:, :n_sinks] += shift[:, :, None] * mu[:, None, :]


def decode_step_cache_torch(units, n, d, G, layers, batch, kv_heads, device, seed=1238,
                            alpha=4.0, n_sinks=4, sink_frac=0.5, n_local=512, n_plants=8,
                            plant_every=4, plant_frac=0.2):
    """The full-decode-step cache on the device (torch, seeded), for sizes where numpy
    generation would take minutes: per unit, tau lognormal(0, 1.5) / max; keys N(0, 1) with the
    outlier channel scales of make_workload and the first n_sinks keys moved along the unit's
    direction mu until they hold about sink_frac of the expected attention mass (attention sinks,
    as in make_workload); values N(0, 1); bf16 by round-to-nearest.  Queries
    [layers][batch][kv_heads * G][d]: alpha mu + N(0, I).  As in make_workload, every unit has
    n_plants planted positions outside the forced set carrying the unit's smallest tau, and every
    plant_every-th (layer, sequence) query is planted: each query head adds a component along one
    planted key of its KV head, scaled so that key holds about plant_frac of the head's attention
    mass.  Returns (tau, kv int16 [units][n][2][d], queries int16, planted bool [layers][batch])."""
    import torch

    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    scales = torch.as_tensor(_channel_scales(d, True), device=device)
    x = torch.exp(1.5 * torch.randn((units, n), generator=gen, device=device))
    tau = (x / x.max(dim=1, keepdim=True).values).float()
    mu = torch.zeros((units, d), device=device)
    mu[:, :8] = torch.randn((units, 8), generator=gen, device=device)
    mu /= mu.norm(dim=1, keepdim=True)
    kv = torch.empty((units, n, 2, d), dtype=torch.int16, device=device)
    for u0 in range(0, units, 64):  # in slices, to bound the float32 temporaries
        u1 = min(units, u0 + 64)
        K = torch.randn((u1 - u0, n, d), generator=gen, device=device) * scales
        _sinks_torch(K, mu[u0:u1], alpha, n_sinks, sink_frac)
        kv[u0:u1, :, 0] = K.to(torch.bfloat16).view(torch.int16)
        del K
        V = torch.randn((u1 - u0, n, d), generator=gen, device=device)
        kv[u0:u1, :, 1] = V.to(torch.bfloat16).view(torch.int16)
        del V
    lo, hi = n_sinks, n - n_local
    n_plants = max(0, min(n_plants, hi - lo))
    plant_pos = None
    if n_plants > 0:
        # n_plants distinct positions in [lo, hi) per unit: the smallest of random keys
        keys = torch.rand((units, hi - lo), generator=gen, device=device)
        plant_pos = keys.topk(n_plants, dim=1, largest=False).indices + lo
        tmin = tau.min(dim=1, keepdim=True).values
        tau.scatter_(1, plant_pos, tmin.expand(-1, n_plants))
    # unit u = (b * layers + l) * kv_heads + h
    mu4 = mu.view(batch, layers, kv_heads, d).permute(1, 0, 2, 3)  # [layers][batch][kv_heads][d]
    q = alpha * mu4[:, :, :, None, :] + torch.randn((layers, batch, kv_heads, G, d), generator=gen,
                                                    device=device)
    planted = torch.zeros((layers, batch), dtype=torch.bool)
    if n_plants > 0 and plant_every > 0:
        flat = planted.view(-1)
        flat[plant_every - 1::plant_every] = True
        inv_sqrt_d = 1.0 / float(np.sqrt(d))
        for l in range(layers):
            for b in range(batch):
                if not planted[l, b]:
                    continue
                for h in range(kv_heads):
                    u = (b * layers + l) * kv_heads + h
                    Kh = kv[u, :, 0].view(torch.bfloat16).float()                 # [n][d]
                    pick = torch.randint(0, n_plants, (G,), generator=gen, device=device)
                    p = plant_pos[u, pick]                                         # [G]
                    # The query moves along the planted key without its outlier channels: those
                    # are shared by every key, so a step along them would lift the other logits
                    # as much as the plant's.  A few steps settle the mass despite the rest.
                    v = Kh[p].clone()                                              # [G][d]
                    v[:, :8] = 0.0
                    vk = (v * Kh[p]).sum(dim=1).double()
                    for _ in range(6):
                        qg = q[l, b, h].to(torch.bfloat16).float()                 # [G][d]
                        s0 = (qg @ Kh.T).double() * inv_sqrt_d                     # [G][n]
                        sp = s0.gather(1, p[:, None])[:, 0]
                        others = s0.scatter(1, p[:, None], float("-inf"))
                        top = others.max(dim=1).values
                        mass = torch.exp(others - top[:, None]).sum(dim=1)
                        target = torch.log(plant_frac / (1.0 - plant_frac) * mass) + top
                        step = (target - sp) / inv_sqrt_d / vk
                        q[l, b, h] += step.float()[:, None] * v
    # contiguous [layers][batch][kv_heads * G][d]: the broadcast against the permuted mu4 would
    # otherwise leave the batch dimension outermost in memory
    queries = q.reshape(layers, batch, kv_heads * G, d).to(torch.bfloat16).contiguous()
    return tau, kv, queries.view(torch.int16), planted


def long_context_torch(units, n, d, G, layers, batch, kv_heads, device, seed=1240, alpha=4.0,
                       n_sinks=4, sink_frac=0.5, n_local=512, boost=3.0, p_range=(0.02, 0.25)):
    """The long-context workload with the fetch path stressed, generated on the device (torch,
    seeded) for sizes where numpy would take minutes: scores, keys, values and sinks as in
    decode_step_cache_torch, and per unit a needle set of p n tokens (p ~ U[p_range]) at uniform
    positions outside the forced set whose keys share a component a u along a random unit
    direction u of the unit; every query of the unit adds the same a u, so a needle's logit rises
    by a^2 / sqrt(d) = boost (as long_context_128k does).  Returns (tau, kv int16 [units][n][2][d],
    queries int16 [layers][batch][kv_heads * G][d], needle fraction per unit)."""
    import torch

    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    scales = torch.as_tensor(_channel_scales(d, True), device=device)
    x = torch.exp(1.5 * torch.randn((units, n), generator=gen, device=device))
    tau = (x / x.max(dim=1, keepdim=True).values).float()
    mu = torch.zeros((units, d), device=device)
    mu[:, :8] = torch.randn((units, 8), generator=gen, device=device)
    mu /= mu.norm(dim=1, keepdim=True)
    un = torch.randn((units, d), generator=gen, device=device)
    un /= un.norm(dim=1, keepdim=True)
    a = float(np.sqrt(boost * np.sqrt(d)))
    lo, hi = n_sinks, n - n_local
    pfrac = torch.empty(units, device=device).uniform_(p_range[0], p_range[1], generator=gen)
    kv = torch.empty((units, n, 2, d), dtype=torch.int16, device=device)
    for u0 in range(0, units, 16):  # in slices, to bound the float32 temporaries
        u1 = min(units, u0 + 16)
        K = torch.randn((u1 - u0, n, d), generator=gen, device=device) * scales
        _sinks_torch(K, mu[u0:u1], alpha, n_sinks, sink_frac)
        # needles: the first p (hi - lo) tokens of a random order of [lo, hi)
        order = torch.rand((u1 - u0, hi - lo), generator=gen, device=device).argsort(dim=1) + lo
        cnt = (pfrac[u0:u1] * (hi - lo)).long()
        take = torch.arange(hi - lo, device=device)[None, :] < cnt[:, None]
        needle = torch.zeros((u1 - u0, n), dtype=torch.bool, device=device)
        needle.scatter_(1, order, take)
        K += needle[:, :, None].float() * (a * un[u0:u1, None, :])
        kv[u0:u1, :, 0] = K.to(torch.bfloat16).view(torch.int16)
        del K, needle, order
        V = torch.randn((u1 - u0, n, d), generator=gen, device=device)
        kv[u0:u1, :, 1] = V.to(torch.bfloat16).view(torch.int16)
        del V
    # unit u = (b * layers + l) * kv_heads + h
    mu4 = mu.view(batch, layers, kv_heads, d).permute(1, 0, 2, 3)
    un4 = un.view(batch, layers, kv_heads, d).permute(1, 0, 2, 3)
    q = (alpha * mu4 + a * un4)[:, :, :, None, :] + torch.randn((layers, batch, kv_heads, G, d),
                                                                generator=gen, device=device)
    queries = q.reshape(layers, batch, kv_heads * G, d).to(torch.bfloat16).contiguous()
    return tau, kv, queries.view(torch.int16), pfrac.cpu().numpy()
